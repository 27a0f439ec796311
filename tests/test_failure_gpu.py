"""Failure detection without a GPU fault.

Every wait inside the GEMM kernels is bounded in time. The test hook makes the
operand producer issue no copies, so the tensor-core issuer's wait on a barrier
that nothing will complete runs out: the kernel must record
QL_ERR_DEVICE_TIMEOUT in the device status word, free its tensor memory and
return, and the context must stay usable (the next call is correct). Covered
for the CUDA-core promotion kernels (single SM and CTA pairs), the single-SM
block-scaled kernel, the CTA-pair kernel and the split-K cluster kernel.
"""
import pytest
import torch

from helpers import check_gemm, np_bytes, np_sf
from quantised_linear_layers_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

QL_ERR_DEVICE_TIMEOUT = 5


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from quantised_linear_layers_gb300 import build, ops as o
    build.build()
    o.load_library()
    yield o
    o.test_stall_gemm_producer(False)
    o.set_wait_limit_ms(2000)
    o.set_gemm_path(0)


@pytest.mark.parametrize("path,fmt", [(1, 0), (5, 0), (7, 0), (2, 2), (3, 2), (4, 2)],
                         ids=["promotion", "promotion_pair", "promotion_split_k", "block_scaled", "pair", "split_k"])
def test_bounded_wait_times_out_and_context_survives(orc, ops, path, fmt):
    m, n, k = 512, 512, 1024
    x = syn.randn((m, k), seed=syn.SEED_X).cuda()
    w = syn.randn((n, k), seed=syn.SEED_W).cuda()
    xq, xs = ops.fp8_cast_per_token(x, 128, fmt, sf_mn_major=True)
    wq, ws = ops.fp8_cast_per_block(w, fmt)
    assert ops.device_status() == 0
    ops.set_gemm_path(path)
    ops.set_wait_limit_ms(200)
    try:
        ops.test_stall_gemm_producer(True)
        try:
            ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt)
        finally:
            ops.test_stall_gemm_producer(False)
        assert ops.device_status() == QL_ERR_DEVICE_TIMEOUT
        assert ops.device_status() == 0                 # reading clears the word
        d = ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt)  # the context is still usable
        assert ops.device_status() == 0
    finally:
        ops.set_wait_limit_ms(2000)
        ops.set_gemm_path(0)
    ref = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt, out="bf16")
    check_gemm(d.float().cpu().numpy(), ref)
