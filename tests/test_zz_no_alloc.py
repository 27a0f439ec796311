"""ql_cast_gemm_host_noalloc: the host-buffer forward call for callers that
cannot allocate device memory when they call it (a plug-in whose host
application owns all device memory through its own pool, a serving process
that allows no new allocation after warm-up). It stages rows in an array
compiled into the library instead of a caller workspace; its results must
equal ql_cast_gemm_host's with a workspace, call after call, because the two
run the same kernels on the same row chunks. Called through the C ABI.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test when it gets here."""

import pytest
import torch

from quantised_linear_layers_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

QL_ERR_INVALID_ARG = 1
QL_ERR_UNSUPPORTED = 2
NOALLOC_BYTES = 64 << 20


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from quantised_linear_layers_gb300 import build, ops as o
    build.build()
    o.load_library()
    return o


def call_noalloc(ops, x, wq, ws, fmt, out, chunk):
    m, k = x.shape
    n = wq.shape[0]
    st = ops.load_library().ql_cast_gemm_host_noalloc(
        x.data_ptr(), x.stride(0), wq.data_ptr(), wq.stride(0), ws.data_ptr(), ws.stride(0), ws.stride(1),
        fmt, out.data_ptr(), out.stride(0), m, n, k, chunk, torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("fmt", [0, 2], ids=["fp32", "packed"])
def test_noalloc_equals_workspace_call_twice(ops, fmt):
    m, n, k, chunk = 1000, 640, 512, 256
    w = syn.randn((n, k), seed=syn.SEED_W, mul=0.02).cuda()
    wq, ws = ops.fp8_cast_per_block(w, fmt)
    wsp = torch.empty(ops.cast_gemm_host_workspace_size(n, k, chunk, fmt), dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((syn.SEED_X, 41)):        # two calls in a row, different inputs
        x = syn.randn((m, k), seed=seed).pin_memory()
        got = torch.full((m, n), -7.0, dtype=torch.bfloat16).pin_memory()
        ref = torch.full((m, n), -7.0, dtype=torch.bfloat16).pin_memory()
        assert call_noalloc(ops, x, wq, ws, fmt, got, chunk) == 0, f"call {call}"
        ops.cast_gemm_host(x, wq, ws, fmt, ref, chunk, wsp)
        torch.cuda.current_stream().synchronize()
        assert ops.device_status() == 0
        assert torch.equal(got, ref), f"call {call} differs from the workspace call"


def test_noalloc_rejects_chunks_beyond_the_array(ops):
    n, k, fmt = 18432, 7168, 2
    fits = NOALLOC_BYTES >= ops.cast_gemm_host_workspace_size(n, k, 512, fmt)
    too_big = ops.cast_gemm_host_workspace_size(n, k, 4096, fmt) > NOALLOC_BYTES
    assert fits and too_big
    x = torch.zeros((8, k), dtype=torch.bfloat16).pin_memory()
    out = torch.zeros((8, n), dtype=torch.bfloat16).pin_memory()
    wq = torch.zeros((n, k), dtype=torch.float8_e4m3fn, device="cuda")
    ws = torch.zeros((n // 128, 14), dtype=torch.int32, device="cuda")
    assert call_noalloc(ops, x, wq, ws, fmt, out, 4096) == QL_ERR_UNSUPPORTED


def test_noalloc_empty_and_bad_format_as_workspace_call(ops):
    """Empty shapes return QL_OK and a bad scale format QL_ERR_INVALID_ARG,
    as the workspace call does, whatever the chunk size."""
    n, k = 18432, 7168
    x = torch.zeros((8, k), dtype=torch.bfloat16).pin_memory()
    out = torch.zeros((8, n), dtype=torch.bfloat16).pin_memory()
    wq = torch.zeros((n, k), dtype=torch.float8_e4m3fn, device="cuda")
    ws = torch.zeros((n // 128, 14), dtype=torch.int32, device="cuda")
    lib = ops.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for m_, n_ in ((0, n), (8, 0)):
        assert lib.ql_cast_gemm_host_noalloc(x.data_ptr(), k, wq.data_ptr(), k, ws.data_ptr(), 14, 1, 2,
                                             out.data_ptr(), n, m_, n_, k, 4096, stream) == 0
    assert call_noalloc(ops, x, wq, ws, 7, out, 4096) == QL_ERR_INVALID_ARG
    torch.cuda.current_stream().synchronize()
    assert torch.count_nonzero(out) == 0
