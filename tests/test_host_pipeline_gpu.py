"""The forward step on host buffers (ql_cast_gemm_host): X copied in, cast,
multiplied and D copied out chunk by chunk with copies and kernels of
successive chunks overlapped. The result must equal, bit for bit, the same
kernels run on device buffers chunk by chunk, and be within the GEMM
tolerance of the CPU oracle ("[Help] Starter script for nn.Linear for
fwd,bwd": cast X per token, GEMM against W's block cast)."""
import numpy as np
import pytest
import torch

from helpers import check_gemm, np_bytes, np_sf
from quantised_linear_layers_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from quantised_linear_layers_gb300 import build, ops as o
    build.build()
    o.load_library()
    return o


def device_reference(ops, x, wq, ws, fmt, chunk):
    outs = []
    for r0 in range(0, x.shape[0], chunk):
        q, s = ops.fp8_cast_per_token(x[r0:r0 + chunk].cuda(), 128, fmt, sf_mn_major=True)
        outs.append(ops.gemm_fp8_nt_bf16(q, s, wq, ws, fmt).cpu())
    return torch.cat(outs)


@pytest.mark.parametrize("fmt", [0, 1, 2], ids=["fp32", "ue8m0", "packed"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_pipeline_equals_device_calls(orc, ops, fmt, pinned):
    m, n, k, chunk = 1000, 640, 512, 256            # a ragged last chunk
    x = syn.randn((m, k), seed=syn.SEED_X)
    w = syn.randn((n, k), seed=syn.SEED_W, mul=0.02).cuda()
    wq, ws = ops.fp8_cast_per_block(w, fmt)
    xh = x.pin_memory() if pinned else x.clone()
    out = torch.full((m, n), -1.0, dtype=torch.bfloat16)
    out = out.pin_memory() if pinned else out
    wsp = torch.empty(ops.cast_gemm_host_workspace_size(n, k, chunk, fmt), dtype=torch.uint8, device="cuda")
    ops.cast_gemm_host(xh, wq, ws, fmt, out, chunk, wsp)
    torch.cuda.current_stream().synchronize()
    assert ops.device_status() == 0
    ref = device_reference(ops, x, wq, ws, fmt, chunk)
    assert torch.equal(out, ref)
    rows = np.array([0, 1, 255, 256, 511, 767, 768, 999])
    q, s = ops.fp8_cast_per_token(x.cuda(), 128, fmt)
    oref = orc.gemm(np_bytes(q), np_sf(s), np_bytes(wq), np_sf(ws), fmt, rows=rows, out="bf16")
    check_gemm(out[rows].float().numpy(), oref, "host pipeline")


def test_host_pipeline_large_workload_sampled(orc, ops):
    """X [16384, 7168] bf16 on the host against W [18432, 7168] * 0.02, packed
    UE8M0, 2048-row chunks: sampled rows against the oracle, whole result
    against the device calls."""
    m, n, k, chunk = 16384, 18432, 7168, 2048
    x = syn.randn((m, k), seed=syn.SEED_X).pin_memory()
    w = syn.randn((n, k), seed=syn.SEED_W, mul=0.02).cuda()
    wq, ws = ops.fp8_cast_per_block(w, 2)
    del w
    out = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
    wsp = torch.empty(ops.cast_gemm_host_workspace_size(n, k, chunk, 2), dtype=torch.uint8, device="cuda")
    ops.cast_gemm_host(x, wq, ws, 2, out, chunk, wsp)
    torch.cuda.current_stream().synchronize()
    assert ops.device_status() == 0
    rows = np.array([0, 2047, 2048, 9000, 16383])
    q, s = ops.fp8_cast_per_token(x[torch.from_numpy(rows)].cuda(), 128, 2)
    oref = orc.gemm(np_bytes(q), np_sf(s), np_bytes(wq), np_sf(ws), 2, out="bf16")
    check_gemm(out[rows].float().numpy(), oref, "host pipeline, large")
    ref = device_reference(ops, x, wq, ws, 2, chunk)
    assert torch.equal(out, ref)
