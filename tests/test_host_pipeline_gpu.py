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


_TWO_THREADS = r"""
import sys, threading
import torch
sys.path.insert(0, sys.argv[1])
from quantised_linear_layers_gb300 import ops
from quantised_linear_layers_gb300 import synthetic as syn

torch.cuda.init()
m, n, k, chunk, fmt = 700, 512, 384, 128, 2
wq, ws = ops.fp8_cast_per_block(syn.randn((n, k), seed=syn.SEED_W, mul=0.02).cuda(), fmt)
xs = [syn.randn((m, k), seed=s).pin_memory() for s in (31, 32)]
outs = [torch.zeros((m, n), dtype=torch.bfloat16).pin_memory() for _ in xs]
streams = [torch.cuda.Stream() for _ in xs]
wsps = [torch.empty(ops.cast_gemm_host_workspace_size(n, k, chunk, fmt), dtype=torch.uint8, device="cuda")
        for _ in xs]
torch.cuda.synchronize()
start = threading.Barrier(2)
errors = []

def run(i):
    try:
        torch.cuda.set_device(0)
        with torch.cuda.stream(streams[i]):
            start.wait()
            ops.cast_gemm_host(xs[i], wq, ws, fmt, outs[i], chunk, wsps[i])
            streams[i].synchronize()
    except Exception as e:  # reported by the parent
        errors.append(repr(e))

threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
assert ops.device_status() == 0
for i in range(2):       # the same calls one after the other
    ref = torch.zeros((m, n), dtype=torch.bfloat16).pin_memory()
    ops.cast_gemm_host(xs[i], wq, ws, fmt, ref, chunk, wsps[i])
    torch.cuda.synchronize()
    assert torch.equal(outs[i], ref), f"thread {i} differs from the sequential call"
print("TWO_THREADS_OK")
"""


def test_first_calls_from_two_threads(ops):
    """Two host threads make the process's first ql_cast_gemm_host calls at
    the same moment, on their own streams and workspaces (a fresh process, so
    the pipeline's one-time set-up is what they race on). Both results equal
    the same calls made one after the other, bit for bit."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _TWO_THREADS, root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "TWO_THREADS_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
