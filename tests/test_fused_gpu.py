"""GPU parity of the GEMM with the per-token cast fused into its epilogue.

The fused output must be exactly the per-token cast ("DeepGEMM Essentials:
High-Performance FP8 Matrix Multiplication" Part 3, with the group and UE8M0
options) of the bf16 output that the bf16 GEMM computes with the same tiles:
the bf16 GEMM's output (itself judged against the exact product elsewhere) is
fed to the CPU oracle's cast, whose bytes and scales must match bit for bit.
The bf16 output is held to the GEMM tolerance against the oracle's exact
product in the same case, and the dequantised fused output is checked against
that product with a bound that adds E4M3's rounding step.
"""
import numpy as np
import pytest
import torch

from helpers import check_gemm, np_bytes, np_input, np_sf
from quantised_linear_layers_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from quantised_linear_layers_gb300 import build, ops as o
    build.build()
    o.load_library()
    yield o
    o.set_gemm_block_n(0)
    o.set_gemm_path(0)


def operands(ops, m, n, k, fmt, seed=0):
    x = syn.randn((m, k), seed=seed)
    w = syn.randn((n, k), seed=seed + 1, mul=0.02)
    xq, xs = ops.fp8_cast_per_token(x.cuda(), 128, fmt, sf_mn_major=True)
    wq, ws = ops.fp8_cast_per_block(w.cuda(), fmt)
    return xq, xs, wq, ws


def dequant(q, sf, gran, out_fmt, n):
    vals = q.float().cpu().numpy().astype(np.float64)
    s = np_sf(sf)
    if out_fmt == 2:
        e = s.astype(np.int64)
        e = np.stack([(e >> (8 * b)) & 0xFF for b in range(4)], axis=-1).reshape(s.shape[0], -1)
        s = np.ldexp(1.0, (e - 127).astype(np.int32))
    s = np.repeat(np.asarray(s, dtype=np.float64), gran, axis=1)[:, :n]
    return vals * s


# (m, n, k, path, input scale format): the CTA-pair kernel, the single-SM
# block-scaled kernel and the CUDA-core promotion kernel, ragged n
KERNELS = [(2048, 2560, 1024, 3, 2), (2048, 2560, 1024, 3, 1), (300, 520, 640, 3, 2), (300, 520, 640, 2, 2),
           (300, 520, 640, 2, 1), (300, 520, 640, 1, 0), (129, 7168, 512, 0, 0)]


@pytest.mark.parametrize("kcase", KERNELS, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}_path{c[3]}_fmt{c[4]}")
@pytest.mark.parametrize("gran", [128, 32])
@pytest.mark.parametrize("out_fmt,recip", [(0, False), (0, True), (1, False), (2, False)],
                         ids=["fp32", "fp32-recip", "ue8m0", "packed"])
def test_fused_cast_equals_cast_of_bf16_output(orc, ops, kcase, gran, out_fmt, recip):
    m, n, k, path, fmt = kcase
    xq, xs, wq, ws = operands(ops, m, n, k, fmt, seed=3)
    ops.set_gemm_path(path)
    ops.set_gemm_block_n(256)
    try:
        q, sf = ops.gemm_fp8_nt_fp8out(xq, xs, wq, ws, fmt, gran, out_fmt, recip, sf_mn_major=True)
        y = ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt)
    finally:
        ops.set_gemm_block_n(0)
        ops.set_gemm_path(0)
    assert ops.device_status() == 0
    # the bf16 output the fused cast starts from is itself the method's output
    ref = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt)
    check_gemm(y.float().cpu().numpy(), orc.round_output(ref, "bf16"), "bf16 output")
    oq, osf = orc.cast_per_token(np_input(y), gran, out_fmt, recip)
    assert np.array_equal(np_bytes(q), oq), "E4M3 bytes differ from the cast of the bf16 output"
    got_sf = np_sf(sf)
    if out_fmt == 2:
        assert np.array_equal(got_sf, osf)
    else:
        assert np.array_equal(got_sf.view(np.uint32), osf.view(np.uint32))
    # against the exact product: GEMM tolerance plus half an E4M3 step
    deq = dequant(q, sf, gran, out_fmt, n)
    rel = np.linalg.norm(deq - ref) / np.linalg.norm(ref)
    assert rel < 0.05, f"relative Frobenius error {rel:.3e}"


def test_worked_shape_default_path(orc, ops):
    """The pages' first shape (LHS [128, 512], RHS [256, 512]) on the default
    path, 1x128 packed UE8M0 output written M-major for the next GEMM."""
    xq, xs, wq, ws = operands(ops, 128, 256, 512, 2, seed=5)
    q, sf = ops.gemm_fp8_nt_fp8out(xq, xs, wq, ws, 2, 128, 2, sf_mn_major=True)
    ops.set_gemm_block_n(256)
    try:
        y = ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, 2)
    finally:
        ops.set_gemm_block_n(0)
    oq, osf = orc.cast_per_token(np_input(y), 128, 2)
    assert np.array_equal(np_bytes(q), oq) and np.array_equal(np_sf(sf), osf)
    # the fused output feeds the next GEMM directly
    w2 = syn.randn((384, 256), seed=9, mul=0.02)
    w2q, w2s = ops.fp8_cast_per_block(w2.cuda(), 2)
    d2 = ops.gemm_fp8_nt_bf16(q, sf, w2q, w2s, 2)
    ref2 = orc.gemm(np_bytes(q), np_sf(sf), np_bytes(w2q), np_sf(w2s), 2, out="bf16")
    check_gemm(d2.float().cpu().numpy(), ref2, "next layer")


@pytest.mark.parametrize("n", [300, 336])
@pytest.mark.parametrize("path", [0, 3], ids=["default", "pair"])
def test_output_views_untouched_outside(ops, path, n):
    """E4M3 output written into a column view of a taller, wider buffer: the
    bytes outside the view stay as they were, and the view holds the same bytes
    as a contiguous output. With n = 336 the view's rows start and end on
    16-byte boundaries, so the pair kernel writes through TMA tile stores (a
    ragged last tile); with n = 300 they do not end on one and it stores
    directly."""
    m, k = 300, 256
    xq, xs, wq, ws = operands(ops, m, n, k, 2, seed=11)
    parent = torch.full((m + 20, 400), 0x5A, dtype=torch.uint8, device="cuda")
    view = parent[:m, 48:48 + n].view(torch.float8_e4m3fn)
    ops.set_gemm_path(path)
    try:
        _, sf_v = ops.gemm_fp8_nt_fp8out(xq, xs, wq, ws, 2, 128, 2, out=view)
        q_c, sf_c = ops.gemm_fp8_nt_fp8out(xq, xs, wq, ws, 2, 128, 2)
    finally:
        ops.set_gemm_path(0)
    p = parent.cpu().numpy()
    assert np.all(p[:, :48] == 0x5A) and np.all(p[:, 48 + n:] == 0x5A) and np.all(p[m:] == 0x5A)
    assert np.array_equal(np_bytes(view), np_bytes(q_c)) and torch.equal(sf_v, sf_c)


@pytest.mark.parametrize("case", range(12))
def test_fused_cast_random_shapes(orc, ops, case):
    """Seeded random shapes, paths, input and output scale formats and group
    widths: the fused output equals the oracle's cast of the same-tiled bf16
    output bit for bit, and that output meets the GEMM tolerance."""
    rng = np.random.default_rng(14000 + case)
    m = int(rng.integers(1, 600))
    n = int(rng.integers(16, 1200))
    k = int(rng.integers(1, 10)) * 128 - 16 * int(rng.integers(0, 8))
    path = [0, 1, 2, 3][case % 4]
    fmt = [0, 1, 2][(case // 4) % 3]
    gran = [128, 32][int(rng.integers(0, 2))]
    out_fmt = int(rng.integers(0, 3))
    recip = bool(out_fmt == 0 and rng.integers(0, 2))
    xq, xs, wq, ws = operands(ops, m, n, k, fmt, seed=14100 + case)
    ops.set_gemm_path(path)
    ops.set_gemm_block_n(256)
    try:
        q, sf = ops.gemm_fp8_nt_fp8out(xq, xs, wq, ws, fmt, gran, out_fmt, recip, sf_mn_major=True)
        y = ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt)
    finally:
        ops.set_gemm_block_n(0)
        ops.set_gemm_path(0)
    assert ops.device_status() == 0
    what = f"m={m} n={n} k={k} path{path} fmt{fmt} g{gran} out{out_fmt} recip={recip}"
    ref = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt)
    check_gemm(y.float().cpu().numpy(), orc.round_output(ref, "bf16"), what + " bf16 output")
    oq, osf = orc.cast_per_token(np_input(y), gran, out_fmt, recip)
    assert np.array_equal(np_bytes(q), oq), what + ": E4M3 bytes differ from the cast of the bf16 output"
    got_sf = np_sf(sf)
    if out_fmt == 2:
        assert np.array_equal(got_sf, osf), what
    else:
        assert np.array_equal(got_sf.view(np.uint32), osf.view(np.uint32)), what
