"""GPU parity of the GEMMs with MN-major operands against the fp64 CPU oracle.

The weight gradient of "[Help] Starter script for nn.Linear for fwd,bwd"
reads dY [T, out] and X [T, in] with K = tokens: given K-outer ([k][m],
[k][n]) the operands need no transposed copies, and the data gradient reads W
[out, in] as a [k][n] operand with its 128x128 grid transposed. The oracle
takes the same E4M3 bytes in K-major order (a transposed copy made on the
CPU), so any mistake in the MN-major descriptors, coordinates or scale rows
changes the result. Exact small-integer cases with power-of-two scales must
match bit for bit; random cases are held to the GEMM tolerance.
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
    o.set_gemm_path(0)


def pow2_grid(rows, cols, seed, lo=-2, hi=2):
    g = torch.Generator().manual_seed(seed)
    return torch.pow(2.0, torch.randint(lo, hi + 1, (rows, cols), generator=g).float())


def pack_words(s):
    e = (s.view(torch.int32) >> 23) & 0xFF
    e = torch.nn.functional.pad(e, (0, (-e.shape[1]) % 4)).view(e.shape[0], -1, 4)
    return (e[..., 0] | (e[..., 1] << 8) | (e[..., 2] << 16) | (e[..., 3] << 24)).contiguous()


PATHS = [(1, "promotion"), (5, "promotion_pair"), (2, "block_scaled"), (3, "pair")]


@pytest.mark.parametrize("path", [p for p, _ in PATHS], ids=[n for _, n in PATHS])
@pytest.mark.parametrize("k", [256, 640, 1152])
@pytest.mark.parametrize("packed", [False, True])
def test_wgrad_mn_exact_pow2(orc, ops, path, k, packed):
    """Both operands K-outer, per-row power-of-two scales: exact fp32 result."""
    m, n = 200, 300
    kb = -(-k // 128)
    a = syn.e4m3_small_ints((m, k), seed=41, lo=-4, hi=4)
    b = syn.e4m3_small_ints((n, k), seed=42, lo=-4, hi=4)
    aq, bq = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn)
    # K-outer copies, rows padded to 16 bytes
    a_t = torch.zeros((k, 208), dtype=torch.float8_e4m3fn)
    a_t[:, :m] = aq.t()
    b_t = torch.zeros((k, 304), dtype=torch.float8_e4m3fn)
    b_t[:, :n] = bq.t()
    sa, sb = pow2_grid(m, kb, 43), pow2_grid(n, kb, 44)
    if packed:
        sa_dev, sb_dev, fmt = pack_words(sa).cuda(), pack_words(sb).cuda(), 2
    else:
        sa_dev, sb_dev, fmt = sa.cuda(), sb.cuda(), 1
    ops.set_gemm_path(path)
    try:
        d = ops.gemm_fp8_wgrad_fp32_mn(a_t.cuda()[:, :m], sa_dev, b_t.cuda()[:, :n], sb_dev, fmt=fmt)
    finally:
        ops.set_gemm_path(0)
    assert ops.device_status() == 0
    ref = orc.gemm(np_bytes(aq), sa.numpy(), np_bytes(bq), sb.numpy(), 1, b_per_row=True)
    got = d.double().cpu().numpy()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mismatches; first {bad[0]} got {got[tuple(bad[0])]} ref {ref[tuple(bad[0])]}"


@pytest.mark.parametrize("path", [p for p, _ in PATHS], ids=[n for _, n in PATHS])
def test_nn_exact_pow2_block_scales(orc, ops, path):
    """B given as [k][n] with its block grid [n/128, k/128] (a transposed view
    of a [k/128, n/128] grid, as W's own grid is for dgrad): bf16 output equals
    bf16_rn of the exact sum."""
    m, n, k = 160, 384, 1152
    kb = 9
    a = syn.e4m3_small_ints((m, k), seed=51, lo=-3, hi=3)
    b = syn.e4m3_small_ints((n, k), seed=52, lo=-3, hi=3)
    aq, bq = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn)
    sa = pow2_grid(m, kb, 53)
    grid_kn = pow2_grid(kb, 3, 54)                 # W's own grid [k-blocks][n-blocks]
    ops.set_gemm_path(path)
    try:
        d = ops.gemm_fp8_nn_bf16(aq.cuda(), sa.cuda(), bq.t().contiguous().cuda(), grid_kn.cuda().t(), 1)
    finally:
        ops.set_gemm_path(0)
    ref = orc.gemm(np_bytes(aq), sa.numpy(), np_bytes(bq), np.ascontiguousarray(grid_kn.numpy().T), 1, out="bf16")
    assert np.array_equal(d.double().cpu().numpy(), ref)


@pytest.mark.parametrize("fmt", [0, 1, 2], ids=["fp32", "ue8m0", "packed"])
@pytest.mark.parametrize("shape", [(4096, 1024, 2048), (300, 520, 200)], ids=["4096x1024x2048", "ragged"])
def test_wgrad_from_column_major_casts(orc, ops, fmt, shape):
    """The weight gradient as the Linear layer computes it: dY and X cast with
    1x128 groups along tokens into their own [T, features] layout, then the
    MN-major GEMM; compared with the oracle on the same bytes."""
    T, OUT, IN = shape
    dy = syn.randn((T, OUT), seed=syn.SEED_DY)
    x = syn.randn((T, IN), seed=syn.SEED_X)

    def cast_cols(t):
        rows, cols = t.shape
        ld = -(-cols // 16) * 16
        q = torch.empty((rows, ld), dtype=torch.float8_e4m3fn, device="cuda")[:, :cols]
        qv, s = ops.fp8_cast_per_token(t.cuda().t(), 128, fmt, out=q.t(), sf_mn_major=(t is dy))
        return q, s

    qdy, sdy = cast_cols(dy)
    qx, sx = cast_cols(x)
    d = ops.gemm_fp8_wgrad_fp32_mn(qdy, sdy, qx, sx, fmt=fmt)
    assert ops.device_status() == 0
    a = np.ascontiguousarray(np_bytes(qdy).T)
    b = np.ascontiguousarray(np_bytes(qx).T)
    if T * OUT * IN > 10 ** 9:
        rows = np.sort(np.random.default_rng(2).choice(OUT, 48, replace=False))
        ref = orc.gemm(a, np_sf(sdy), b, np_sf(sx), fmt, b_per_row=True, rows=rows, out="f32")
        check_gemm(d[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, "wgrad mn")
    else:
        ref = orc.gemm(a, np_sf(sdy), b, np_sf(sx), fmt, b_per_row=True, out="f32")
        check_gemm(d.cpu().numpy(), ref, "wgrad mn")
    # the casts are the per-token cast of dY^T / X^T, bit for bit
    oq, _ = orc.cast_per_token(np_input(dy).T, 128, fmt)
    assert np.array_equal(a, oq)


@pytest.mark.parametrize("fmt", [0, 1], ids=["fp32", "ue8m0"])
def test_dgrad_nn_with_w_own_cast(orc, ops, fmt):
    """dX = dY W with W's own block cast (data [out, in] read as [k][n], grid
    read transposed) equals the GEMM against the cast of W^T."""
    T, OUT, IN = 512, 1024, 768
    dy = syn.randn((T, OUT), seed=syn.SEED_DY).cuda()
    w = syn.randn((OUT, IN), seed=syn.SEED_W, mul=0.02).cuda()
    dq, ds = ops.fp8_cast_per_token(dy, 128, fmt, sf_mn_major=True)
    wq, ws = ops.fp8_cast_per_block(w, fmt)                # [out, in], grid [out/128, in/128]
    d_nn = ops.gemm_fp8_nn_bf16(dq, ds, wq, ws.t(), fmt)
    ref = orc.gemm(np_bytes(dq), np_sf(ds), np.ascontiguousarray(np_bytes(wq).T), np.ascontiguousarray(np_sf(ws).T),
                   fmt, out="bf16")
    check_gemm(d_nn.float().cpu().numpy(), ref, "dgrad nn")


@pytest.mark.parametrize("path", [0, 1, 5, 2, 3], ids=["default", "promotion", "promotion_pair", "block_scaled", "pair"])
@pytest.mark.parametrize("fmt", [0, 1, 2], ids=["fp32", "ue8m0", "packed"])
@pytest.mark.parametrize("shape", [(512, 1024, 768), (300, 640, 520)], ids=["512x1024x768", "ragged"])
def test_dgrad_from_dual_block_cast(orc, ops, fmt, path, shape):
    """dX = dY W from W's one block cast: the dual cast's second scale grid is
    the scale grid of cast_per_block(W^T) byte for byte (a block's amax does
    not depend on orientation; packed words run along W^T's column blocks),
    W's E4M3 bytes are W^T's cast transposed, and the NN GEMM over them meets
    the GEMM tolerance against the oracle on W^T's cast, in every format and
    on every kernel."""
    T, OUT, IN = shape
    dy = syn.randn((T, OUT), seed=syn.SEED_DY).cuda()
    w = syn.randn((OUT, IN), seed=syn.SEED_W, mul=0.02)
    wq, ws, ws_t = ops.fp8_cast_per_block_dual(w.cuda(), fmt)
    otq, ots = orc.cast_per_block(np_input(w).T, fmt)
    oq, os_ = orc.cast_per_block(np_input(w), fmt)
    assert np.array_equal(np_bytes(wq), oq) and np.array_equal(np_sf(ws).view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(np_bytes(wq).T, otq)
    assert np.array_equal(np_sf(ws_t).view(np.uint32), ots.view(np.uint32))
    dq, ds = ops.fp8_cast_per_token(dy, 128, fmt, sf_mn_major=True)
    ops.set_gemm_path(path)
    try:
        dx = ops.gemm_fp8_nn_bf16(dq, ds, wq, ws_t, fmt)
    finally:
        ops.set_gemm_path(0)
    assert ops.device_status() == 0
    ref = orc.gemm(np_bytes(dq), np_sf(ds), otq, ots, fmt, out="bf16")
    check_gemm(dx.float().cpu().numpy(), ref, "dgrad from the dual cast")
