"""Pins of the CPU oracle against things other than itself (no GPU).

Each test names what fixes the expected result: a library routine (torch /
ml_dtypes E4M3 conversion, numpy matmul), a closed form of the format, an
invariant of the method, brute force on exact small inputs, or a shape the
pages print. A plausible slip in the oracle (dropped clamp, wrong rounding
direction, transposed scale grid, wrong group boundary, lost sign) fails at
least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

from quantised_linear_layers_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FLOOR = float(np.float32(1e-4))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f32_of_bf16(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


# ---------------------------------------------------------------- I1: E4M3
def _stratified_f32():
    """fp32 values with |v| <= 464 covering every exponent, every 12-bit
    mantissa prefix and the rounding-relevant low-bit patterns."""
    exps = np.arange(0, 136, dtype=np.uint32)              # biased exponents 0..135 (2^8 binade)
    hi = np.arange(4096, dtype=np.uint32) << 11             # top 12 mantissa bits
    lo = np.array([0, 1, 0x3FF, 0x400, 0x401, 0x7FF], dtype=np.uint32)
    bits = (exps[:, None, None] << 23) | hi[None, :, None] | lo[None, None, :]
    bits = bits.ravel()
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    v = bits.view(np.float32)
    return v[np.abs(v) <= 464.0]


def test_e4m3_encoder_matches_torch_stratified(orc):
    v = _stratified_f32()
    assert v.size > 5_000_000
    ours = orc.e4m3_encode(v)
    ref = torch_e4m3(v)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {v[bad[:5]]} ours {ours[bad[:5]]} torch {ref[bad[:5]]}"


def test_e4m3_encoder_matches_torch_random(orc):
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2**32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 464.0)]
    assert np.array_equal(orc.e4m3_encode(v), torch_e4m3(v))


def test_e4m3_encoder_matches_ml_dtypes(orc):
    ml = pytest.importorskip("ml_dtypes")
    v = _stratified_f32()[::7]
    ref = v.astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(orc.e4m3_encode(v), ref)


def test_e4m3_decode_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(ours, ref, equal_nan=True)
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_closed_forms(orc):
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_closed_forms.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            val, code = line.split()
            rows.append((float(eval(val, {"__builtins__": {}})), int(code, 16)))
    v = np.array([r[0] for r in rows], dtype=np.float32)
    expect = np.array([r[1] for r in rows], dtype=np.uint8)
    assert np.array_equal(orc.e4m3_encode(v), expect)
    # round trip of every finite code
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(orc.e4m3_encode(orc.e4m3_decode(codes).astype(np.float32)), codes)


# ------------------------------------------------------- cast helpers
def sweep_input(m, n, dtype, gran, seed=syn.SEED_X, huge_row=None):
    x = syn.randn_row_exp(m, n, seed=seed, dtype=dtype)
    syn.plant_edges(x, gran, zero_group=True, huge_row=huge_row)
    if dtype == torch.bfloat16:
        return x, bf16_bits(x), x.float().numpy()
    return x, x.numpy().copy(), x.numpy().copy()


def group_amax(xf: np.ndarray, gran: int) -> np.ndarray:
    m, n = xf.shape
    G = -(-n // gran)
    pad = np.zeros((m, G * gran), dtype=np.float32)
    pad[:, :n] = np.abs(xf)
    return pad.reshape(m, G, gran).max(axis=2)


# ------------------------------------------------------- I2 amax invariant
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("gran", [32, 128])
def test_amax_element_maps_to_448(orc, dtype, gran):
    _, xo, xf = sweep_input(64, 1000, dtype, gran, huge_row=5)
    q, s = orc.cast_per_token(xo, gran, orc.SF_FP32)
    amax = group_amax(xf, gran)
    m, n = xf.shape
    for i in range(m):
        for g in range(amax.shape[1]):
            if amax[i, g] < FLOOR:
                continue
            sl = slice(g * gran, min(n, (g + 1) * gran))
            hit = np.abs(xf[i, sl]) == amax[i, g]
            assert np.all((q[i, sl][hit] & 0x7F) == 0x7E)
    assert orc.overflow_count() == 0


@pytest.mark.parametrize("gran", [32, 128])
def test_amax_element_ue8m0_range(orc, gran):
    _, xo, xf = sweep_input(64, 1000, torch.bfloat16, gran, huge_row=7)
    q, s = orc.cast_per_token(xo, gran, orc.SF_UE8M0)
    amax = group_amax(xf, gran)
    m, n = xf.shape
    for i in range(m):
        for g in range(amax.shape[1]):
            if amax[i, g] < FLOOR:
                continue
            sl = slice(g * gran, min(n, (g + 1) * gran))
            hit = np.abs(xf[i, sl]) == amax[i, g]
            mag = q[i, sl][hit] & 0x7F
            assert np.all((mag >= 0x76) & (mag <= 0x7E))      # (224, 448] after rounding


# ------------------------------------------------------- I3 all-zero group
@pytest.mark.parametrize("fmt,expect", [(0, np.float32(np.float32(1e-4) / np.float32(448.0))),
                                        (1, np.float32(2.0 ** -22))])
def test_all_zero_group(orc, fmt, expect):
    x = np.zeros((3, 256), dtype=np.float32)
    x[1, 128:] = np.linspace(-2, 3, 128, dtype=np.float32)
    q, s = orc.cast_per_token(x, 128, fmt)
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0)
    assert s[0, 0] == expect and s[0, 1] == expect and s[1, 0] == expect
    # packed: exponent byte of 2^-22 is 105
    qp, sp = orc.cast_per_token(x, 128, orc.SF_PACKED_UE8M0)
    assert sp.shape == (3, 1) and (int(sp[0, 0]) & 0xFFFF) == (105 | (105 << 8))
    assert int(sp[0, 0]) >> 16 == 0                         # groups 2, 3 do not exist


# ------------------------------------------------------- I4 partial group
@pytest.mark.parametrize("gran,groups", [(128, 8), (32, 32)])
@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_partial_last_group_equals_zero_padded(orc, gran, groups, fmt):
    _, xo, _ = sweep_input(64, 1000, torch.bfloat16, gran)
    q, s = orc.cast_per_token(xo, gran, fmt)
    padded = np.zeros((64, 1024), dtype=np.uint16)
    padded[:, :1000] = xo
    qp, sp = orc.cast_per_token(padded, gran, fmt)
    assert np.array_equal(q, qp[:, :1000])
    if fmt != 2:
        assert s.shape == (64, groups)
        assert np.array_equal(s, sp[:, :groups])
    else:
        assert s.shape == (64, -(-groups // 4))


# ------------------------------------------------------- I5 UE8M0 closed form
def test_ue8m0_closed_form(orc):
    _, xo, xf = sweep_input(129, 7168, torch.bfloat16, 128, huge_row=3)
    _, s32 = orc.cast_per_token(xo, 128, orc.SF_FP32)
    q, sue = orc.cast_per_token(xo, 128, orc.SF_UE8M0)
    s32 = s32.astype(np.float64)
    sue = sue.astype(np.float64)
    mant, ex = np.frexp(sue)
    assert np.all(mant == 0.5)                               # exact powers of two
    assert np.all(sue >= s32) and np.all(sue < 2 * s32)
    # packed bytes are the biased exponents of the same powers of two
    _, sp = orc.cast_per_token(xo, 128, orc.SF_PACKED_UE8M0)
    b = sp.view(np.uint8).reshape(129, -1)[:, :56]
    assert np.array_equal(b.astype(np.int64), (ex - 1 + 127).astype(np.int64))
    # powers of two map to themselves: amax/448 = 2^j exactly
    x = np.zeros((4, 128), dtype=np.float32)
    for j, p in enumerate([-20, -3, 0, 7]):
        x[j, 5] = np.float32(448.0 * 2.0 ** p)
        x[j, 9] = np.float32(-0.3 * 448.0 * 2.0 ** p)
    _, s = orc.cast_per_token(x, 128, orc.SF_UE8M0)
    assert np.array_equal(s[:, 0], np.float32([2.0 ** -20, 2.0 ** -3, 1.0, 2.0 ** 7]))


# ------------------------------------------------------- I6 transpose invariance
@pytest.mark.parametrize("fmt", [0, 1])
def test_block_cast_transpose_invariance(orc, fmt):
    w = syn.randn((256, 384), seed=syn.SEED_W, mul=0.02)
    wb = bf16_bits(w)
    q, s = orc.cast_per_block(wb, fmt)
    qt, st = orc.cast_per_block(np.ascontiguousarray(wb.T), fmt)
    assert np.array_equal(qt, q.T) and np.array_equal(st, s.T)
    # the transposed *view* gives the same bytes as the transposed copy
    qv, sv = orc.cast_per_block(wb.T, fmt)
    assert np.array_equal(qv, qt) and np.array_equal(sv, st)


def test_block_cast_matches_per_block_amax(orc):
    w = syn.randn((300, 200), seed=syn.SEED_W, mul=0.02)
    wb = bf16_bits(w)
    q, s = orc.cast_per_block(wb, orc.SF_FP32)
    wf = f32_of_bf16(wb)
    assert s.shape == (3, 2)
    for r in range(3):
        for c in range(2):
            blk = np.abs(wf[r * 128:(r + 1) * 128, c * 128:(c + 1) * 128])
            a = max(blk.max(), np.float32(1e-4))
            assert s[r, c] == np.float32(np.float64(a) / 448.0)
            hit = np.abs(wf[r * 128:(r + 1) * 128, c * 128:(c + 1) * 128]) == blk.max()
            assert np.all((q[r * 128:(r + 1) * 128, c * 128:(c + 1) * 128][hit] & 0x7F) == 0x7E)


# ------------------------------------------------------- I7 brute-force GEMM
@pytest.mark.parametrize("m,n,k", [(7, 5, 32), (33, 130, 256), (128, 256, 512)])
def test_gemm_exact_small_integers(orc, m, n, k):
    a = syn.e4m3_small_ints((m, k), seed=11).numpy()
    b = syn.e4m3_small_ints((n, k), seed=12).numpy()
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    assert np.array_equal(orc.e4m3_decode(qa), a.astype(np.float64))
    KB = -(-k // 128)
    sfa = np.ones((m, KB), dtype=np.float32)
    sfb = np.ones((-(-n // 128), KB), dtype=np.float32)
    d = orc.gemm(qa, sfa, qb, sfb, orc.SF_FP32)
    ref = a.astype(np.int64) @ b.astype(np.int64).T
    assert np.array_equal(d, ref.astype(np.float64))
    # wgrad form: per-row B scales, accumulate into an existing fp32 gradient
    sfb_rows = np.ones((n, KB), dtype=np.float32)
    d_in = np.arange(m * n, dtype=np.float64).reshape(m, n) - 7.0
    d2 = orc.gemm(qa, sfa, qb, sfb_rows, orc.SF_FP32, b_per_row=True, d_in=d_in)
    assert np.array_equal(d2, ref + d_in)


# ------------------------------------------------------- I8 RHS-scale orientation
def test_rhs_scale_grid_is_read_row_wise(orc):
    m, n, k = 40, 384, 640                                   # n/128 = 3 != k/128 = 5
    a = syn.e4m3_small_ints((m, k), seed=21).numpy()
    b = syn.e4m3_small_ints((n, k), seed=22).numpy()
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    sfa = np.ones((m, 5), dtype=np.float32)
    sfb = np.array([[2.0 ** (i - 2 * j) for j in range(5)] for i in range(3)], dtype=np.float32)
    d = orc.gemm(qa, sfa, qb, sfb, orc.SF_FP32)
    # dequantise B block by block (row block i = n // 128, column block j = k // 128)
    bdeq = b.astype(np.float64) * np.repeat(np.repeat(sfb.astype(np.float64), 128, 0), 128, 1)
    ref = a.astype(np.float64) @ bdeq.T
    assert np.array_equal(d, ref)
    # a transposed reading of the grid would differ (the pin discriminates)
    with pytest.raises(AssertionError):
        wrong = np.repeat(np.repeat(sfb.T.astype(np.float64)[:3, :3], 128, 0), 128, 1)
        assert np.array_equal(d[:, :384], (a[:, :384].astype(np.float64) @ (b[:, :384] * wrong).T))


def test_lhs_scales_per_row_per_kblock(orc):
    m, n, k = 16, 128, 384
    a = syn.e4m3_small_ints((m, k), seed=31).numpy()
    b = syn.e4m3_small_ints((n, k), seed=32).numpy()
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    sfa = np.array([[2.0 ** ((i % 5) - j) for j in range(3)] for i in range(m)], dtype=np.float32)
    sfb = np.ones((1, 3), dtype=np.float32)
    d = orc.gemm(qa, sfa, qb, sfb, orc.SF_FP32)
    adeq = a.astype(np.float64) * np.repeat(sfa.astype(np.float64), 128, 1)
    assert np.array_equal(d, adeq @ b.astype(np.float64).T)


def test_packed_scales_equal_fp32_scales_in_gemm(orc):
    m, n, k = 32, 256, 1024
    a = syn.e4m3_small_ints((m, k), seed=41).numpy()
    b = syn.e4m3_small_ints((n, k), seed=42).numpy()
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    rng = np.random.default_rng(5)
    ea = rng.integers(120, 134, size=(m, 8)).astype(np.uint8)
    eb = rng.integers(120, 134, size=(2, 8)).astype(np.uint8)
    fa = np.ldexp(1.0, ea.astype(np.int32) - 127).astype(np.float32)
    fb = np.ldexp(1.0, eb.astype(np.int32) - 127).astype(np.float32)
    pa = ea.view(np.int32).reshape(m, 2)                     # 4 bytes per word, little-endian
    pb = eb.view(np.int32).reshape(2, 2)
    d1 = orc.gemm(qa, fa, qb, fb, orc.SF_UE8M0)
    d2 = orc.gemm(qa, pa, qb, pb, orc.SF_PACKED_UE8M0)
    assert np.array_equal(d1, d2)


def test_gemm_matches_numpy_dequantised_matmul(orc):
    """Random fp32 scales: the per-K-block promotion equals the fp64 matmul of
    the dequantised operands up to fp64 rounding."""
    x = syn.randn((96, 512), seed=syn.SEED_X)
    w = syn.randn((256, 512), seed=syn.SEED_W, mul=0.02)
    qa, sa = orc.cast_per_token(bf16_bits(x), 128, orc.SF_FP32)
    qb, sb = orc.cast_per_block(bf16_bits(w), orc.SF_FP32)
    d = orc.gemm(qa, sa, qb, sb, orc.SF_FP32)
    adeq = orc.e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 128, 1)
    bdeq = orc.e4m3_decode(qb) * np.repeat(np.repeat(sb.astype(np.float64), 128, 0), 128, 1)
    ref = adeq @ bdeq.T
    assert np.max(np.abs(d - ref)) <= 1e-12 * np.max(np.abs(ref))
    # and the quantised product is close to the bf16 product (informational bound)
    full = x.double().numpy() @ w.double().numpy().T
    rel = np.linalg.norm(d - full) / np.linalg.norm(full)
    assert rel < 0.05


def test_gemm_sampled_rows_equal_full(orc):
    x = syn.randn((64, 256), seed=syn.SEED_X)
    w = syn.randn((128, 256), seed=syn.SEED_W)
    qa, sa = orc.cast_per_token(bf16_bits(x), 128, orc.SF_FP32)
    qb, sb = orc.cast_per_block(bf16_bits(w), orc.SF_FP32)
    full = orc.gemm(qa, sa, qb, sb, orc.SF_FP32)
    rows = [0, 5, 63, 17]
    assert np.array_equal(orc.gemm(qa, sa, qb, sb, orc.SF_FP32, rows=rows), full[rows])


# ------------------------------------------------------- I9 worked shapes
def test_worked_shapes(orc):
    with open(os.path.join(GOLDEN, "worked_shapes.json")) as fh:
        ws = json.load(fh)
    for key in ("fwd_worked", "small_worked"):
        c = ws[key]
        lhs = syn.randn(tuple(c["lhs"]), seed=syn.SEED_X)
        rhs = syn.randn(tuple(c["rhs"]), seed=syn.SEED_W)
        qa, sa = orc.cast_per_token(bf16_bits(lhs), 128, orc.SF_FP32)
        qb, sb = orc.cast_per_block(bf16_bits(rhs), orc.SF_FP32)
        assert list(sa.shape) == c["lhs_scales"] and list(sb.shape) == c["rhs_scales"]
        d = orc.gemm(qa, sa, qb, sb, orc.SF_FP32)
        assert list(d.shape) == c["out"]
    g = ws["wgrad_worked"]
    T, K, N = g["tokens"], g["in_features"], g["out_features"]
    x = syn.randn((T, K), seed=syn.SEED_X)
    dy = syn.randn((T, N), seed=syn.SEED_DY)
    # wgrad operands: transposed views cast per token along the token axis
    qdy, sdy = orc.cast_per_token(bf16_bits(dy).T, 128, orc.SF_FP32)
    qx, sx = orc.cast_per_token(bf16_bits(x).T, 128, orc.SF_FP32)
    dw = orc.gemm(qdy, sdy, qx, sx, orc.SF_FP32, b_per_row=True)
    assert list(dw.shape) == g["weight_grad"]
    full = dy.double().numpy().T @ x.double().numpy()
    assert np.linalg.norm(dw - full) / np.linalg.norm(full) < 0.05


# ------------------------------------------------------- I10 view isolation
def test_cast_writes_only_inside_views(orc):
    x = syn.randn((7, 4096), seed=syn.SEED_X)
    xb = bf16_bits(x)
    parent = syn.random_bytes(16 * 8192, seed=99).numpy()
    ref_parent = parent.copy()
    out = parent[:16 * 8192].reshape(16, 8192)[3:10, 100:4196]          # strided view
    sfp = syn.random_bytes(4 * 40 * 64, seed=98).numpy().view(np.float32).reshape(40, 64)
    ref_sfp = sfp.copy()
    out_sf = sfp[2:9, 1:65:2]                                            # [7, 32], strided
    q, s = orc.cast_per_token(xb, 128, orc.SF_FP32, out=out, out_sf=out_sf)
    qc, sc = orc.cast_per_token(xb, 128, orc.SF_FP32)
    assert np.array_equal(out, qc) and np.array_equal(out_sf, sc)
    mask = np.ones_like(parent, dtype=bool).reshape(16, 8192)
    mask[3:10, 100:4196] = False
    assert np.array_equal(parent.reshape(16, 8192)[mask], ref_parent.reshape(16, 8192)[mask])
    smask = np.ones(sfp.shape, dtype=bool)
    smask[2:9, 1:65:2] = False
    assert np.array_equal(sfp.view(np.uint32)[smask], ref_sfp.view(np.uint32)[smask])


# ------------------------------------------------------- I11 reference formula
def _torch_per_token(x: torch.Tensor, gran: int, ue8m0: bool, recip: bool):
    """Part 3's computation restated in torch CPU ops (own code, not shared)."""
    m, n = x.shape
    G = -(-n // gran)
    xp = torch.zeros((m, G * gran), dtype=x.dtype)
    xp[:, :n] = x
    xv = xp.view(m, G, gran)
    amax = xv.abs().float().amax(dim=2).clamp(min=1e-4)
    scale = amax / 448.0
    if ue8m0:
        scale = torch.pow(2.0, torch.ceil(torch.log2(scale)))
        factor = torch.ones_like(scale) / scale
    else:
        # tensor / tensor is a correctly rounded division; torch evaluates
        # "scalar / tensor" as reciprocal-then-multiply, which rounds twice.
        factor = (torch.ones_like(scale) / scale) if recip else (torch.full_like(amax, 448.0) / amax)
    q = (xv * factor.unsqueeze(2)).to(torch.float8_e4m3fn).view(m, G * gran)[:, :n]
    return q.contiguous().view(torch.uint8).numpy(), scale.numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("gran", [32, 128])
@pytest.mark.parametrize("ue8m0,recip", [(False, False), (False, True), (True, False)])
def test_cast_equals_torch_restatement(orc, dtype, gran, ue8m0, recip):
    x, xo, _ = sweep_input(129, 1000, dtype, gran, huge_row=11)
    q, s = orc.cast_per_token(xo, gran, orc.SF_UE8M0 if ue8m0 else orc.SF_FP32, recip=recip)
    tq, ts = _torch_per_token(x, gran, ue8m0, recip)
    assert np.array_equal(q, tq)
    assert np.array_equal(s, ts)


def test_block_cast_equals_torch_restatement(orc):
    w = syn.randn((300, 260), seed=syn.SEED_W, mul=0.02)
    q, s = orc.cast_per_block(bf16_bits(w), orc.SF_FP32)
    wp = torch.zeros((384, 384), dtype=torch.bfloat16)
    wp[:300, :260] = w
    v = wp.view(3, 128, 3, 128)
    amax = v.abs().float().amax(dim=(1, 3), keepdim=True).clamp(min=1e-4)
    tq = (v * (torch.full_like(amax, 448.0) / amax)).to(torch.float8_e4m3fn).view(384, 384)[:300, :260]
    assert np.array_equal(q, tq.contiguous().view(torch.uint8).numpy())
    assert np.array_equal(s, (amax / 448.0).view(3, 3).numpy())


def _torch_per_block(w: torch.Tensor, ue8m0: bool, recip: bool):
    """Part 4's computation restated in torch CPU ops (own code, not shared)."""
    m, n = w.shape
    R, C = -(-m // 128), -(-n // 128)
    wp = torch.zeros((R * 128, C * 128), dtype=w.dtype)
    wp[:m, :n] = w
    v = wp.view(R, 128, C, 128)
    amax = v.abs().float().amax(dim=(1, 3), keepdim=True).clamp(min=1e-4)
    scale = amax / 448.0
    if ue8m0:
        scale = torch.pow(2.0, torch.ceil(torch.log2(scale)))
    factor = (torch.ones_like(scale) / scale) if (recip or ue8m0) else (torch.full_like(amax, 448.0) / amax)
    q = (v * factor).to(torch.float8_e4m3fn).view(R * 128, C * 128)[:m, :n]
    return q.contiguous().view(torch.uint8).numpy(), scale.view(R, C).numpy()


@pytest.mark.parametrize("shape", [(300, 260), (256, 512)])
@pytest.mark.parametrize("ue8m0,recip", [(False, False), (False, True), (True, False)])
def test_block_cast_options_equal_torch_restatement(orc, shape, ue8m0, recip):
    """The block cast's fp32, reciprocal-of-scale and UE8M0 branches against
    Part 4's formula restated in torch, on randn weights and on fp32 blocks
    built so that the two readings of the factor give different bytes."""
    import recip_inputs
    fmt = orc.SF_UE8M0 if ue8m0 else orc.SF_FP32
    w = syn.randn(shape, seed=syn.SEED_W, mul=0.02)
    q, s = orc.cast_per_block(bf16_bits(w), fmt, recip=recip)
    tq, ts = _torch_per_block(w, ue8m0, recip)
    assert np.array_equal(q, tq) and np.array_equal(s, ts)
    ws = recip_inputs.sensitive_blocks(*shape, seed=4)
    q, s = orc.cast_per_block(ws, fmt, recip=recip)
    tq, ts = _torch_per_block(torch.from_numpy(ws), ue8m0, recip)
    assert np.array_equal(q, tq) and np.array_equal(s, ts)


def test_recip_branches_differ_where_the_readings_do(orc):
    """On inputs built for it, the reciprocal-of-scale branch of both casts
    gives bytes different from the default factor (the pins above would not
    notice a branch that ignored the option otherwise) while the scales are
    the same."""
    import recip_inputs
    wb = recip_inputs.sensitive_blocks(256, 384, seed=5)
    q0, s0 = orc.cast_per_block(wb, orc.SF_FP32)
    q1, s1 = orc.cast_per_block(wb, orc.SF_FP32, recip=True)
    assert np.array_equal(s0, s1) and not np.array_equal(q0, q1)
    for gran in (32, 128):
        xr = recip_inputs.sensitive_rows(6, 520, gran, seed=6)
        q0, s0 = orc.cast_per_token(xr, gran, orc.SF_FP32)
        q1, s1 = orc.cast_per_token(xr, gran, orc.SF_FP32, recip=True)
        assert np.array_equal(s0, s1) and not np.array_equal(q0, q1)
        tq, ts = _torch_per_token(torch.from_numpy(xr), gran, False, True)
        assert np.array_equal(q1, tq) and np.array_equal(s1, ts)


# ------------------------------------------------------- strided / dtype paths
def test_cast_transposed_view_equals_copy(orc):
    x = syn.randn_row_exp(300, 256, dtype=torch.bfloat16)
    xb = bf16_bits(x)
    q1, s1 = orc.cast_per_token(xb.T, 128, orc.SF_UE8M0)
    q2, s2 = orc.cast_per_token(np.ascontiguousarray(xb.T), 128, orc.SF_UE8M0)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_bf16_and_fp32_inputs_agree_on_bf16_values(orc):
    x = syn.randn_row_exp(16, 4096, dtype=torch.bfloat16)
    q1, s1 = orc.cast_per_token(bf16_bits(x), 32, orc.SF_PACKED_UE8M0)
    q2, s2 = orc.cast_per_token(x.float().numpy(), 32, orc.SF_PACKED_UE8M0)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_huge_values_no_overflow(orc):
    orc.reset_overflow_count()
    x = syn.randn_row_exp(8, 4096, dtype=torch.bfloat16)
    syn.plant_edges(x, 128, huge_row=2)
    for fmt in (0, 1, 2):
        q, s = orc.cast_per_token(bf16_bits(x), 128, fmt)
        mag = q[2] & 0x7F
        if fmt == 0:
            assert np.all(mag == 0x7E)
        else:                                   # a power-of-two scale puts amax in (224, 448]
            assert np.all((mag >= 0x76) & (mag <= 0x7E))
    assert orc.overflow_count() == 0


# ------------------------------------------------------- GEMM output rounding
def test_bf16_output_rounding(orc):
    """bf16 RNE of the exact result: equals torch's fp32 -> bf16 conversion on
    fp32 values, and resolves ties in doubles to the even neighbour."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal(1_000_000).astype(np.float32) * np.float32(1e3)
    ours = orc.round_output(v.astype(np.float64), "bf16")
    assert np.array_equal(ours, torch.from_numpy(v).to(torch.bfloat16).double().numpy())
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -40,
                     2.0 ** 100 * (1 + 2.0 ** -8)])
    expect = np.array([1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7, 2.0 ** 100])
    assert np.array_equal(orc.round_output(ties, "bf16"), expect)
    assert np.array_equal(orc.round_output(np.array([1 + 2.0 ** -30]), "f32"), np.array([1.0]))


def test_gemm_output_rounding_option(orc):
    x = syn.randn((64, 256), seed=syn.SEED_X)
    w = syn.randn((128, 256), seed=syn.SEED_W)
    qa, sa = orc.cast_per_token(bf16_bits(x), 128, orc.SF_FP32)
    qb, sb = orc.cast_per_block(bf16_bits(w), orc.SF_FP32)
    exact = orc.gemm(qa, sa, qb, sb, orc.SF_FP32)
    rounded = orc.gemm(qa, sa, qb, sb, orc.SF_FP32, out="bf16")
    assert np.array_equal(rounded, orc.round_output(exact, "bf16"))
    assert np.max(np.abs(rounded - exact) / np.maximum(np.abs(exact), 1e-30)) <= 2.0 ** -8


def test_block_cast_packed_words(orc):
    """Packed block scales hold the biased exponents of the UE8M0 block scales,
    four column blocks per word, pad bytes zero (odd column-block count)."""
    w = syn.randn((300, 5 * 128 + 7), seed=syn.SEED_W, mul=0.02)
    wb = bf16_bits(w)
    q1, s1 = orc.cast_per_block(wb, orc.SF_UE8M0)
    q2, s2 = orc.cast_per_block(wb, orc.SF_PACKED_UE8M0)
    assert np.array_equal(q1, q2)
    assert s2.shape == (3, 2) and s1.shape == (3, 6)
    e = ((s1.view(np.uint32) >> 23) & 0xFF).astype(np.uint8)
    padded = np.zeros((3, 8), dtype=np.uint8)
    padded[:, :6] = e
    assert np.array_equal(s2.view(np.uint8).reshape(3, 8), padded)


# ------------------------------------------- M-grouped contiguous GEMM (Parts 8-11)
def test_contiguous_layout_worked_example():
    shapes = json.load(open(os.path.join(GOLDEN, "worked_shapes.json")))
    for key in ("grouped_worked", "grouped_challenge"):
        w = shapes[key]
        idx, aligned = syn.contiguous_layout(w["tokens_per_expert"], w["alignment"])
        assert aligned == w["aligned"] and idx.numel() == w["total_aligned"]
        start = 0
        for e, (t, a) in enumerate(zip(w["tokens_per_expert"], aligned)):
            assert start % w["alignment"] == 0
            assert bool((idx[start:start + t] == e).all()) and bool((idx[start + t:start + a] == -1).all())
            start += a
    w = shapes["grouped_worked"]
    idx, _ = syn.contiguous_layout(w["tokens_per_expert"], w["alignment"])
    assert int((idx == -1).sum()) == w["padding_rows"]


def _grouped_int_case(G_tokens, n, k, seed):
    idx, aligned = syn.contiguous_layout(G_tokens, 128)
    m, G = idx.numel(), len(G_tokens)
    a = syn.e4m3_small_ints((m, k), seed=seed).numpy()
    b = syn.e4m3_small_ints((G, n, k), seed=seed + 1).numpy()
    return idx.numpy(), a, b


def test_grouped_gemm_exact_small_integers(orc):
    w = json.load(open(os.path.join(GOLDEN, "worked_shapes.json")))["grouped_worked"]
    n, k = w["n"], w["k"]
    idx, a, b = _grouped_int_case(w["tokens_per_expert"], n, k, 51)
    G, KB = b.shape[0], k // 128
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    sfa = np.ones((a.shape[0], KB), dtype=np.float32)
    # each expert's own grid: expert e scales its whole B by 2^(e-1)
    sfb = np.stack([np.full((n // 128, KB), 2.0 ** (e - 1), dtype=np.float32) for e in range(G)])
    d = orc.gemm_m_grouped_contiguous(qa, sfa, qb, sfb, orc.SF_FP32, idx)
    for i in range(a.shape[0]):
        e = idx[i]
        if e < 0:
            assert np.all(np.isnan(d[i]))
        else:
            ref = (a[i].astype(np.int64) @ b[e].astype(np.int64).T).astype(np.float64) * 2.0 ** (e - 1)
            assert np.array_equal(d[i], ref)
    # taking expert 0's weights for every row would not match (the pin discriminates)
    rows1 = np.nonzero(idx == 1)[0]
    wrong = a[rows1].astype(np.int64) @ b[0].astype(np.int64).T
    assert not np.array_equal(d[rows1], wrong.astype(np.float64))


def test_grouped_gemm_expert_scale_grid_row_wise(orc):
    n, k = 384, 640                                            # n/128 = 3 != k/128 = 5
    idx, a, b = _grouped_int_case([100, 0, 200], n, k, 61)      # an expert with no tokens
    G = b.shape[0]
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    sfa = np.array([[2.0 ** ((i % 3) - j) for j in range(5)] for i in range(a.shape[0])], dtype=np.float32)
    sfb = np.array([[[2.0 ** (e + i - 2 * j) for j in range(5)] for i in range(3)] for e in range(G)],
                   dtype=np.float32)
    d = orc.gemm_m_grouped_contiguous(qa, sfa, qb, sfb, orc.SF_FP32, idx)
    adeq = a.astype(np.float64) * np.repeat(sfa.astype(np.float64), 128, 1)
    for e in (0, 2):
        rows = np.nonzero(idx == e)[0]
        bdeq = b[e].astype(np.float64) * np.repeat(np.repeat(sfb[e].astype(np.float64), 128, 0), 128, 1)
        assert np.array_equal(d[rows], adeq[rows] @ bdeq.T)
    assert np.all(np.isnan(d[idx < 0]))


def test_grouped_gemm_packed_equals_fp32_powers(orc):
    idx, a, b = _grouped_int_case([130, 60], 256, 1024, 71)
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    m, G = a.shape[0], b.shape[0]
    rng = np.random.default_rng(9)
    ea = rng.integers(120, 134, size=(m, 8)).astype(np.uint8)
    eb = rng.integers(120, 134, size=(G, 2, 8)).astype(np.uint8)
    fa = np.ldexp(1.0, ea.astype(np.int32) - 127).astype(np.float32)
    fb = np.ldexp(1.0, eb.astype(np.int32) - 127).astype(np.float32)
    d1 = orc.gemm_m_grouped_contiguous(qa, fa, qb, fb, orc.SF_UE8M0, idx)
    d2 = orc.gemm_m_grouped_contiguous(qa, ea.view(np.int32).reshape(m, 2), qb,
                                       eb.view(np.int32).reshape(G, 2, 2), orc.SF_PACKED_UE8M0, idx)
    assert np.array_equal(d1, d2, equal_nan=True)


def test_grouped_gemm_rejects_bad_index(orc):
    idx, a, b = _grouped_int_case([128], 128, 128, 81)
    qa, qb = orc.e4m3_encode(a), orc.e4m3_encode(b)
    idx = idx.copy()
    idx[5] = 1                                                  # only expert 0 exists
    with pytest.raises(ValueError):
        orc.gemm_m_grouped_contiguous(qa, np.ones((128, 1), np.float32), qb, np.ones((1, 1, 1), np.float32),
                                      orc.SF_FP32, idx)
