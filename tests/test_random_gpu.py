"""Seeded random sweeps of the cast and GEMM entry points against the CPU oracle.

Each case draws its shape, input type, group width, scale format, layout
(row-contiguous, transposed view, column-contiguous, output views with
offsets) or GEMM path from a fixed seed, so a failure names a reproducible
case. Casts must match the oracle bit for bit ("DeepGEMM Essentials:
High-Performance FP8 Matrix Multiplication" Part 3 with the options of the
fused-cast PR); GEMMs (Parts 1 and 6, RHS scales row-wise per "[Help] Starter
script for nn.Linear for fwd,bwd") must meet the GEMM tolerance.
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


def _scales_equal(got, want, fmt):
    g = np.ascontiguousarray(np_sf(got))
    w = np.ascontiguousarray(want)
    if fmt == 2:
        return np.array_equal(g, w)
    return np.array_equal(g.view(np.uint32), w.view(np.uint32))


@pytest.mark.parametrize("case", range(64))
def test_random_cast(orc, ops, case):
    rng = np.random.default_rng(1000 + case)
    m = int(rng.integers(1, 700))
    n = int(rng.integers(1, 900))
    dtype = [torch.bfloat16, torch.float32][int(rng.integers(0, 2))]
    gran = [32, 128][int(rng.integers(0, 2))]
    fmt = int(rng.integers(0, 3))
    recip = bool(fmt == 0 and rng.integers(0, 2))
    layout = ["rows", "transposed", "colmajor", "rows_view"][int(rng.integers(0, 4))]
    x = syn.randn_row_exp(m, n, seed=2000 + case, dtype=dtype)
    if layout == "rows":
        q, s = ops.fp8_cast_per_token(x.cuda(), gran, fmt, recip=recip, sf_mn_major=bool(rng.integers(0, 2)))
        oq, os_ = orc.cast_per_token(np_input(x), gran, fmt, recip=recip)
        got = np_bytes(q)
    elif layout == "rows_view":
        # input and output rows inside wider buffers at column offsets
        off_in, off_out = int(rng.integers(0, 9)), int(rng.integers(0, 17))
        xin = torch.zeros((m, n + off_in + 5), dtype=dtype)
        xin[:, off_in:off_in + n] = x
        parent = torch.full((m, n + off_out + 7), 0x5A, dtype=torch.uint8, device="cuda")
        view = parent[:, off_out:off_out + n].view(torch.float8_e4m3fn)
        xg = xin.cuda()[:, off_in:off_in + n]
        q, s = ops.fp8_cast_per_token(xg, gran, fmt, recip=recip, out=view)
        oq, os_ = orc.cast_per_token(np_input(x), gran, fmt, recip=recip)
        got = np_bytes(q)
        p = parent.cpu().numpy()
        assert np.all(p[:, :off_out] == 0x5A) and np.all(p[:, off_out + n:] == 0x5A), "bytes outside the view"
    else:
        # the cast of x^T: from a transposed view (row-major output) or kept
        # in x's layout (column-major output)
        oq, os_ = orc.cast_per_token(np_input(x).T, gran, fmt, recip=recip)
        if layout == "transposed":
            q, s = ops.fp8_cast_per_token(x.cuda().t(), gran, fmt, recip=recip)
            got = np_bytes(q)
        else:
            q_phys = torch.empty((m, n), dtype=torch.float8_e4m3fn, device="cuda")
            q, s = ops.fp8_cast_per_token(x.cuda().t(), gran, fmt, recip=recip, out=q_phys.t(), sf_mn_major=True)
            got = np_bytes(q_phys).T
    assert ops.device_status() == 0
    bad = np.argwhere(got != oq)
    assert bad.size == 0, f"{layout} m={m} n={n} {dtype} g{gran} fmt{fmt}: {len(bad)} bytes differ, first {bad[0]}"
    assert _scales_equal(s, os_, fmt), f"{layout} m={m} n={n}: scales differ"


@pytest.mark.parametrize("case", range(24))
def test_random_dual_cast(orc, ops, case):
    """fp8_cast_per_token_dual on random shapes, input types, formats and row
    offsets (unaligned rows read element by element): the cast of x and that
    of x^T kept in x's layout, each bit for bit the oracle's cast."""
    rng = np.random.default_rng(9000 + case)
    m = int(rng.integers(1, 700))
    n = int(rng.integers(1, 900))
    dtype = [torch.bfloat16, torch.float32][int(rng.integers(0, 2))]
    fmt = int(rng.integers(0, 3))
    recip = bool(fmt == 0 and rng.integers(0, 2))
    off = int(rng.integers(0, 2)) * int(rng.integers(1, 8))      # 0, or a column offset of 1..7
    base = syn.randn_row_exp(m, n + off, seed=9500 + case, dtype=dtype)
    x = base[:, off:]
    qr, sr, qc, sc = ops.fp8_cast_per_token_dual(base.cuda()[:, off:], fmt, recip)
    assert ops.device_status() == 0
    oq, os_ = orc.cast_per_token(np_input(x), 128, fmt, recip=recip)
    oqt, ost = orc.cast_per_token(np_input(x).T, 128, fmt, recip=recip)
    what = f"m={m} n={n} {dtype} fmt{fmt} recip={recip} off={off}"
    assert np.array_equal(np_bytes(qr), oq), what + ": row-cast bytes differ"
    assert np.array_equal(np_bytes(qc).T, oqt), what + ": column-cast bytes differ"
    assert _scales_equal(sr, os_, fmt) and _scales_equal(sc, ost, fmt), what + ": scales differ"


@pytest.mark.parametrize("case", range(16))
def test_random_block_cast_dual(orc, ops, case):
    """fp8_cast_per_block_dual on random shapes, input types and formats: W's
    E4M3 bytes and 128 x 128 scale grid, and the grid of W^T's cast, bit for
    bit the oracle's block casts of W and W^T."""
    rng = np.random.default_rng(9800 + case)
    m = int(rng.integers(1, 800))
    n = int(rng.integers(1, 900))
    dtype = [torch.bfloat16, torch.float32][int(rng.integers(0, 2))]
    fmt = int(rng.integers(0, 3))
    recip = bool(fmt == 0 and rng.integers(0, 2))
    w = syn.randn((m, n), seed=9900 + case, mul=0.02, dtype=dtype)
    q, s, st = ops.fp8_cast_per_block_dual(w.cuda(), fmt, recip=recip)
    assert ops.device_status() == 0
    oq, os_ = orc.cast_per_block(np_input(w), fmt, recip=recip)
    otq, ots = orc.cast_per_block(np_input(w).T, fmt, recip=recip)
    what = f"m={m} n={n} {dtype} fmt{fmt} recip={recip}"
    assert np.array_equal(np_bytes(q), oq), what + ": bytes differ"
    assert np.array_equal(np_bytes(q).T, otq), what + ": W^T bytes differ"
    assert _scales_equal(s, os_, fmt) and _scales_equal(st, ots, fmt), what + ": scale grids differ"


@pytest.mark.parametrize("case", range(32))
def test_random_gemm(orc, ops, case):
    rng = np.random.default_rng(3000 + case)
    m = int(rng.integers(1, 600))
    n = int(rng.integers(16, 800))
    k = int(rng.integers(16, 1200))
    fmt = int(rng.integers(0, 3))
    path = [0, 1, 2, 3][int(rng.integers(0, 4))]
    wgrad = bool(rng.integers(0, 2))
    x = syn.randn((m, k), seed=4000 + case)
    w = syn.randn((n, k), seed=5000 + case, mul=0.05)
    # operand rows padded to 16 bytes, as the GEMM requires
    ldk = -(-k // 16) * 16
    aq_buf = torch.empty((m, ldk), dtype=torch.float8_e4m3fn, device="cuda")[:, :k]
    xq, xs = ops.fp8_cast_per_token(x.cuda(), 128, fmt, out=aq_buf, sf_mn_major=True)
    ops.set_gemm_path(path)
    try:
        if wgrad:
            bq_buf = torch.empty((n, ldk), dtype=torch.float8_e4m3fn, device="cuda")[:, :k]
            wq, ws = ops.fp8_cast_per_token(w.cuda(), 128, fmt, out=bq_buf)
            d = ops.gemm_fp8_wgrad_fp32(xq, xs, wq, ws, fmt=fmt)
            ref = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt, b_per_row=True, out="f32")
        else:
            bq_buf = torch.empty((n, ldk), dtype=torch.float8_e4m3fn, device="cuda")[:, :k]
            wq, ws = ops.fp8_cast_per_block(w.cuda(), fmt, out=bq_buf)
            d = ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt)
            ref = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt, out="bf16")
    finally:
        ops.set_gemm_path(0)
    assert ops.device_status() == 0
    check_gemm(d.double().cpu().numpy(), ref, f"m={m} n={n} k={k} fmt{fmt} path{path} wgrad={wgrad}")


@pytest.mark.parametrize("case", range(15))
def test_random_gemm_small_m_long_k(orc, ops, case):
    """Small M with 16-32 K blocks, where the split-K forms apply: the automatic
    choice (split-K for 16 K blocks or more), the forced block-scaled (4) and
    promotion (7) split-K forms, the CTA-pair (5) and single-SM (6) promotion
    kernels, under random SM budgets, for the forward and weight-gradient
    forms; every result within the GEMM tolerance of the oracle."""
    rng = np.random.default_rng(6000 + case)
    m = int(rng.integers(1, 260))
    n = int(rng.integers(16, 1600))
    k = 128 * int(rng.integers(16, 33)) - 16 * int(rng.integers(0, 8))   # 16 to 32 K blocks, ragged
    fmt, path = case // 5, [0, 4, 5, 6, 7][case % 5]       # every (format, path) pair once
    sms = [0, 64, 96, 128][int(rng.integers(0, 4))]
    wgrad = case % 4 == 3
    x = syn.randn((m, k), seed=7000 + case)
    w = syn.randn((n, k), seed=8000 + case, mul=0.05)
    ldk = -(-k // 16) * 16
    aq_buf = torch.empty((m, ldk), dtype=torch.float8_e4m3fn, device="cuda")[:, :k]
    xq, xs = ops.fp8_cast_per_token(x.cuda(), 128, fmt, out=aq_buf, sf_mn_major=True)
    bq_buf = torch.empty((n, ldk), dtype=torch.float8_e4m3fn, device="cuda")[:, :k]
    ops.set_gemm_path(path)
    ops.set_num_sms(sms)
    try:
        if wgrad:
            wq, ws = ops.fp8_cast_per_token(w.cuda(), 128, fmt, out=bq_buf)
            d = ops.gemm_fp8_wgrad_fp32(xq, xs, wq, ws, fmt=fmt)
            ref = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt, b_per_row=True, out="f32")
        else:
            wq, ws = ops.fp8_cast_per_block(w.cuda(), fmt, out=bq_buf)
            d = ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt)
            ref = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt, out="bf16")
    finally:
        ops.set_gemm_path(0)
        ops.set_num_sms(0)
    assert ops.device_status() == 0
    check_gemm(d.double().cpu().numpy(), ref, f"m={m} n={n} k={k} fmt{fmt} path{path} sms{sms} wgrad={wgrad}")
