"""GPU parity of the M-grouped contiguous GEMM against the fp64 CPU oracle.

"DeepGEMM Essentials: High-Performance FP8 Matrix Multiplication" Parts 8-11
(m_grouped_gemm_fp8_fp8_bf16_nt_contiguous): the tokens of all experts stacked
in one matrix, each expert's segment padded to a multiple of 128 with rows
marked -1, each row multiplied by its expert's weights with that expert's own
128x128 scale grid. Valid rows are judged with the GEMM tolerance against the
exact product rounded to bf16; padding rows must stay untouched; invalid
indices must be reported through the device status word.
"""
import numpy as np
import pytest
import torch

from helpers import check_gemm, np_bytes, np_sf
from quantised_linear_layers_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

QL_ERR_INVALID_ARG = 1
CANARY = -3072.0                       # exactly representable in bf16


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


def grouped_operands(ops, tokens, n, k, fmt, seed=0, w_mul=1.0):
    """Per-token cast of the stacked tokens, per-expert block casts of B."""
    idx, _ = syn.contiguous_layout(tokens, 128)
    m, G = idx.numel(), len(tokens)
    x = syn.randn((m, k), seed=seed)
    w = syn.randn((G, n, k), seed=seed + 1, mul=w_mul)
    xq, xs = ops.fp8_cast_per_token(x.cuda(), 128, fmt, sf_mn_major=True)
    wq = torch.empty((G, n, k), dtype=torch.float8_e4m3fn, device="cuda")
    cols = -(-k // 128)
    if fmt == 2:
        ws = torch.empty((G, -(-n // 128), -(-cols // 4)), dtype=torch.int32, device="cuda")
    else:
        ws = torch.empty((G, -(-n // 128), cols), dtype=torch.float32, device="cuda")
    wc = w.cuda()
    for e in range(G):
        ops.fp8_cast_per_block(wc[e], fmt, out=wq[e], out_sf=ws[e])
    return idx, xq, xs, wq, ws


def run_and_check(orc, ops, idx, xq, xs, wq, ws, fmt, rows=None):
    m, n = xq.shape[0], wq.shape[1]
    d = torch.full((m, n), CANARY, dtype=torch.bfloat16, device="cuda")
    ops.m_grouped_gemm_fp8_nt_bf16_contiguous(xq, xs, wq, ws, idx.cuda(), fmt, out=d)
    assert ops.device_status() == 0
    got = d.float().cpu().numpy()
    idn = idx.numpy()
    pad = idn < 0
    assert np.all(got[pad] == CANARY), "padding rows were written"
    if rows is None:
        ref = orc.gemm_m_grouped_contiguous(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), fmt, idn, out="bf16")
        check_gemm(got[~pad], ref[~pad], "grouped")
    else:
        rows = np.asarray([r for r in rows if idn[r] >= 0])
        ref = np.empty((rows.size, n))
        for e in np.unique(idn[rows]):
            sel = rows[idn[rows] == e]
            ref[idn[rows] == e] = orc.gemm(np_bytes(xq), np_sf(xs), np_bytes(wq[e]), np_sf(ws[e]), fmt,
                                           rows=sel, out="bf16")
        check_gemm(got[rows], ref, "grouped sampled rows")
    return d


@pytest.mark.parametrize("fmt", [0, 1, 2], ids=["fp32", "ue8m0", "packed"])
def test_worked_four_experts(orc, ops, fmt):
    """Part 8: 4 experts with [128, 96, 112, 144] tokens, expert_dim 512."""
    assert ops.get_m_alignment_for_contiguous_layout() == 128
    idx, xq, xs, wq, ws = grouped_operands(ops, [128, 96, 112, 144], 256, 512, fmt)
    run_and_check(orc, ops, idx, xq, xs, wq, ws, fmt)


@pytest.mark.parametrize("fmt", [0, 2], ids=["fp32", "packed"])
def test_practice_challenge_eight_experts(orc, ops, fmt):
    """The pages' challenge: 8 experts, [64, 128, 96, 112, 88, 144, 72, 104]
    tokens, hidden 2048."""
    idx, xq, xs, wq, ws = grouped_operands(ops, [64, 128, 96, 112, 88, 144, 72, 104], 2048, 2048, fmt, seed=5)
    run_and_check(orc, ops, idx, xq, xs, wq, ws, fmt)


@pytest.mark.parametrize("bn", [32, 64, 128, 256])
@pytest.mark.parametrize("path,fmt", [(1, 0), (1, 1), (2, 2), (3, 2)], ids=["prom-fp32", "prom-ue8m0", "mx", "pair-req"])
def test_every_tile_width_and_path(orc, ops, bn, path, fmt):
    """Ragged n (300), an expert with no tokens, K not a multiple of 128. The
    pair path is never taken for grouped problems (asked for, it falls back to
    the single-SM block-scaled kernel)."""
    idx, xq, xs, wq, ws = grouped_operands(ops, [200, 0, 37, 128, 1], 300, 592, fmt, seed=9)
    ops.set_gemm_block_n(bn)
    ops.set_gemm_path(path)
    try:
        run_and_check(orc, ops, idx, xq, xs, wq, ws, fmt)
    finally:
        ops.set_gemm_block_n(0)
        ops.set_gemm_path(0)


@pytest.mark.parametrize("bn", [32, 128, 256])
def test_exact_small_integers(orc, ops, bn):
    """Exact E4M3 integers in [-2, 2], unit scales, k = 256: every partial sum
    is an exact fp32 integer and |D| <= 256 is exact in bf16, so the result
    equals the integer product of each row with its expert's B."""
    tokens, n, k = [130, 250, 7], 384, 256
    idx, _ = syn.contiguous_layout(tokens, 128)
    m, G = idx.numel(), len(tokens)
    a = syn.e4m3_small_ints((m, k), seed=91, lo=-2, hi=2)
    b = syn.e4m3_small_ints((G, n, k), seed=92, lo=-2, hi=2)
    xq = a.to(torch.float8_e4m3fn).cuda()
    wq = b.to(torch.float8_e4m3fn).cuda()
    xs = torch.ones((k // 128, m), dtype=torch.float32, device="cuda").t()
    ws = torch.ones((G, n // 128, k // 128), dtype=torch.float32, device="cuda")
    d = torch.full((m, n), CANARY, dtype=torch.bfloat16, device="cuda")
    ops.set_gemm_block_n(bn)
    try:
        ops.m_grouped_gemm_fp8_nt_bf16_contiguous(xq, xs, wq, ws, idx.cuda(), 0, out=d)
    finally:
        ops.set_gemm_block_n(0)
    assert ops.device_status() == 0
    got = d.float().cpu().numpy()
    idn = idx.numpy()
    for e in range(G):
        rows = np.nonzero(idn == e)[0]
        ref = a[rows].numpy().astype(np.int64) @ b[e].numpy().astype(np.int64).T
        assert np.abs(ref).max() <= 256
        assert np.array_equal(got[rows], ref.astype(np.float64))
    assert np.all(got[idn < 0] == CANARY)


def test_padding_tile_is_skipped(orc, ops):
    """A whole 128-row block of padding between two experts is not computed
    and not written."""
    tokens, n, k = [128, 100], 256, 512
    idx, xq, xs, wq, ws = grouped_operands(ops, tokens, n, k, 2, seed=13)
    # insert a block of -1 rows between the experts
    idx2 = torch.cat([idx[:128], torch.full((128,), -1, dtype=torch.int32), idx[128:]])
    xq2 = torch.cat([xq[:128], xq[:128], xq[128:]])
    xs_rows = xs.t().contiguous()                       # [KB words, m] -> M-major copy
    xs2 = torch.cat([xs_rows[:, :128], xs_rows[:, :128], xs_rows[:, 128:]], dim=1).contiguous().t()
    run_and_check(orc, ops, idx2, xq2, xs2, wq, ws, 2)


@pytest.mark.parametrize("fmt", [0, 2], ids=["fp32", "packed"])
def test_moe_hidden7168_sampled_rows(orc, ops, fmt):
    """8 experts of about 512 tokens each (uneven), N = 4096, K = 7168,
    W = randn * 0.02: checked on a sample of rows from every expert."""
    tokens = syn.tokens_per_expert(8, 512, seed=17)
    idx, xq, xs, wq, ws = grouped_operands(ops, tokens, 4096, 7168, fmt, seed=21, w_mul=0.02)
    g = np.random.default_rng(3)
    rows = np.sort(g.choice(idx.numel(), size=96, replace=False))
    run_and_check(orc, ops, idx, xq, xs, wq, ws, fmt, rows=rows)


def test_invalid_indices_are_reported(orc, ops):
    """An index outside [-1, G) at a tile's first row skips the tile; a row
    whose expert differs from its tile's is not stored; both raise
    QL_ERR_INVALID_ARG in the status word and leave the context usable."""
    tokens, n, k = [256, 128], 256, 256
    idx, xq, xs, wq, ws = grouped_operands(ops, tokens, n, k, 0, seed=31)
    bad = idx.clone()
    bad[128] = 7                       # first row of expert 0's second tile: out of range
    bad[300] = 0                       # inside expert 1's tile: another expert
    d = torch.full((idx.numel(), n), CANARY, dtype=torch.bfloat16, device="cuda")
    ops.m_grouped_gemm_fp8_nt_bf16_contiguous(xq, xs, wq, ws, bad.cuda(), 0, out=d)
    assert ops.device_status() == QL_ERR_INVALID_ARG
    assert ops.device_status() == 0
    got = d.float().cpu().numpy()
    assert np.all(got[128:256] == CANARY)           # skipped tile
    assert np.all(got[300] == CANARY)               # row of the wrong expert
    ref = orc.gemm_m_grouped_contiguous(np_bytes(xq), np_sf(xs), np_bytes(wq), np_sf(ws), 0, idx.numpy(),
                                        out="bf16")
    keep = np.r_[0:128, 256:300, 301:384]
    check_gemm(got[keep], ref[keep], "rows around the invalid ones")
    # the next call is correct
    run_and_check(orc, ops, idx, xq, xs, wq, ws, 0)


@pytest.mark.parametrize("case", range(12))
def test_random_expert_layouts(orc, ops, case):
    """Seeded random mixtures: 1 to 10 experts, each with 0 to 400 tokens
    (empty experts included), ragged n and k, every scale format and the
    kernel paths the grouped GEMM takes; valid rows within the GEMM tolerance,
    padding rows untouched."""
    rng = np.random.default_rng(13000 + case)
    G = int(rng.integers(1, 11))
    tokens = [int(t) for t in rng.integers(0, 401, size=G)]
    if case % 2 == 1:
        tokens[int(rng.integers(0, G))] = 0          # an expert without tokens
    if sum(tokens) == 0:
        tokens[0] = 1
    n = int(rng.integers(16, 700))
    k = int(rng.integers(1, 12)) * 128 - 16 * int(rng.integers(0, 8))
    fmt = case % 3
    path = [0, 1, 2, 3][(case // 3) % 4]
    idx, xq, xs, wq, ws = grouped_operands(ops, tokens, n, k, fmt, seed=13100 + case, w_mul=0.05)
    ops.set_gemm_path(path)
    try:
        run_and_check(orc, ops, idx, xq, xs, wq, ws, fmt)
    finally:
        ops.set_gemm_path(0)
