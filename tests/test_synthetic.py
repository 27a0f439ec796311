"""The seeded input generators that both the CUDA path and the oracle draw
from: deterministic per seed, and shaped as the input recipe states (per-row
10**u scaling with u in [-3, 3], the planted edge cases, the contiguous
grouped layout of "DeepGEMM Essentials" Parts 8-9, uneven expert loads)."""
import torch

from quantised_linear_layers_gb300 import synthetic as syn


def test_seeded_and_distinct():
    a = syn.randn((64, 96), seed=5)
    assert torch.equal(a, syn.randn((64, 96), seed=5))
    assert not torch.equal(a, syn.randn((64, 96), seed=6))
    assert a.dtype == torch.bfloat16
    w = syn.randn((64, 96), seed=5, mul=0.02, dtype=torch.float32)
    base = syn.randn((64, 96), seed=5, dtype=torch.float32)
    assert torch.allclose(w, base * 0.02, rtol=0, atol=0)


def test_row_exponent_recipe():
    m, n = 200, 256
    x = syn.randn_row_exp(m, n, seed=syn.SEED_X, dtype=torch.float32)
    g = torch.Generator().manual_seed(syn.SEED_X)
    base = torch.randn((m, n), generator=g, dtype=torch.float32)
    ratio = (x / base).median(dim=1).values
    assert torch.all(ratio >= 10.0 ** -3 * (1 - 1e-6)) and torch.all(ratio <= 10.0 ** 3 * (1 + 1e-6))
    # the per-row factor spans the range: some rows below 10^-2, some above 10^2
    assert (ratio < 1e-2).any() and (ratio > 1e2).any()
    # one factor per row: the ratio is constant along a row up to fp32 rounding
    r = x / base
    assert torch.allclose(r, ratio[:, None].expand_as(r), rtol=1e-6, atol=0)
    xb = syn.randn_row_exp(m, n, seed=syn.SEED_X)
    assert torch.equal(xb, x.to(torch.bfloat16))


def test_planted_edges():
    x = syn.randn((7, 300), seed=1)
    syn.plant_edges(x, 128, zero_group=True, huge_row=3)
    assert torch.all(x[0, :128] == 0) and torch.any(x[0, 128:] != 0)
    row = x[3].float()
    assert torch.all(torch.isfinite(row))
    assert torch.all(row.abs() > 2.9e38)
    assert torch.all(row[0::2] > 0) and torch.all(row[1::2] < 0)
    y = syn.randn((1, 20), seed=1)
    syn.plant_edges(y, 32)                      # group wider than the row
    assert torch.all(y == 0)


def test_small_integers_are_exact_e4m3():
    v = syn.e4m3_small_ints((50, 70), seed=2)
    assert v.dtype == torch.float32
    assert torch.all(v == v.round()) and v.min() >= -8 and v.max() <= 8
    assert torch.equal(v.to(torch.float8_e4m3fn).float(), v)
    assert torch.equal(v, syn.e4m3_small_ints((50, 70), seed=2))


def test_contiguous_layout_of_the_pages_example():
    # Part 8's token counts with the 128-row alignment
    idx, aligned = syn.contiguous_layout([128, 96, 112, 144], 128)
    assert aligned == [128, 128, 128, 256]
    assert idx.dtype == torch.int32 and idx.numel() == 640
    expect = ([0] * 128 + [1] * 96 + [-1] * 32 + [2] * 112 + [-1] * 16 + [3] * 144 + [-1] * 112)
    assert idx.tolist() == expect
    idx0, aligned0 = syn.contiguous_layout([0, 5], 128)
    assert aligned0 == [0, 128] and idx0.tolist() == [1] * 5 + [-1] * 123


def test_uneven_expert_loads():
    t = syn.tokens_per_expert(8, 2048, seed=17)
    assert t == syn.tokens_per_expert(8, 2048, seed=17)
    assert len(t) == 8 and all(1536 <= v <= 2560 for v in t)
    assert len(set(t)) > 1


def test_canary_bytes():
    b = syn.random_bytes(4096, seed=9)
    assert b.dtype == torch.uint8 and b.numel() == 4096
    assert torch.equal(b, syn.random_bytes(4096, seed=9))
    assert len(torch.unique(b)) > 200
