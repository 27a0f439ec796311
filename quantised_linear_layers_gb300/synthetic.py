"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers: it holds none of the cast's or the
GEMM's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.

Seeds: LHS / X = 0, RHS / W = 1, dY = 2, per-row exponent = 3.

Recipes (the pages use no dataset; these stand in for the activations and
weights of "DeepGEMM Essentials: High-Performance FP8 Matrix Multiplication"
Parts 1, 12 and 18 and for the hidden-4096 token batches of "deep-gemm: fused
per-token FP8 cast in Triton (fused_per_token_cast_to_fp8), version 3"
[Results]):
  * ``randn``           standard normal, optionally times a constant (W: 0.02)
  * ``randn_row_exp``   standard normal times 10**u per row, u ~ U(-3, 3)
  * edge planting       one all-zero group (row 0, first group) and one row
                        of +-3.0e38 entries (representable in bf16)
  * ``contiguous_layout`` the expert-id vector of "DeepGEMM Essentials"
                        Parts 8-9: each expert's tokens padded up to the
                        alignment, padding rows marked -1
"""
from __future__ import annotations

import torch

SEED_X, SEED_W, SEED_DY, SEED_EXP = 0, 1, 2, 3


def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, seed: int, dtype=torch.bfloat16, mul: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """Standard-normal tensor (drawn in fp32, then rounded to ``dtype``) times ``mul``."""
    t = torch.randn(shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    if mul != 1.0:
        t = t * mul
    return t.to(dtype)


def randn_row_exp(m: int, n: int, seed: int = SEED_X, dtype=torch.bfloat16, device: str = "cpu",
                  exp_lo: float = -3.0, exp_hi: float = 3.0) -> torch.Tensor:
    """randn(m, n) times 10**u_r per row, u_r ~ U(exp_lo, exp_hi) (the cast-sweep recipe)."""
    base = torch.randn((m, n), generator=_gen(seed, device), dtype=torch.float32, device=device)
    u = torch.rand((m, 1), generator=_gen(SEED_EXP, device), dtype=torch.float32, device=device)
    u = exp_lo + (exp_hi - exp_lo) * u
    return (base * torch.pow(10.0, u)).to(dtype)


def plant_edges(x: torch.Tensor, gran: int, zero_group: bool = True, huge_row: int | None = None) -> torch.Tensor:
    """Plant the sweep's edge cases in place: an all-zero first group of row 0,
    and (optionally) one row of alternating +-3.0e38."""
    m, n = x.shape
    if zero_group and m > 0:
        x[0, : min(gran, n)] = 0
    if huge_row is not None and 0 <= huge_row < m:
        sign = torch.ones(n, dtype=torch.float32, device=x.device)
        sign[1::2] = -1.0
        x[huge_row, :] = (3.0e38 * sign).to(x.dtype)
    return x


def e4m3_small_ints(shape, seed: int, lo: int = -8, hi: int = 8, device: str = "cpu") -> torch.Tensor:
    """Integers in [lo, hi] (every one an exact E4M3 value) as float32, for brute-force GEMM pins."""
    return torch.randint(lo, hi + 1, shape, generator=_gen(seed, device), device=device).to(torch.float32)


def random_bytes(nbytes: int, seed: int, device: str = "cpu") -> torch.Tensor:
    """Canary bytes for view-isolation checks."""
    return torch.randint(0, 256, (nbytes,), generator=_gen(seed, device), dtype=torch.int32,
                         device=device).to(torch.uint8)


def contiguous_layout(tokens_per_expert, alignment: int = 128):
    """Expert index per row of the contiguous grouped layout: expert e's
    tokens, then -1 up to the next multiple of ``alignment``, expert after
    expert. Returns (int32 tensor [sum of aligned counts], aligned counts)."""
    aligned = [(t + alignment - 1) // alignment * alignment for t in tokens_per_expert]
    idx = torch.full((sum(aligned),), -1, dtype=torch.int32)
    start = 0
    for e, (t, a) in enumerate(zip(tokens_per_expert, aligned)):
        idx[start:start + t] = e
        start += a
    return idx, aligned


def tokens_per_expert(num_experts: int, mean: int, seed: int, spread: float = 0.25) -> list:
    """Uneven token counts per expert: mean * U(1 - spread, 1 + spread), rounded."""
    g = _gen(seed)
    u = torch.rand(num_experts, generator=g, dtype=torch.float64)
    return [int(round(mean * (1 - spread + 2 * spread * float(v)))) for v in u]
