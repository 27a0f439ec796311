"""Inputs on which the two readings of the quantisation factor give
different E4M3 bytes.

The factor is either fl32(448 / amax) (the formula "DeepGEMM Essentials"
Part 3 prints) or fl32(1 / fl32(amax / 448)) (the reciprocal of the scale the
fused-cast PR speaks of). The two differ by an ulp for about a quarter of all
amax values, but that ulp rarely moves a product x * f across an E4M3 rounding
boundary, so random data cannot tell the readings apart. These inputs place
elements next to the boundaries (midpoints between neighbouring E4M3 values)
so that it does. The construction uses numpy fp32 arithmetic and torch's
E4M3 conversion only; it shares nothing with the oracle or the CUDA path.
"""
import numpy as np
import torch


def _factors(a: np.float32):
    f_div = np.float32(np.float32(448.0) / a)                       # fl32(448 / a)
    f_rcp = np.float32(np.float32(1.0) / np.float32(a / np.float32(448.0)))
    return f_div, f_rcp


def _e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def sensitive_group(width: int, rng: np.random.Generator) -> np.ndarray:
    """One group (or block, flattened) of `width` fp32 values: its amax a has
    fl32(448/a) != fl32(1/fl32(a/448)), and at least one element (usually
    many) quantises to different bytes under the two factors."""
    while True:
        a = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** int(rng.integers(-12, 12)))
        f_div, f_rcp = _factors(a)
        if f_div == f_rcp:
            continue
        found = []
        for e in range(-6, 9):
            for j in range(7 if e == 8 else 8):
                mid = np.float32(2.0 ** e * (1.0 + (2 * j + 1) / 16.0))
                x0 = np.float32(mid / f_div)
                for step in range(-3, 4):
                    x = x0
                    for _ in range(abs(step)):
                        x = np.nextafter(x, np.float32(np.inf if step > 0 else -np.inf), dtype=np.float32)
                    if not (0 < x < a):
                        continue
                    y = np.array([np.float32(x * f_div), np.float32(x * f_rcp)], dtype=np.float32)
                    q = _e4m3(y)
                    if q[0] != q[1]:
                        found.append(x)
        if not found:
            continue
        g = (rng.standard_normal(width).astype(np.float32) * np.float32(a / 8.0)).clip(-a / 2, a / 2)
        k = min(len(found), width - 1)
        pos = rng.choice(np.arange(1, width), size=k, replace=False)
        sign = np.where(rng.random(k) < 0.5, np.float32(-1.0), np.float32(1.0))
        g[pos] = np.asarray(found[:k], dtype=np.float32) * sign
        g[0] = -a if rng.random() < 0.5 else a
        return g.astype(np.float32)


def sensitive_rows(m: int, n: int, gran: int, seed: int) -> np.ndarray:
    """[m, n] fp32, every 1 x gran group built by sensitive_group (the last
    group of a row may be partial: it is cut from a full group that keeps its
    amax element first)."""
    rng = np.random.default_rng(seed)
    x = np.empty((m, n), dtype=np.float32)
    for r in range(m):
        for c0 in range(0, n, gran):
            w = min(gran, n - c0)
            x[r, c0:c0 + w] = sensitive_group(gran, rng)[:w]
    return x


def sensitive_blocks(m: int, n: int, seed: int) -> np.ndarray:
    """[m, n] fp32, every 128 x 128 block (edge blocks partial) built by
    sensitive_group, its amax element at the block's first row and column."""
    rng = np.random.default_rng(seed)
    x = np.empty((m, n), dtype=np.float32)
    for r0 in range(0, m, 128):
        for c0 in range(0, n, 128):
            h, w = min(128, m - r0), min(128, n - c0)
            g = sensitive_group(128 * 128, rng).reshape(128, 128)
            x[r0:r0 + h, c0:c0 + w] = g[:h, :w]
            x[r0, c0] = g[0, 0]
    return x
