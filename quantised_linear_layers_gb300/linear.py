"""FP8 linear layer: forward, dgrad and wgrad over the library's cast and GEMM.

Follows the three functions of "[Help] Starter script for nn.Linear for
fwd,bwd" (maintainer's pseudo-code) and the integration of "DeepGEMM
Essentials: High-Performance FP8 Matrix Multiplication" Part 18:

  fwd    Y  = X  W^T  : cast X per token; GEMM against W's 128x128 block cast
  dgrad  dX = dY W    : cast dY per token; GEMM reading W's own E4M3 cast
                        MN-major with the scale grid of W^T's cast, which W's
                        block cast writes in the same pass (a block's amax
                        does not depend on orientation)
  wgrad  dW = dY^T X  : cast dY and X with 1x128 groups along the token axis
                        into their own [T, features] layout; wgrad GEMM with
                        both operands MN-major and fp32 output, optionally
                        accumulated into a main grad

``mn_major=False`` selects the transposed form instead: dgrad always against
W^T's cast, wgrad with dY^T and X^T cast from transposed views into K-major
operands. On GB300 the MN-major weight gradient is the faster one (its casts
take 18 + 23 us against 25 + 38 us at dY [4096, 4096], X [4096, 7168], the
GEMMs run at the same speed), so it is the default.

W is cast once per weight update (``FP8Weight``), not every forward. With
``mn_major`` each activation is read once for both of its casts: the forward
casts X along its features and along the tokens in one pass and keeps the
latter (E4M3, half the bytes of X) for the weight gradient, and the backward
casts dY both ways in one pass (``forward_saving`` / ``backward``). Every step
runs in the CUDA library; torch only allocates outputs.
"""
from __future__ import annotations

import torch

from . import ops


class FP8Weight:
    """A weight W [out, in] and its E4M3 cast with 128x128 block scales (the
    forward operand ``wq`` / ``ws``). With ``mn_major`` the same pass also
    writes ``ws_t``, the scale grid of W^T's cast, and the dgrad GEMM reads
    ``wq`` MN-major with it (``wtq`` / ``wts`` are None); otherwise W^T is cast
    on its own (``wtq`` / ``wts``, read from W column-wise)."""

    def __init__(self, w: torch.Tensor, fmt: int = ops.SF_PACKED_UE8M0, mn_major: bool = True):
        self.fmt = fmt
        self.mn_major = mn_major
        self.update(w)

    def update(self, w: torch.Tensor) -> None:
        if w.dim() != 2:
            raise ValueError("weight must be 2-D [out_features, in_features]")
        self.shape = tuple(w.shape)
        if self.mn_major:
            self.wq, self.ws, self.ws_t = ops.fp8_cast_per_block_dual(w, self.fmt)
            self.wtq = self.wts = None
        else:
            self.wq, self.ws = ops.fp8_cast_per_block(w, self.fmt)
            self.ws_t = None
            self.wtq, self.wts = ops.fp8_cast_per_block(w.t(), self.fmt)


def _cast_rows(x: torch.Tensor, fmt: int, mn_major: bool = True):
    """Per-token cast into a buffer whose rows start on 16-byte boundaries (the
    GEMM's operand loads need it; the rows' padding is never read)."""
    m, n = x.shape
    ld = -(-max(n, 1) // 16) * 16
    out = torch.empty((m, ld), dtype=torch.float8_e4m3fn, device=x.device)[:, :n]
    return ops.fp8_cast_per_token(x, 128, fmt, out=out, sf_mn_major=mn_major)


def _cast_cols(x: torch.Tensor, fmt: int):
    """Per-token cast of x^T (groups of 128 down the columns of x [T, C]) with
    the E4M3 output kept in x's own layout: returns (q [T, C] with 16-byte
    aligned rows, scales [C, ceil(T/128)] M-major)."""
    t, c = x.shape
    ld = -(-max(c, 1) // 16) * 16
    q = torch.empty((t, ld), dtype=torch.float8_e4m3fn, device=x.device)[:, :c]
    _, s = ops.fp8_cast_per_token(x.t(), 128, fmt, out=q.t(), sf_mn_major=True)
    return q, s


def forward(x: torch.Tensor, w: FP8Weight, out: torch.Tensor | None = None) -> torch.Tensor:
    """Y [T, out] = X [T, in] W^T (bf16)."""
    xq, xs = _cast_rows(x, w.fmt)
    return ops.gemm_fp8_nt_bf16(xq, xs, w.wq, w.ws, w.fmt, out=out)


def forward_saving(x: torch.Tensor, w: FP8Weight):
    """Y = X W^T plus X's cast along the tokens for the weight gradient, both
    from one read of X: returns (Y, (x_cols, x_cols_scales))."""
    xq, xs, xcq, xcs = ops.fp8_cast_per_token_dual(x, w.fmt)
    return ops.gemm_fp8_nt_bf16(xq, xs, w.wq, w.ws, w.fmt), (xcq, xcs)


def backward(dy: torch.Tensor, w: FP8Weight, x_cols, need_dx: bool = True, dw_out: torch.Tensor | None = None,
             accumulate: bool = False):
    """dX = dY W and dW (+)= dY^T X for an MN-major weight (``w.mn_major``),
    with dY cast along its features and along the tokens from one read and
    x_cols from ``forward_saving``. Returns (dX or None, dW)."""
    if not w.mn_major:
        raise ValueError("backward() takes an MN-major FP8Weight")
    dq, ds, dcq, dcs = ops.fp8_cast_per_token_dual(dy, w.fmt)
    dx = ops.gemm_fp8_nn_bf16(dq, ds, w.wq, w.ws_t, w.fmt) if need_dx else None
    xcq, xcs = x_cols
    dw = ops.gemm_fp8_wgrad_fp32_mn(dcq, dcs, xcq, xcs, out=dw_out, accumulate=accumulate, fmt=w.fmt)
    return dx, dw


def dgrad(dy: torch.Tensor, w: FP8Weight, out: torch.Tensor | None = None) -> torch.Tensor:
    """dX [T, in] = dY [T, out] W (bf16)."""
    dq, ds = _cast_rows(dy, w.fmt)
    if w.wtq is None:
        return ops.gemm_fp8_nn_bf16(dq, ds, w.wq, w.ws_t, w.fmt, out=out)
    return ops.gemm_fp8_nt_bf16(dq, ds, w.wtq, w.wts, w.fmt, out=out)


def wgrad(dy: torch.Tensor, x: torch.Tensor, fmt: int = ops.SF_PACKED_UE8M0,
          out: torch.Tensor | None = None, accumulate: bool = False, mn_major: bool = True) -> torch.Tensor:
    """dW [out, in] (+)= dY^T X (fp32); K is the token axis, both operands with
    1x128 scales along it: cast from the transposed views, or with
    ``mn_major`` cast into their own [T, features] layout and read MN-major."""
    if mn_major:
        aq, sa = _cast_cols(dy, fmt)
        bq, sb = _cast_cols(x, fmt)
        return ops.gemm_fp8_wgrad_fp32_mn(aq, sa, bq, sb, out=out, accumulate=accumulate, fmt=fmt)
    # both scale grids M-major: the scale loaders read 32 consecutive rows'
    # scales per load (K-major per-row B scales do not coalesce)
    aq, sa = _cast_rows(dy.t(), fmt)
    bq, sb = _cast_rows(x.t(), fmt)
    return ops.gemm_fp8_wgrad_fp32(aq, sa, bq, sb, out=out, accumulate=accumulate, fmt=fmt)


class _FP8LinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, w8, module):
        ctx.w8 = w8
        ctx.module = module
        ctx.x_dtype = x.dtype
        if w8.mn_major:
            # keep X's token-axis cast (E4M3) for the weight gradient, not X
            y, (xcq, xcs) = forward_saving(x, w8)
            ctx.save_for_backward(xcq, xcs)
            return y
        ctx.save_for_backward(x)
        return forward(x, w8)

    @staticmethod
    def backward(ctx, dy):
        dy = dy.contiguous()
        module = ctx.module
        to_main = module is not None and module.main_grad is not None
        w8 = ctx.w8
        if w8.mn_major:
            xcq, xcs = ctx.saved_tensors
            if not to_main and not ctx.needs_input_grad[1]:
                return (dgrad(dy, w8) if ctx.needs_input_grad[0] else None), None, None, None
            dx, dw = backward(dy, w8, (xcq, xcs), need_dx=ctx.needs_input_grad[0],
                              dw_out=module.main_grad if to_main else None, accumulate=to_main)
            return dx, (None if to_main else dw.to(ctx.x_dtype)), None, None
        (x,) = ctx.saved_tensors
        dx = dgrad(dy, w8) if ctx.needs_input_grad[0] else None
        if to_main:
            wgrad(dy, x, w8.fmt, out=module.main_grad, accumulate=True, mn_major=False)
            dw = None
        else:
            dw = wgrad(dy, x, w8.fmt, mn_major=False).to(x.dtype) if ctx.needs_input_grad[1] else None
        return dx, dw, None, None


class FP8Linear(torch.nn.Module):
    """nn.Linear (no bias) whose fwd / dgrad / wgrad run through the FP8 cast and
    GEMM. With ``accumulate_main_grad`` the weight gradient accumulates into the
    fp32 buffer ``main_grad`` (as the wgrad GEMM's accumulate form) instead of
    being returned to autograd; ``mn_major`` selects the MN-major backward
    (no transposed operands)."""

    def __init__(self, in_features: int, out_features: int, fmt: int = ops.SF_PACKED_UE8M0,
                 device=None, dtype=torch.bfloat16, accumulate_main_grad: bool = False, mn_major: bool = True):
        super().__init__()
        self.mn_major = mn_major
        self.weight = torch.nn.Parameter(torch.empty((out_features, in_features), device=device, dtype=dtype))
        torch.nn.init.normal_(self.weight, std=0.02)
        self.fmt = fmt
        self.main_grad = (torch.zeros((out_features, in_features), device=device, dtype=torch.float32)
                          if accumulate_main_grad else None)
        self._w8 = None
        self._w8_version = None

    def fp8_weight(self) -> FP8Weight:
        """The cached casts of the weight, refreshed when the weight changed."""
        v = self.weight._version
        if self._w8 is None or self._w8_version != v:
            with torch.no_grad():
                self._w8 = FP8Weight(self.weight.detach(), self.fmt, self.mn_major)
            self._w8_version = v
        return self._w8

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        """x [..., in_features] -> [..., out_features]: leading dimensions are
        flattened into tokens, as nn.Linear accepts them."""
        if x.shape[-1] != self.weight.shape[1]:
            raise ValueError(f"expected {self.weight.shape[1]} input features, got {x.shape[-1]}")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1])
        if x2.stride(1) != 1:
            x2 = x2.contiguous()
        y = _FP8LinearFn.apply(x2, self.weight, self.fp8_weight(), self)
        return y.reshape(*lead, y.shape[-1])
