"""The Linear layer's fwd / dgrad / wgrad on the GPU against the CPU oracle.

"[Help] Starter script for nn.Linear for fwd,bwd" (maintainer's pseudo-code):
fwd casts X per token and multiplies by W's block cast; dgrad casts dY and
multiplies by W^T's block cast (W transposed and requantised in 128x128
blocks: the same bytes as W's cast read MN-major, by transpose invariance);
wgrad casts dY^T and X^T per token along the token axis and writes fp32. Every cast is compared bit for bit with the oracle, every GEMM within
the GEMM tolerance, at the full nn.Linear workload (X [4096, 7168],
dY [4096, 4096], W [4096, 7168] * 0.02) on sampled rows.
"""
import numpy as np
import pytest
import torch

from helpers import check_gemm, np_bytes, np_input, np_sf
from quantised_linear_layers_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lin():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from quantised_linear_layers_gb300 import build, ops
    build.build()
    ops.load_library()
    from quantised_linear_layers_gb300 import linear
    return linear


def oracle_fmt(fmt):
    return fmt


@pytest.mark.parametrize("mn_major", [False, True], ids=["transposed", "mn_major"])
@pytest.mark.parametrize("fmt", [0, 2], ids=["fp32", "packed"])
@pytest.mark.parametrize("shape", [(4096, 7168, 4096), (300, 640, 384)], ids=["full", "ragged"])
def test_linear_fwd_dgrad_wgrad(orc, lin, fmt, shape, mn_major):
    T, IN, OUT = shape
    x = syn.randn((T, IN), seed=syn.SEED_X)
    dy = syn.randn((T, OUT), seed=syn.SEED_DY)
    w = syn.randn((OUT, IN), seed=syn.SEED_W, mul=0.02)
    xg, dyg, wg = x.cuda(), dy.cuda(), w.cuda()
    w8 = lin.FP8Weight(wg, fmt, mn_major)
    # weight casts: W and W^T, bit-exact
    bfmt = fmt
    oq, os_ = orc.cast_per_block(np_input(w), bfmt)
    assert np.array_equal(np_bytes(w8.wq), oq) and np.array_equal(np_sf(w8.ws).view(np.uint32), os_.view(np.uint32))
    otq, ots = orc.cast_per_block(np_input(w).T, bfmt)
    if w8.wtq is not None:                    # dgrad's own W^T cast
        assert not mn_major
        assert np.array_equal(np_bytes(w8.wtq), otq)
        assert np.array_equal(np_sf(w8.wts).view(np.uint32), ots.view(np.uint32))
    else:                                     # dgrad reads W's cast MN-major with W^T's scale grid
        assert mn_major
        assert np.array_equal(np_bytes(w8.wq).T, otq)
        assert np.array_equal(np_sf(w8.ws_t).view(np.uint32), ots.view(np.uint32))

    rng = np.random.default_rng(11)
    rows_t = np.sort(rng.choice(T, min(T, 24), replace=False))
    rows_o = np.sort(rng.choice(OUT, min(OUT, 16), replace=False))

    # fwd
    y = lin.forward(xg, w8)
    xq, xs = orc.cast_per_token(np_input(x), 128, fmt)
    ref = orc.gemm(xq, xs, oq, os_, fmt, rows=rows_t, out="bf16")
    check_gemm(y[torch.from_numpy(rows_t).cuda()].float().cpu().numpy(), ref, "fwd")
    # dgrad
    dx = lin.dgrad(dyg, w8)
    dq, ds = orc.cast_per_token(np_input(dy), 128, fmt)
    ref = orc.gemm(dq, ds, otq, ots, fmt, rows=rows_t, out="bf16")
    check_gemm(dx[torch.from_numpy(rows_t).cuda()].float().cpu().numpy(), ref, "dgrad")
    # wgrad, fresh and accumulated into an fp32 main grad
    dw = lin.wgrad(dyg, xg, fmt, mn_major=mn_major)
    aq, sa = orc.cast_per_token(np_input(dy).T, 128, fmt)
    bq, sb = orc.cast_per_token(np_input(x).T, 128, fmt)
    ref = orc.gemm(aq, sa, bq, sb, fmt, b_per_row=True, rows=rows_o, out="f32")
    check_gemm(dw[torch.from_numpy(rows_o).cuda()].double().cpu().numpy(), ref, "wgrad")
    main = syn.randn((OUT, IN), seed=5, dtype=torch.float32, mul=0.1).cuda()
    main0 = main.clone()
    lin.wgrad(dyg, xg, fmt, out=main, accumulate=True, mn_major=mn_major)
    ref_acc = orc.gemm(aq, sa, bq, sb, fmt, b_per_row=True, rows=rows_o,
                       d_in=main0.double().cpu().numpy(), out="f32")
    check_gemm(main[torch.from_numpy(rows_o).cuda()].double().cpu().numpy(), ref_acc, "wgrad accumulate")
    # informational: the quantised layer stays close to the bf16 product
    full = (xg.float() @ wg.float().t())
    rel = (torch.linalg.norm(y.float() - full) / torch.linalg.norm(full)).item()
    assert rel < 0.05


@pytest.mark.parametrize("fmt,mn_major", [(2, False), (0, True), (2, True)], ids=["packed", "fp32-mn", "packed-mn"])
def test_fp8_linear_module_autograd(orc, lin, fmt, mn_major):
    torch.manual_seed(0)
    T, IN, OUT = 512, 1024, 768
    m = lin.FP8Linear(IN, OUT, fmt=fmt, device="cuda", mn_major=mn_major)
    x = syn.randn((T, IN), seed=syn.SEED_X).cuda().requires_grad_(True)
    y = m(x)
    dy = syn.randn((T, OUT), seed=syn.SEED_DY).cuda()
    y.backward(dy)
    w8 = m.fp8_weight()
    ref_y = lin.forward(x.detach(), w8)
    assert torch.equal(y, ref_y)
    assert torch.equal(x.grad, lin.dgrad(dy, w8))
    dw = lin.wgrad(dy, x.detach(), m.fmt, mn_major=mn_major)
    assert torch.equal(m.weight.grad, dw.to(torch.bfloat16))
    # a weight update refreshes the cached casts
    with torch.no_grad():
        m.weight.mul_(2.0)
    assert m.fp8_weight() is not w8


def test_fp8_linear_main_grad_accumulates(lin):
    T, IN, OUT = 256, 512, 384
    m = lin.FP8Linear(IN, OUT, device="cuda", accumulate_main_grad=True)
    x = syn.randn((T, IN), seed=syn.SEED_X).cuda().requires_grad_(True)
    dy = syn.randn((T, OUT), seed=syn.SEED_DY).cuda()
    m(x).backward(dy)
    g1 = m.main_grad.clone()
    m(x).backward(dy)
    assert m.weight.grad is None
    assert torch.allclose(m.main_grad, 2 * g1, rtol=1e-5, atol=1e-5)


def test_fp8_linear_batched_input(lin):
    """A [batch, seq, features] input is flattened into tokens like nn.Linear:
    the output and both gradients equal those of the 2-D call."""
    B, S, IN, OUT = 3, 100, 512, 384
    m = lin.FP8Linear(IN, OUT, device="cuda")
    x = syn.randn((B * S, IN), seed=syn.SEED_X).cuda()
    dy = syn.randn((B * S, OUT), seed=syn.SEED_DY).cuda()
    x3 = x.reshape(B, S, IN).clone().requires_grad_(True)
    y3 = m(x3)
    assert y3.shape == (B, S, OUT)
    y3.backward(dy.reshape(B, S, OUT))
    g3, gw3 = x3.grad.clone(), m.weight.grad.clone()
    m.weight.grad = None
    x2 = x.clone().requires_grad_(True)
    y2 = m(x2)
    y2.backward(dy)
    assert torch.equal(y3.reshape(B * S, OUT), y2)
    assert torch.equal(g3.reshape(B * S, IN), x2.grad)
    assert torch.equal(gw3, m.weight.grad)


@pytest.mark.parametrize("fmt", [0, 2], ids=["fp32", "packed"])
def test_one_pass_casts_equal_separate_calls(lin, fmt):
    """forward_saving / backward (each activation cast both ways in one pass)
    give exactly the outputs and gradients of forward / dgrad / wgrad, which
    cast each orientation separately; the accumulate form adds into a main grad."""
    T, IN, OUT = 640, 1024, 768
    x = syn.randn((T, IN), seed=syn.SEED_X).cuda()
    dy = syn.randn((T, OUT), seed=syn.SEED_DY).cuda()
    w8 = lin.FP8Weight(syn.randn((OUT, IN), seed=syn.SEED_W, mul=0.02).cuda(), fmt)
    y1, xc = lin.forward_saving(x, w8)
    assert torch.equal(y1, lin.forward(x, w8))
    dx1, dw1 = lin.backward(dy, w8, xc)
    assert torch.equal(dx1, lin.dgrad(dy, w8))
    assert torch.equal(dw1, lin.wgrad(dy, x, fmt, mn_major=True))
    main = syn.randn((OUT, IN), seed=5, dtype=torch.float32, mul=0.1).cuda()
    main2 = main.clone()
    lin.backward(dy, w8, xc, need_dx=False, dw_out=main, accumulate=True)
    lin.wgrad(dy, x, fmt, out=main2, accumulate=True, mn_major=True)
    assert torch.equal(main, main2)


@pytest.mark.parametrize("case", range(12))
def test_linear_mn_major_random_shapes(orc, lin, case):
    """The default layer path (forward_saving + backward: dual casts, NN
    dgrad with W's bytes read MN-major, MN-major wgrad) on seeded ragged
    shapes, token counts from 1 up: every output element within the GEMM
    tolerance of the oracle on the oracle's own casts, which the GPU's casts
    equal bit for bit."""
    rng = np.random.default_rng(12000 + case)
    T = {0: 1, 3: 7}.get(case, int(rng.integers(1, 520)))     # one token, a few tokens, then any
    IN = int(rng.integers(16, 700))
    OUT = int(rng.integers(16, 700))
    fmt = [0, 1, 2][case % 3]
    x = syn.randn_row_exp(T, IN, seed=12100 + case)
    dy = syn.randn((T, OUT), seed=12200 + case)
    w = syn.randn((OUT, IN), seed=12300 + case, mul=0.02)
    w8 = lin.FP8Weight(w.cuda(), fmt, mn_major=True)
    y, xc = lin.forward_saving(x.cuda(), w8)
    dx, dw = lin.backward(dy.cuda(), w8, xc)
    what = f"T={T} IN={IN} OUT={OUT} fmt{fmt}"
    wq, ws = orc.cast_per_block(np_input(w), fmt)
    wtq, wts = orc.cast_per_block(np_input(w).T, fmt)
    xq, xs = orc.cast_per_token(np_input(x), 128, fmt)
    dq, ds = orc.cast_per_token(np_input(dy), 128, fmt)
    aq, sa = orc.cast_per_token(np_input(dy).T, 128, fmt)
    bq, sb = orc.cast_per_token(np_input(x).T, 128, fmt)
    # the cast of X along the tokens kept for the weight gradient, bit for bit
    assert np.array_equal(np_bytes(xc[0]).T, bq), what + ": X's token-axis cast differs"
    check_gemm(y.float().cpu().numpy(), orc.gemm(xq, xs, wq, ws, fmt, out="bf16"), what + " fwd")
    check_gemm(dx.float().cpu().numpy(), orc.gemm(dq, ds, wtq, wts, fmt, out="bf16"), what + " dgrad")
    check_gemm(dw.double().cpu().numpy(), orc.gemm(aq, sa, bq, sb, fmt, b_per_row=True, out="f32"), what + " wgrad")
