"""GPU parity of the FP8 casts against the CPU oracle: bit-exact data and scales.

Cases follow "deep-gemm: fused per-token FP8 cast in Triton
(fused_per_token_cast_to_fp8), version 3" [Results, Tests]: bf16 and fp32
input, group 32 and 128, fp32 / UE8M0 / packed-UE8M0 scales, shapes 1x512,
7x4096, 129x7168, 64x1000 (partial last group), 3000x4096, an all-zero group
and very large values; writing into views of a larger buffer leaves the rest
untouched. Plus the hidden-4096 token sweep and the 128x128 block cast of
"DeepGEMM Essentials: High-Performance FP8 Matrix Multiplication" Part 4.
"""
import numpy as np
import pytest
import torch

from helpers import np_bytes, np_input, np_sf
from quantised_linear_layers_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float32]
GRANS = [32, 128]
FMTS = [0, 1, 2]
MATRIX_SHAPES = [(1, 512), (7, 4096), (129, 7168), (64, 1000), (3000, 4096)]


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from quantised_linear_layers_gb300 import build, ops as o
    build.build()
    o.load_library()
    return o


def make_x(m, n, dtype, gran, huge=True):
    x = syn.randn_row_exp(m, n, seed=syn.SEED_X, dtype=dtype)
    syn.plant_edges(x, gran, zero_group=True, huge_row=(m // 2 if huge and m > 1 else None))
    return x


def assert_cast_equal(orc, ops, x, gran, fmt, recip=False, sf_mn_major=False):
    q, s = ops.fp8_cast_per_token(x.cuda(), gran, fmt, recip=recip, sf_mn_major=sf_mn_major)
    oq, os_ = orc.cast_per_token(np_input(x), gran, fmt, recip=recip)
    gq = np_bytes(q)
    bad = np.argwhere(gq != oq)
    assert bad.size == 0, f"{len(bad)} data bytes differ; first {bad[0]}: gpu {gq[tuple(bad[0])]:#x} oracle {oq[tuple(bad[0])]:#x}"
    gs = np_sf(s)
    assert gs.shape == os_.shape
    assert np.array_equal(gs.view(np.uint32), np.ascontiguousarray(os_).view(np.uint32)), "scale bytes differ"


@pytest.mark.parametrize("shape", MATRIX_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("fmt", FMTS, ids=["fp32", "ue8m0", "packed"])
@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
def test_cast_matrix_60(orc, ops, dtype, gran, fmt, shape):
    m, n = shape
    assert_cast_equal(orc, ops, make_x(m, n, dtype, gran), gran, fmt)


@pytest.mark.parametrize("tokens", [1, 64, 512, 4096, 16384])
@pytest.mark.parametrize("fmt", FMTS, ids=["fp32", "ue8m0", "packed"])
@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
def test_cast_token_sweep_hidden4096(orc, ops, dtype, gran, fmt, tokens):
    assert_cast_equal(orc, ops, make_x(tokens, 4096, dtype, gran), gran, fmt)


@pytest.mark.parametrize("shape", [(7, 4096), (64, 1000), (3000, 4096)])
def test_cast_recip_of_scale_variant(orc, ops, shape):
    assert_cast_equal(orc, ops, make_x(*shape, torch.bfloat16, 128), 128, 0, recip=True)


@pytest.mark.parametrize("fmt", FMTS)
def test_cast_mn_major_scales(orc, ops, fmt):
    x = make_x(129, 7168, torch.bfloat16, 128)
    q, s = ops.fp8_cast_per_token(x.cuda(), 128, fmt, sf_mn_major=True)
    assert s.stride(0) == 1 and s.stride(1) % 4 == 0
    oq, os_ = orc.cast_per_token(np_input(x), 128, fmt)
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np.ascontiguousarray(np_sf(s)).view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
def test_cast_into_views_leaves_rest_untouched(orc, ops, dtype, fmt):
    m, n = 7, 4096
    x = make_x(m, n, dtype, 128)
    parent = syn.random_bytes(16 * 8192, seed=99).cuda()
    ref_parent = parent.clone()
    out = parent.view(16, 8192)[3:3 + m, 128:128 + n].view(torch.float8_e4m3fn)
    cols = -(-n // 128) if fmt != 2 else -(-(-(-n // 128)) // 4)
    sbuf = syn.random_bytes(4 * 40 * 80, seed=98).cuda().view(torch.int32).view(40, 80)
    ref_sbuf = sbuf.clone()
    sview = sbuf[2:2 + m, 1:1 + 2 * cols:2]
    if fmt != 2:
        sview = sview.view(torch.float32)
    ops.fp8_cast_per_token(x.cuda(), 128, fmt, out=out, out_sf=sview)
    oq, os_ = orc.cast_per_token(np_input(x), 128, fmt)
    assert np.array_equal(np_bytes(out), oq)
    assert np.array_equal(np.ascontiguousarray(np_sf(sview)).view(np.uint32), os_.view(np.uint32))
    mask = torch.ones(16, 8192, dtype=torch.bool, device="cuda")
    mask[3:3 + m, 128:128 + n] = False
    assert torch.equal(parent.view(16, 8192)[mask], ref_parent.view(16, 8192)[mask])
    smask = torch.ones(40, 80, dtype=torch.bool, device="cuda")
    smask[2:2 + m, 1:1 + 2 * cols:2] = False
    assert torch.equal(sbuf[smask], ref_sbuf[smask])


@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
@pytest.mark.parametrize("shape", [(4096, 1024), (300, 200), (7168, 640)])
def test_cast_transposed_view(orc, ops, dtype, gran, fmt, shape):
    """Cast of x^T (x_stride_m == 1): the wgrad operands dY^T and X^T."""
    t_rows, feats = shape
    x = make_x(t_rows, feats, dtype, gran, huge=False)
    xt = x.t()                                            # [feats, tokens], stride (1, feats)
    q, s = ops.fp8_cast_per_token(x.cuda().t(), gran, fmt)
    oq, os_ = orc.cast_per_token(np_input(x).T, gran, fmt)
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np.ascontiguousarray(np_sf(s)).view(np.uint32), os_.view(np.uint32))
    assert xt.shape == q.shape


@pytest.mark.parametrize("fmt", FMTS)
def test_cast_generic_strides(orc, ops, fmt):
    base = make_x(64, 2000, torch.bfloat16, 32, huge=False)
    q, s = ops.fp8_cast_per_token(base.cuda()[:, ::2], 32, fmt)   # strides (2000, 2)
    oq, os_ = orc.cast_per_token(np_input(base)[:, ::2], 32, fmt)
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np.ascontiguousarray(np_sf(s)).view(np.uint32), os_.view(np.uint32))


def test_cast_misaligned_rows_take_scalar_path(orc, ops):
    base = make_x(33, 4100, torch.bfloat16, 128, huge=False)
    xv = base[:, 3:3 + 4095]                              # odd offset and width
    q, s = ops.fp8_cast_per_token(base.cuda()[:, 3:3 + 4095], 128, 2)
    oq, os_ = orc.cast_per_token(np_input(base)[:, 3:3 + 4095], 128, 2)
    assert xv.shape == q.shape
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np_sf(s).view(np.uint32), os_.view(np.uint32))


def test_cast_empty_is_noop(ops):
    x = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    q, s = ops.fp8_cast_per_token(x, 128, 0)
    assert q.shape == (0, 512)
    x = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    q, s = ops.fp8_cast_per_token(x, 128, 0)
    assert q.shape == (5, 0)


def test_cast_invalid_arguments(ops):
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.QLError) as e:
        ops.fp8_cast_per_token(x, 64, 0)
    assert e.value.status == 1
    with pytest.raises(ops.QLError):
        ops.fp8_cast_per_token(x, 128, 1, recip=True)
    with pytest.raises(ops.QLError):
        ops.fp8_cast_per_block(x, 3)


# ---------------------------------------------------------------- block cast
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
@pytest.mark.parametrize("shape", [(256, 512), (300, 200), (4096, 7168), (1, 130)])
def test_block_cast(orc, ops, dtype, fmt, shape):
    w = syn.randn(shape, seed=syn.SEED_W, dtype=dtype, mul=0.02)
    if shape[0] > 200:
        w[128:256, 0:128] = 0                             # an all-zero block
    q, s = ops.fp8_cast_per_block(w.cuda(), fmt)
    oq, os_ = orc.cast_per_block(np_input(w), fmt)
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np_sf(s).view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(4096, 7168), (300, 200)])
def test_block_cast_writes_transpose(orc, ops, fmt, shape):
    """cast_per_block(W^T) written in the same pass (dgrad operand); equals the
    oracle's cast of the transposed view."""
    m, n = shape
    w = syn.randn(shape, seed=syn.SEED_W, mul=0.02)
    wt_store = torch.empty((n, m), dtype=torch.float8_e4m3fn, device="cuda")
    st_store = torch.empty((-(-n // 128), -(-m // 128)), dtype=torch.float32, device="cuda")
    ops.fp8_cast_per_block(w.cuda(), fmt, out=wt_store.t(), out_sf=st_store.t())
    oq, os_ = orc.cast_per_block(np.ascontiguousarray(np_input(w).T), fmt)
    assert np.array_equal(np_bytes(wt_store), oq)
    assert np.array_equal(np_sf(st_store).view(np.uint32), os_.view(np.uint32))
    # reading a transposed input view gives the same bytes
    q2, s2 = ops.fp8_cast_per_block(w.cuda().t(), fmt)
    assert torch.equal(q2.view(torch.uint8), wt_store.view(torch.uint8))
    assert torch.equal(s2, st_store)


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
@pytest.mark.parametrize("shape", [(300, 200), (1, 130), (129, 384), (4096, 7168)],
                         ids=lambda s: f"{s[0]}x{s[1]}")
def test_block_cast_recip_of_scale(orc, ops, dtype, shape):
    """QL_CAST_RECIP_OF_SCALE on the block cast and its dual form (factor
    fl32(1 / fl32(amax / 448))): bytes, W's scale grid and W^T's grid all equal
    the oracle's recip branch, on ragged shapes and the 4096 x 7168 weight."""
    w = syn.randn(shape, seed=syn.SEED_W, dtype=dtype, mul=0.02)
    if shape[0] >= 256:
        w[128:256, 0:128] = 0                             # an all-zero block
    oq, os_ = orc.cast_per_block(np_input(w), 0, recip=True)
    q, s = ops.fp8_cast_per_block(w.cuda(), 0, recip=True)
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np_sf(s).view(np.uint32), os_.view(np.uint32))
    qd, sd, sdt = ops.fp8_cast_per_block_dual(w.cuda(), 0, recip=True)
    otq, ots = orc.cast_per_block(np_input(w).T, 0, recip=True)
    assert np.array_equal(np_bytes(qd), oq)
    assert np.array_equal(np_bytes(qd).T, otq)
    assert np.array_equal(np_sf(sd).view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(np_sf(sdt).view(np.uint32), ots.view(np.uint32))


@pytest.mark.parametrize("shape", [(256, 384), (300, 520)], ids=lambda s: f"{s[0]}x{s[1]}")
def test_block_cast_recip_where_readings_differ(orc, ops, shape):
    """fp32 blocks built so that the two readings of the factor give different
    bytes: the kernel follows the oracle in each branch, so the option is not
    ignored, and the transposed-view cast agrees too."""
    import recip_inputs
    x = recip_inputs.sensitive_blocks(*shape, seed=9)
    xt = torch.from_numpy(x)
    for recip in (False, True):
        oq, os_ = orc.cast_per_block(x, 0, recip=recip)
        q, s = ops.fp8_cast_per_block(xt.cuda(), 0, recip=recip)
        assert np.array_equal(np_bytes(q), oq), f"recip={recip}"
        assert np.array_equal(np_sf(s).view(np.uint32), os_.view(np.uint32))
        qt, st = ops.fp8_cast_per_block(xt.cuda().t(), 0, recip=recip)
        otq, ots = orc.cast_per_block(x.T, 0, recip=recip)
        assert np.array_equal(np_bytes(qt), otq) and np.array_equal(np_sf(st).view(np.uint32), ots.view(np.uint32))
    assert not np.array_equal(orc.cast_per_block(x, 0)[0], orc.cast_per_block(x, 0, recip=True)[0])


@pytest.mark.parametrize("gran", GRANS)
def test_token_cast_recip_where_readings_differ(orc, ops, gran):
    """The per-token cast's recip option on rows built so that the two
    readings give different bytes: row, transposed-view and dual kernels."""
    import recip_inputs
    x = recip_inputs.sensitive_rows(130, 520, gran, seed=10)
    xt = torch.from_numpy(x).cuda()
    for recip in (False, True):
        oq, os_ = orc.cast_per_token(x, gran, 0, recip=recip)
        q, s = ops.fp8_cast_per_token(xt, gran, 0, recip=recip)
        assert np.array_equal(np_bytes(q), oq), f"recip={recip}"
        assert np.array_equal(np_sf(s).view(np.uint32), os_.view(np.uint32))
        qt, st = ops.fp8_cast_per_token(xt.t().contiguous().t(), gran, 0, recip=recip)   # column-major input
        assert np.array_equal(np_bytes(qt), oq) and np.array_equal(np_sf(st).view(np.uint32), os_.view(np.uint32))
        if gran == 128:
            qr, sr, qc, sc = ops.fp8_cast_per_token_dual(xt, 0, recip)
            assert np.array_equal(np_bytes(qr), oq)
            assert np.array_equal(np.ascontiguousarray(np_sf(sr)).view(np.uint32), os_.view(np.uint32))
            oqt, ost = orc.cast_per_token(x.T, 128, 0, recip=recip)
            assert np.array_equal(np_bytes(qc).T, oqt)
            assert np.array_equal(np.ascontiguousarray(np_sf(sc)).view(np.uint32),
                                  np.ascontiguousarray(ost).view(np.uint32))
    oq0 = orc.cast_per_token(x, gran, 0)[0]
    assert not np.array_equal(oq0, orc.cast_per_token(x, gran, 0, recip=True)[0])


def test_block_cast_large_weight_ue8m0(orc, ops):
    """The 18432 x 7168 weight of the large cast+GEMM workload, UE8M0."""
    w = syn.randn((18432, 7168), seed=syn.SEED_W, mul=0.02)
    q, s = ops.fp8_cast_per_block(w.cuda(), 1)
    oq, os_ = orc.cast_per_block(np_input(w), 1)
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np_sf(s), os_)


@pytest.mark.parametrize("transposed_input", [False, True])
@pytest.mark.parametrize("shape", [(300, 5 * 128 + 7), (4096, 7168)])
def test_block_cast_packed(orc, ops, shape, transposed_input):
    """Packed UE8M0 block scales (four column blocks per word, pad bytes 0),
    from a row-major or a transposed input view."""
    w = syn.randn(shape, seed=syn.SEED_W, mul=0.02)
    if transposed_input:
        q, s = ops.fp8_cast_per_block(w.cuda().t(), 2)
        oq, os_ = orc.cast_per_block(np_input(w).T, 2)
    else:
        q, s = ops.fp8_cast_per_block(w.cuda(), 2)
        oq, os_ = orc.cast_per_block(np_input(w), 2)
    assert np.array_equal(np_bytes(q), oq)
    assert np.array_equal(np_sf(s).view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("fmt", FMTS, ids=["fp32", "ue8m0", "packed"])
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
@pytest.mark.parametrize("shape", [(4096, 1024), (300, 200), (300, 336), (7168, 640), (130, 36), (1, 24)],
                         ids=lambda s: f"{s[0]}x{s[1]}")
def test_cast_column_major_in_and_out(orc, ops, dtype, gran, fmt, shape):
    """Cast of x^T written as q^T (x_stride_m == out_stride_m == 1): groups run
    down the columns of the physical [tokens, features] array and the E4M3
    output keeps that layout (the MN-major GEMM operand); ragged token counts,
    ragged and narrow feature counts, all-zero and huge groups."""
    t_rows, feats = shape
    x = make_x(t_rows, feats, dtype, gran, huge=False)
    x[min(5, t_rows - 1), :] = 3.0e38 if t_rows > 1 else x[0, :]
    q_phys = torch.empty((t_rows, feats), dtype=torch.float8_e4m3fn, device="cuda")
    q, s = ops.fp8_cast_per_token(x.cuda().t(), gran, fmt, out=q_phys.t(), sf_mn_major=True)
    oq, os_ = orc.cast_per_token(np_input(x).T, gran, fmt)
    assert np.array_equal(np_bytes(q_phys).T, oq), "E4M3 bytes differ"
    gs = np_sf(s)
    if fmt == 2:
        assert np.array_equal(np.ascontiguousarray(gs), os_)
    else:
        assert np.array_equal(np.ascontiguousarray(gs).view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("fmt", FMTS, ids=["fp32", "ue8m0", "packed"])
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
def test_cast_column_major_subnormal_and_signed_zero(orc, ops, dtype, gran, fmt):
    """Column-major cast over a group of subnormal inputs, a group of negative
    zeros with one negative subnormal, and one value near the format's maximum:
    the amax the kernel reduces (bf16 pairs, for bf16 input) must be the
    maximum of |x| exactly as defined, so bytes and scales match the oracle."""
    t_rows, feats = 384, 256
    x = syn.randn((t_rows, feats), seed=77, dtype=torch.float32)
    x[:128, :64] *= 1e-39
    x[128:256, 64:128] = -0.0
    x[130, 70] = -5.0e-39
    x[300, 200] = -2.5e38
    x = x.to(dtype)
    q_phys = torch.empty((t_rows, feats), dtype=torch.float8_e4m3fn, device="cuda")
    q, s = ops.fp8_cast_per_token(x.cuda().t(), gran, fmt, out=q_phys.t(), sf_mn_major=True)
    oq, os_ = orc.cast_per_token(np_input(x).T, gran, fmt)
    assert np.array_equal(np_bytes(q_phys).T, oq), "E4M3 bytes differ"
    gs = np.ascontiguousarray(np_sf(s))
    if fmt == 2:
        assert np.array_equal(gs, os_)
    else:
        assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("feats", [208, 200])
@pytest.mark.parametrize("fmt", [0, 2], ids=["fp32", "packed"])
def test_cast_column_major_into_view(orc, ops, fmt, feats):
    """Column-major cast written into a view of a wider buffer (row pitch 256
    bytes): with 208 features the view's rows start and end on 16-byte
    boundaries and the E4M3 rows leave through TMA tile stores, with 200 they
    end mid-chunk and are stored directly. The bytes outside the view keep
    their canary and the view matches the oracle."""
    t_rows = 300
    x = make_x(t_rows, feats, torch.bfloat16, 128, huge=False)
    parent = torch.full((t_rows + 8, 256), 0x5A, dtype=torch.uint8, device="cuda")
    view = parent[:t_rows, :feats].view(torch.float8_e4m3fn)
    _, s = ops.fp8_cast_per_token(x.cuda().t(), 128, fmt, out=view.t(), sf_mn_major=True)
    oq, os_ = orc.cast_per_token(np_input(x).T, 128, fmt)
    p = parent.cpu().numpy()
    assert np.all(p[:, feats:] == 0x5A) and np.all(p[t_rows:] == 0x5A)
    assert np.array_equal(p[:t_rows, :feats].T, oq)
    gs = np.ascontiguousarray(np_sf(s))
    if fmt == 2:
        assert np.array_equal(gs, os_)
    else:
        assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("fmt,recip", [(0, False), (0, True), (1, False), (2, False)],
                         ids=["fp32", "fp32-recip", "ue8m0", "packed"])
@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f32"])
@pytest.mark.parametrize("shape", [(4096, 1024), (300, 200), (300, 336), (129, 7168), (1, 24), (640, 4096),
                                   (4096, 7168), (3000, 4100), (3000, 4104)],
                         ids=lambda s: f"{s[0]}x{s[1]}")
def test_cast_dual_per_token(orc, ops, dtype, fmt, recip, shape):
    """fp8_cast_per_token_dual: from one read of x [T, C], the per-token cast of
    x and that of x^T (kept in x's layout), each bit for bit the oracle's cast,
    with partial tiles in both directions, an all-zero group and huge values
    (3000 x 4104: ragged tiles with 16-byte aligned bf16 rows; 3000 x 4100:
    rows off that alignment, read element by element)."""
    t_rows, feats = shape
    x = make_x(t_rows, feats, dtype, 128, huge=t_rows > 1)
    qr, sr, qc, sc = ops.fp8_cast_per_token_dual(x.cuda(), fmt, recip)
    assert ops.device_status() == 0
    oq, os_ = orc.cast_per_token(np_input(x), 128, fmt, recip=recip)
    assert np.array_equal(np_bytes(qr), oq), "row-cast bytes differ"
    oqt, ost = orc.cast_per_token(np_input(x).T, 128, fmt, recip=recip)
    assert np.array_equal(np_bytes(qc).T, oqt), "column-cast bytes differ"
    for got, want in ((sr, os_), (sc, ost)):
        g = np.ascontiguousarray(np_sf(got))
        if fmt == 2:
            assert np.array_equal(g, want)
        else:
            assert np.array_equal(g.view(np.uint32), np.ascontiguousarray(want).view(np.uint32))


@pytest.mark.parametrize("fmt", [0, 2], ids=["fp32", "packed"])
def test_cast_dual_unaligned_rows_many_tiles(orc, ops, fmt):
    """A view whose rows do not start on 16-byte boundaries (no prefetch path)
    with more tiles than resident CTAs: bit for bit the oracle's two casts."""
    base = syn.randn_row_exp(2600, 4101, dtype=torch.bfloat16)
    x = base[:, 1:4100]
    xg = base.cuda()[:, 1:4100]             # row stride 4101 elements, offset one element
    assert xg.stride(0) == 4101
    qr, sr, qc, sc = ops.fp8_cast_per_token_dual(xg, fmt)
    assert ops.device_status() == 0
    oq, os_ = orc.cast_per_token(np_input(x), 128, fmt)
    oqt, ost = orc.cast_per_token(np_input(x).T, 128, fmt)
    assert np.array_equal(np_bytes(qr), oq) and np.array_equal(np_bytes(qc).T, oqt)
    for got, want in ((sr, os_), (sc, ost)):
        g = np.ascontiguousarray(np_sf(got))
        assert np.array_equal(g.view(np.uint32), np.ascontiguousarray(want).view(np.uint32))
