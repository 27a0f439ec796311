"""Thin ctypes binding over libqlinear.so (include/qlinear.h).

Argument marshalling only: every step of the cast and the GEMM runs in the
library's CUDA kernels. torch supplies device memory and the current stream.
If the library is missing or cannot be loaded every op raises; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# QL_LIBRARY selects another build of the library (the bounds-checked
# libqlinear_bounds.so, for instance); the default is the product build.
LIB_PATH = os.environ.get("QL_LIBRARY") or os.path.join(_HERE, "libqlinear.so")

QL_BF16, QL_F32 = 0, 1
SF_FP32, SF_UE8M0, SF_PACKED_UE8M0 = 0, 1, 2
CAST_RECIP_OF_SCALE = 0x100

_lock = threading.Lock()
_lib = None

_i64, _vp, _int, _sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

_SIGS = {
    "fp8_cast_per_token": [_vp, _int, _i64, _i64, _i64, _i64, _int, _int, _vp, _i64, _i64, _vp, _i64, _i64, _vp],
    "fp8_cast_per_block": [_vp, _int, _i64, _i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64, _i64, _vp],
    "fp8_cast_per_token_dual": [_vp, _int, _i64, _i64, _i64, _int, _vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp,
                                _i64, _i64, _vp],
    "fp8_cast_per_block_dual": [_vp, _int, _i64, _i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64, _i64,
                                _vp, _i64, _i64, _vp],
    "gemm_fp8_nt_bf16": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                         _i64, _i64, _i64, _vp, _sz, _vp],
    "gemm_fp8_wgrad_fp32": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                            _i64, _i64, _i64, _int, _vp, _sz, _vp],
    "m_grouped_gemm_fp8_nt_bf16_contiguous": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _i64,
                                              _int, _vp, _i64, _vp, _int, _i64, _i64, _i64, _vp],
    "ql_get_m_alignment_for_contiguous_layout": [],
    "gemm_fp8_nt_fp8out": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64, _vp, _i64,
                           _i64, _int, _int, _i64, _i64, _i64, _vp],
    "gemm_fp8_wgrad_fp32_mn": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                               _i64, _i64, _i64, _int, _vp],
    "gemm_fp8_nn_bf16": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                         _i64, _i64, _i64, _vp],
    "ql_cast_gemm_host_workspace_size": [_i64, _i64, _i64, _int],
    "ql_cast_gemm_host": [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64, _i64, _i64, _i64, _i64,
                          _vp, _sz, _vp],
    "ql_cast_gemm_host_noalloc": [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64, _i64, _i64, _i64, _i64,
                                  _vp],
    "ql_gemm_workspace_size": [_i64, _i64, _i64],
    "ql_set_num_sms": [_int],
    "ql_get_num_sms": [],
    "ql_binary_version": [],
    "ql_set_wait_limit_ms": [_int],
    "ql_set_gemm_block_n": [_int],
    "ql_set_gemm_path": [_int],
    "ql_test_stall_gemm_producer": [_int],
    "ql_device_status": [_vp],
    "ql_device_status_detail": [_vp, _vp, _vp],
    "ql_bounds_checked": [],
    "ql_status_string": [_int],
}


class QLError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg}")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load libqlinear.so (raises if it is missing: no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libqlinear.so not found at {path}; run quantised_linear_layers_gb300.build.build()")
            lib = ctypes.CDLL(path)
            for name, args in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = _int
            lib.ql_status_string.restype = ctypes.c_char_p
            lib.ql_gemm_workspace_size.restype = _sz
            lib.ql_cast_gemm_host_workspace_size.restype = _sz
            _lib = lib
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        msg = load_library().ql_status_string(status).decode()
        raise QLError(fn, status, msg)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _dtype_code(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return QL_BF16
    if x.dtype == torch.float32:
        return QL_F32
    raise TypeError(f"input must be bfloat16 or float32, got {x.dtype}")


def _bytes8(t: torch.Tensor) -> torch.Tensor:
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"expected an E4M3 (float8_e4m3fn or uint8) tensor, got {t.dtype}")
    return t


def _ceil(a: int, b: int) -> int:
    return -(-a // b)


def sf_shape(n: int, gran_k: int, fmt: int) -> int:
    """Number of scale columns per row: groups, or int32 words for packed UE8M0."""
    g = _ceil(n, gran_k)
    return _ceil(g, 4) if (fmt & 0xFF) == SF_PACKED_UE8M0 else g


def empty_sf(m: int, cols: int, fmt: int, device, mn_major: bool = False) -> torch.Tensor:
    """Scale tensor [m, cols]; mn_major gives the M-major, TMA-aligned layout
    (stride (1, align(m, 4)))."""
    dt = torch.int32 if (fmt & 0xFF) == SF_PACKED_UE8M0 else torch.float32
    if not mn_major:
        return torch.empty((m, cols), dtype=dt, device=device)
    ld = _ceil(max(m, 1), 4) * 4
    return torch.empty((cols, ld), dtype=dt, device=device).t()[:m]


def fp8_cast_per_token(x: torch.Tensor, gran_k: int = 128, fmt: int = SF_FP32, recip: bool = False,
                       out: torch.Tensor | None = None, out_sf: torch.Tensor | None = None,
                       sf_mn_major: bool = False):
    """Per-token FP8 cast of a 2-D bf16/fp32 tensor (any strides).

    Returns (data float8_e4m3fn [m, n], scales). ``out`` / ``out_sf`` may be
    views of larger buffers; only their elements are written."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D")
    m, n = x.shape
    if out is None:
        out = torch.empty((m, n), dtype=torch.float8_e4m3fn, device=x.device)
    if out_sf is None:
        out_sf = empty_sf(m, sf_shape(n, gran_k, fmt), fmt, x.device, sf_mn_major)
    _bytes8(out)
    code = fmt | (CAST_RECIP_OF_SCALE if recip else 0)
    st = load_library().fp8_cast_per_token(
        x.data_ptr(), _dtype_code(x), m, n, x.stride(0), x.stride(1), gran_k, code,
        out.data_ptr(), out.stride(0), out.stride(1), out_sf.data_ptr(), out_sf.stride(0), out_sf.stride(1),
        _stream(x))
    _check("fp8_cast_per_token", st)
    return out, out_sf


def fp8_cast_per_block(x: torch.Tensor, fmt: int = SF_FP32, recip: bool = False,
                       out: torch.Tensor | None = None, out_sf: torch.Tensor | None = None):
    """128x128 block FP8 cast. Returns (data [m, n], scales fp32 [ceil(m/128), ceil(n/128)],
    or int32 words [ceil(m/128), ceil(ceil(n/128)/4)] packed along the column blocks
    for SF_PACKED_UE8M0). ``out`` / ``out_sf`` may be transposed views (e.g.
    ``wt.t()``) to write W^T's cast."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D")
    m, n = x.shape
    if out is None:
        out = torch.empty((m, n), dtype=torch.float8_e4m3fn, device=x.device)
    if out_sf is None:
        cols = _ceil(n, 128)
        if fmt == SF_PACKED_UE8M0:
            out_sf = torch.empty((_ceil(m, 128), _ceil(cols, 4)), dtype=torch.int32, device=x.device)
        else:
            out_sf = torch.empty((_ceil(m, 128), cols), dtype=torch.float32, device=x.device)
    _bytes8(out)
    code = fmt | (CAST_RECIP_OF_SCALE if recip else 0)
    st = load_library().fp8_cast_per_block(
        x.data_ptr(), _dtype_code(x), m, n, x.stride(0), x.stride(1), code,
        out.data_ptr(), out.stride(0), out.stride(1), out_sf.data_ptr(), out_sf.stride(0), out_sf.stride(1),
        _stream(x))
    _check("fp8_cast_per_block", st)
    return out, out_sf


def fp8_cast_per_token_dual(x: torch.Tensor, fmt: int = SF_FP32, recip: bool = False):
    """Both per-token casts of x [T, C] from one read (1x128 groups): returns
    (q_rows [T, C], s_rows [T, ceil(C/128)] M-major) = fp8_cast_per_token(x)
    and (q_cols [T, C], s_cols [C, ceil(T/128)] M-major), the cast of x^T kept
    in x's layout (the MN-major weight-gradient operand). E4M3 rows start on
    16-byte boundaries; their padding is never written or read."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with contiguous rows")
    t, c = x.shape
    ld = _ceil(max(c, 1), 16) * 16
    q_rows = torch.empty((t, ld), dtype=torch.float8_e4m3fn, device=x.device)[:, :c]
    q_cols = torch.empty((t, ld), dtype=torch.float8_e4m3fn, device=x.device)[:, :c]
    s_rows = empty_sf(t, sf_shape(c, 128, fmt), fmt, x.device, mn_major=True)
    s_cols = empty_sf(c, sf_shape(t, 128, fmt), fmt, x.device, mn_major=True)
    code = fmt | (CAST_RECIP_OF_SCALE if recip else 0)
    st = load_library().fp8_cast_per_token_dual(
        x.data_ptr(), _dtype_code(x), t, c, x.stride(0), code,
        q_rows.data_ptr(), q_rows.stride(0), s_rows.data_ptr(), s_rows.stride(0), s_rows.stride(1),
        q_cols.data_ptr(), q_cols.stride(0), s_cols.data_ptr(), s_cols.stride(0), s_cols.stride(1), _stream(x))
    _check("fp8_cast_per_token_dual", st)
    return q_rows, s_rows, q_cols, s_cols


def fp8_cast_per_block_dual(x: torch.Tensor, fmt: int = SF_FP32, recip: bool = False):
    """fp8_cast_per_block plus, from the same pass, the scale grid of the
    transposed cast (equal to fp8_cast_per_block(x.t())'s scales): returns
    (data [m, n], scales of x, scales of x^T). With the data read MN-major,
    the second grid is the data-gradient operand of gemm_fp8_nn_bf16. The
    data's rows start on 16-byte boundaries (the GEMMs' operand rows must),
    whatever n is; the padding bytes are never written or read."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D")
    m, n = x.shape
    ld = _ceil(max(n, 1), 16) * 16
    out = torch.empty((m, ld), dtype=torch.float8_e4m3fn, device=x.device)[:, :n]
    rb, cb = _ceil(m, 128), _ceil(n, 128)
    if fmt == SF_PACKED_UE8M0:
        out_sf = torch.empty((rb, _ceil(cb, 4)), dtype=torch.int32, device=x.device)
        out_sf_t = torch.empty((cb, _ceil(rb, 4)), dtype=torch.int32, device=x.device)
    else:
        out_sf = torch.empty((rb, cb), dtype=torch.float32, device=x.device)
        out_sf_t = torch.empty((cb, rb), dtype=torch.float32, device=x.device)
    code = fmt | (CAST_RECIP_OF_SCALE if recip else 0)
    st = load_library().fp8_cast_per_block_dual(
        x.data_ptr(), _dtype_code(x), m, n, x.stride(0), x.stride(1), code,
        out.data_ptr(), out.stride(0), out.stride(1), out_sf.data_ptr(), out_sf.stride(0), out_sf.stride(1),
        out_sf_t.data_ptr(), out_sf_t.stride(0), out_sf_t.stride(1), _stream(x))
    _check("fp8_cast_per_block_dual", st)
    return out, out_sf, out_sf_t


def _gemm_args(a, sfa, b, sfb):
    _bytes8(a)
    _bytes8(b)
    if a.dim() != 2 or b.dim() != 2 or a.stride(1) != 1 or b.stride(1) != 1:
        raise ValueError("a and b must be 2-D with contiguous K")
    if a.shape[1] != b.shape[1]:
        raise ValueError("a and b must share K")
    return a.shape[0], b.shape[0], a.shape[1]


def gemm_fp8_nt_bf16(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor,
                     fmt: int = SF_FP32, out: torch.Tensor | None = None) -> torch.Tensor:
    """D = A B^T, bf16 [m, n]: A [m, k] with 1x128 scales sfa [m, ceil(k/128)],
    B [n, k] with 128x128 scales sfb [ceil(n/128), ceil(k/128)] (packed UE8M0:
    int32 words along K)."""
    m, n, k = _gemm_args(a, sfa, b, sfb)
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    if out.dtype != torch.bfloat16 or out.stride(1) != 1:
        raise ValueError("out must be bf16 with contiguous rows")
    st = load_library().gemm_fp8_nt_bf16(
        a.data_ptr(), a.stride(0), sfa.data_ptr(), sfa.stride(0), sfa.stride(1),
        b.data_ptr(), b.stride(0), sfb.data_ptr(), sfb.stride(0), sfb.stride(1),
        fmt, out.data_ptr(), out.stride(0), m, n, k, None, 0, _stream(a))
    _check("gemm_fp8_nt_bf16", st)
    return out


def gemm_fp8_nt_fp8out(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor,
                       fmt: int = SF_FP32, gran_k: int = 128, out_fmt: int = SF_FP32, recip: bool = False,
                       out: torch.Tensor | None = None, out_sf: torch.Tensor | None = None,
                       sf_mn_major: bool = False):
    """D = A B^T cast per token inside the GEMM: returns (E4M3 [m, n], scales),
    equal to fp8_cast_per_token(gemm_fp8_nt_bf16(...), gran_k, out_fmt)."""
    m, n, k = _gemm_args(a, sfa, b, sfb)
    if out is None:
        out = torch.empty((m, n), dtype=torch.float8_e4m3fn, device=a.device)
    _bytes8(out)
    if out.stride(1) != 1:
        raise ValueError("out must have contiguous rows")
    if out_sf is None:
        out_sf = empty_sf(m, sf_shape(n, gran_k, out_fmt), out_fmt, a.device, mn_major=sf_mn_major)
    code = out_fmt | (CAST_RECIP_OF_SCALE if recip else 0)
    st = load_library().gemm_fp8_nt_fp8out(
        a.data_ptr(), a.stride(0), sfa.data_ptr(), sfa.stride(0), sfa.stride(1),
        b.data_ptr(), b.stride(0), sfb.data_ptr(), sfb.stride(0), sfb.stride(1),
        fmt, out.data_ptr(), out.stride(0), out_sf.data_ptr(), out_sf.stride(0), out_sf.stride(1),
        gran_k, code, m, n, k, _stream(a))
    _check("gemm_fp8_nt_fp8out", st)
    return out, out_sf


def gemm_fp8_wgrad_fp32(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor,
                        out: torch.Tensor | None = None, accumulate: bool = False,
                        fmt: int = SF_FP32) -> torch.Tensor:
    """D (+)= A B^T, fp32 [m, n]: both operands with 1x128 per-row scales along K."""
    m, n, k = _gemm_args(a, sfa, b, sfb)
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs an existing out")
        out = torch.empty((m, n), dtype=torch.float32, device=a.device)
    if out.dtype != torch.float32 or out.stride(1) != 1:
        raise ValueError("out must be fp32 with contiguous rows")
    st = load_library().gemm_fp8_wgrad_fp32(
        a.data_ptr(), a.stride(0), sfa.data_ptr(), sfa.stride(0), sfa.stride(1),
        b.data_ptr(), b.stride(0), sfb.data_ptr(), sfb.stride(0), sfb.stride(1),
        fmt, out.data_ptr(), out.stride(0), m, n, k, int(bool(accumulate)), None, 0, _stream(a))
    _check("gemm_fp8_wgrad_fp32", st)
    return out


def m_grouped_gemm_fp8_nt_bf16_contiguous(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor,
                                          sfb: torch.Tensor, m_indices: torch.Tensor, fmt: int = SF_FP32,
                                          out: torch.Tensor | None = None) -> torch.Tensor:
    """Grouped D = A B_e^T over the contiguous layout: A [m, k] (m a multiple of
    128) with 1x128 scales, B [G, n, k] with scales sfb [G, ceil(n/128),
    ceil(k/128)], m_indices int32 [m] (expert per row, -1 for padding rows,
    which are left unwritten in ``out``)."""
    _bytes8(a)
    _bytes8(b)
    if a.dim() != 2 or b.dim() != 3 or a.stride(1) != 1 or b.stride(2) != 1:
        raise ValueError("a must be [m, k] and b [G, n, k], both with contiguous K")
    if b.stride(0) != b.shape[1] * b.stride(1):
        raise ValueError("b's experts must be stacked without gaps (stride(0) == n * stride(1))")
    if a.shape[1] != b.shape[2] or sfb.dim() != 3 or sfb.shape[0] != b.shape[0]:
        raise ValueError("shapes of a, b and sfb do not agree")
    if m_indices.dtype != torch.int32 or m_indices.dim() != 1 or m_indices.shape[0] != a.shape[0] \
            or not m_indices.is_contiguous() or m_indices.device != a.device:
        raise ValueError("m_indices must be a contiguous int32 [m] tensor on a's device")
    m, k = a.shape
    G, n = b.shape[0], b.shape[1]
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    if out.dtype != torch.bfloat16 or out.stride(1) != 1:
        raise ValueError("out must be bf16 with contiguous rows")
    st = load_library().m_grouped_gemm_fp8_nt_bf16_contiguous(
        a.data_ptr(), a.stride(0), sfa.data_ptr(), sfa.stride(0), sfa.stride(1),
        b.data_ptr(), b.stride(1), sfb.data_ptr(), sfb.stride(0), sfb.stride(1), sfb.stride(2),
        fmt, out.data_ptr(), out.stride(0), m_indices.data_ptr(), G, m, n, k, _stream(a))
    _check("m_grouped_gemm_fp8_nt_bf16_contiguous", st)
    return out


def get_m_alignment_for_contiguous_layout() -> int:
    return int(load_library().ql_get_m_alignment_for_contiguous_layout())


def gemm_fp8_wgrad_fp32_mn(a_t: torch.Tensor, sfa: torch.Tensor, b_t: torch.Tensor, sfb: torch.Tensor,
                           out: torch.Tensor | None = None, accumulate: bool = False,
                           fmt: int = SF_FP32) -> torch.Tensor:
    """D [m, n] (+)= A B^T, fp32, with both operands given K-outer: a_t [k, m]
    and b_t [k, n] (contiguous rows); sfa [m, ceil(k/128)], sfb [n, ceil(k/128)]."""
    _bytes8(a_t)
    _bytes8(b_t)
    if a_t.dim() != 2 or b_t.dim() != 2 or a_t.stride(1) != 1 or b_t.stride(1) != 1:
        raise ValueError("a_t and b_t must be 2-D with contiguous rows")
    if a_t.shape[0] != b_t.shape[0]:
        raise ValueError("a_t and b_t must share K (their first dimension)")
    k, m = a_t.shape
    n = b_t.shape[1]
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs an existing out")
        out = torch.empty((m, n), dtype=torch.float32, device=a_t.device)
    if out.dtype != torch.float32 or out.stride(1) != 1:
        raise ValueError("out must be fp32 with contiguous rows")
    st = load_library().gemm_fp8_wgrad_fp32_mn(
        a_t.data_ptr(), a_t.stride(0), sfa.data_ptr(), sfa.stride(0), sfa.stride(1),
        b_t.data_ptr(), b_t.stride(0), sfb.data_ptr(), sfb.stride(0), sfb.stride(1),
        fmt, out.data_ptr(), out.stride(0), m, n, k, int(bool(accumulate)), _stream(a_t))
    _check("gemm_fp8_wgrad_fp32_mn", st)
    return out


def gemm_fp8_nn_bf16(a: torch.Tensor, sfa: torch.Tensor, b_kn: torch.Tensor, sfb: torch.Tensor,
                     fmt: int = SF_FP32, out: torch.Tensor | None = None) -> torch.Tensor:
    """D = A B, bf16 [m, n]: A [m, k] with 1x128 scales, B given as [k, n]
    (contiguous rows) with 128x128 scales sfb [ceil(n/128), ceil(k/128)] (any strides)."""
    _bytes8(a)
    _bytes8(b_kn)
    if a.dim() != 2 or b_kn.dim() != 2 or a.stride(1) != 1 or b_kn.stride(1) != 1:
        raise ValueError("a and b_kn must be 2-D with contiguous rows")
    if a.shape[1] != b_kn.shape[0]:
        raise ValueError("a [m, k] and b_kn [k, n] must share K")
    m, k = a.shape
    n = b_kn.shape[1]
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    if out.dtype != torch.bfloat16 or out.stride(1) != 1:
        raise ValueError("out must be bf16 with contiguous rows")
    st = load_library().gemm_fp8_nn_bf16(
        a.data_ptr(), a.stride(0), sfa.data_ptr(), sfa.stride(0), sfa.stride(1),
        b_kn.data_ptr(), b_kn.stride(0), sfb.data_ptr(), sfb.stride(0), sfb.stride(1),
        fmt, out.data_ptr(), out.stride(0), m, n, k, _stream(a))
    _check("gemm_fp8_nn_bf16", st)
    return out


def cast_gemm_host_workspace_size(n: int, k: int, chunk_rows: int, fmt: int) -> int:
    return int(load_library().ql_cast_gemm_host_workspace_size(n, k, chunk_rows, fmt))


def cast_gemm_host(x_host: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor, fmt: int, out_host: torch.Tensor,
                   chunk_rows: int, workspace: torch.Tensor) -> torch.Tensor:
    """out_host [m, n] = bf16(cast_per_token(x_host) @ b^T) with x_host / out_host
    bf16 tensors in host memory (pinned for overlap), b / sfb on the device and
    a device workspace of cast_gemm_host_workspace_size bytes; copies and
    kernels of successive row chunks overlap. Stream-ordered on the current stream."""
    if x_host.device.type != "cpu" or out_host.device.type != "cpu":
        raise ValueError("x_host and out_host must be host tensors")
    if x_host.dtype != torch.bfloat16 or out_host.dtype != torch.bfloat16:
        raise ValueError("x_host and out_host must be bf16")
    if x_host.stride(1) != 1 or out_host.stride(1) != 1 or b.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    _bytes8(b)
    m, k = x_host.shape
    n = b.shape[0]
    if b.shape[1] != k or tuple(out_host.shape) != (m, n):
        raise ValueError("shapes of x_host, b and out_host do not agree")
    if not workspace.is_cuda or workspace.device != b.device:
        raise ValueError("workspace must be device memory on b's device")
    st = load_library().ql_cast_gemm_host(
        x_host.data_ptr(), x_host.stride(0), b.data_ptr(), b.stride(0), sfb.data_ptr(), sfb.stride(0), sfb.stride(1),
        fmt, out_host.data_ptr(), out_host.stride(0), m, n, k, chunk_rows,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(b))
    _check("ql_cast_gemm_host", st)
    return out_host


def set_num_sms(n: int) -> None:
    _check("ql_set_num_sms", load_library().ql_set_num_sms(int(n)))


def get_num_sms() -> int:
    return int(load_library().ql_get_num_sms())


def set_gemm_block_n(bn: int) -> None:
    _check("ql_set_gemm_block_n", load_library().ql_set_gemm_block_n(int(bn)))


def set_gemm_path(path: int) -> None:
    """GEMM kernel choice (ql_set_gemm_path): 0 auto; CUDA-core promotion: 1
    (default kernel), 5 on CTA pairs, 6 on one SM per tile, 7 split-K over a
    cluster where a split applies; block-scaled MMA (UE8M0 formats): 2 on one
    SM per tile, 3 on CTA pairs, 4 split-K over a cluster where it applies."""
    _check("ql_set_gemm_path", load_library().ql_set_gemm_path(int(path)))


def test_stall_gemm_producer(enable: bool) -> None:
    """Failure-path test hook: GEMM producers issue no copies while enabled."""
    _check("ql_test_stall_gemm_producer", load_library().ql_test_stall_gemm_producer(int(bool(enable))))


def set_wait_limit_ms(ms: int) -> None:
    _check("ql_set_wait_limit_ms", load_library().ql_set_wait_limit_ms(int(ms)))


def device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status code."""
    s = torch.cuda.current_stream(device).cuda_stream
    return int(load_library().ql_device_status(s))
