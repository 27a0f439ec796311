"""numpy wrappers over the plain-C oracle (``qlinear_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring). Every wrapper takes
numpy arrays; bf16 data is passed as its raw ``uint16`` bit patterns so the C
code sees exactly the bytes the GPU sees.

Functions and the passages they follow:
  e4m3_encode / e4m3_decode  OCP FP8 E4M3FN definition (round to nearest even)
  cast_per_token  "DeepGEMM Essentials: High-Performance FP8 Matrix
                  Multiplication" Part 3, with the gran_k / UE8M0 / packed-UE8M0
                  options of "deep-gemm: fused per-token FP8 cast in Triton
                  (fused_per_token_cast_to_fp8), version 3"
  cast_per_block  "DeepGEMM Essentials" Part 4
  gemm            "DeepGEMM Essentials" Parts 6 and 12-13; RHS scales read
                  row-wise per "[Help] Starter script for nn.Linear for
                  fwd,bwd" (maintainer's reply on RHS scales)
  gemm_m_grouped_contiguous
                  "DeepGEMM Essentials" Parts 8-11: each row of the
                  contiguous token matrix times its expert's B; rows marked
                  -1 are padding and are not computed

Parity unpinned: the byte order of packed UE8M0 words (the pages never print
it; little-endian, group j in byte j % 4 of word j // 4, is the reading).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16, F32 = 0, 1
SF_FP32, SF_UE8M0, SF_PACKED_UE8M0 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlinear_oracle.c")
_SO = os.path.join(_HERE, "_qlinear_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE: no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            lib.oracle_e4m3_encode_f32_array.argtypes = [_vp, _i64, _vp]
            lib.oracle_e4m3_decode_array.argtypes = [_vp, _i64, _vp]
            lib.oracle_overflow_count.restype = ctypes.c_longlong
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_cast_per_token.restype = ctypes.c_int
            lib.oracle_cast_per_token.argtypes = [
                _vp, ctypes.c_int, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _vp, _i64, _i64, _vp, _i64, _i64]
            lib.oracle_cast_per_block.restype = ctypes.c_int
            lib.oracle_cast_per_block.argtypes = [
                _vp, ctypes.c_int, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int,
                _vp, _i64, _i64, _vp, _i64, _i64]
            lib.oracle_round_bf16.restype = ctypes.c_double
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_array.argtypes = [_vp, _i64, ctypes.c_int]
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_gemm.argtypes = [
                _vp, _i64, _vp, _i64, _i64,
                _vp, _i64, _vp, _i64, _i64,
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _i64, _i64, _i64, _vp, _i64,
                _vp, _i64, _vp, _i64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def overflow_count() -> int:
    return int(_load().oracle_overflow_count())


def reset_overflow_count() -> None:
    _load().oracle_reset_overflow_count()


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(t: int) -> None:
    _load().oracle_set_num_threads(int(t))


def e4m3_encode(v) -> np.ndarray:
    """E4M3FN bytes of fp32 values (round to nearest even)."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_f32_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(b) -> np.ndarray:
    """Values (float64) of E4M3FN bytes."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint8))
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_e4m3_decode_array(_ptr(b), b.size, _ptr(out))
    return out


def round_output(v: np.ndarray, out: str) -> np.ndarray:
    """Round exact (float64) results to the GEMM's output type: 'bf16' (round
    to nearest even from the exact value), 'f32' (RNE) or 'f64' (unchanged)."""
    v = np.array(v, dtype=np.float64, copy=True, order="C")
    mode = {"f64": 0, "bf16": 1, "f32": 2}[out]
    if mode:
        _load().oracle_round_array(_ptr(v), v.size, mode)
    return v


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return F32
    raise TypeError("x must be uint16 (bf16 bits) or float32")


def _elem_strides(a: np.ndarray):
    return tuple(s // a.itemsize for s in a.strides)


def cast_per_token(x: np.ndarray, gran: int, fmt: int, recip: bool = False,
                   out: np.ndarray | None = None, out_sf: np.ndarray | None = None):
    """Per-token cast of a 2-D array (any strides). Returns (data uint8 [m,n], scales).

    Scales are float32 [m, ceil(n/gran)] for fmt 0/1, int32 [m, ceil(G/4)] packed.
    ``out`` / ``out_sf`` may be strided views (written in place)."""
    m, n = x.shape
    G = -(-n // gran)
    if out is None:
        out = np.empty((m, n), dtype=np.uint8)
    if out_sf is None:
        out_sf = (np.empty((m, G), dtype=np.float32) if fmt != SF_PACKED_UE8M0
                  else np.empty((m, -(-G // 4)), dtype=np.int32))
    sx, so, ss = _elem_strides(x), _elem_strides(out), _elem_strides(out_sf)
    rc = _load().oracle_cast_per_token(_ptr(x), _dtype_code(x), m, n, sx[0], sx[1], gran, fmt,
                                       int(bool(recip)), _ptr(out), so[0], so[1],
                                       _ptr(out_sf), ss[0], ss[1])
    if rc != 0:
        raise ValueError("oracle_cast_per_token: bad arguments")
    return out, out_sf


def cast_per_block(x: np.ndarray, fmt: int, recip: bool = False,
                   out: np.ndarray | None = None, out_sf: np.ndarray | None = None):
    """128x128 block cast. Returns (data uint8 [m,n], scales float32 [ceil(m/128), ceil(n/128)],
    or int32 words [ceil(m/128), ceil(ceil(n/128)/4)] packed along column blocks for fmt 2)."""
    m, n = x.shape
    if out is None:
        out = np.empty((m, n), dtype=np.uint8)
    if out_sf is None:
        C = -(-n // 128)
        out_sf = (np.empty((-(-m // 128), C), dtype=np.float32) if fmt != SF_PACKED_UE8M0
                  else np.empty((-(-m // 128), -(-C // 4)), dtype=np.int32))
    sx, so, ss = _elem_strides(x), _elem_strides(out), _elem_strides(out_sf)
    rc = _load().oracle_cast_per_block(_ptr(x), _dtype_code(x), m, n, sx[0], sx[1], fmt,
                                       int(bool(recip)), _ptr(out), so[0], so[1],
                                       _ptr(out_sf), ss[0], ss[1])
    if rc != 0:
        raise ValueError("oracle_cast_per_block: bad arguments")
    return out, out_sf


def gemm(a: np.ndarray, sfa: np.ndarray, b: np.ndarray, sfb: np.ndarray, fmt: int,
         b_per_row: bool = False, kgran: int = 128, rows=None, d_in: np.ndarray | None = None,
         out: str = "f64"):
    """fp64 block-scaled D = A B^T over E4M3 bytes. Returns float64 [len(rows) or m, n].

    a: uint8 [m,k] (row stride may exceed k), b: uint8 [n,k]. sfa / sfb any
    strides (float32, or int32 packed UE8M0 when fmt == 2). ``out`` rounds the
    exact result to the method's output type: 'bf16' for the fwd/dgrad GEMM
    (Part 6 writes a bf16 output), 'f32' for wgrad (Parts 12-13), 'f64' none."""
    assert a.dtype == np.uint8 and b.dtype == np.uint8
    assert a.strides[1] == 1 and b.strides[1] == 1
    m, k = a.shape
    n = b.shape[0]
    assert b.shape[1] == k
    if rows is not None:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        R = rows.size
        rp = _ptr(rows)
    else:
        R, rp = m, None
    d = np.empty((R, n), dtype=np.float64)
    if d_in is not None:
        assert d_in.dtype == np.float64 and d_in.strides[1] == 8
        dip, ldi = _ptr(d_in), d_in.strides[0] // 8
    else:
        dip, ldi = None, 0
    sa, sb = _elem_strides(sfa), _elem_strides(sfb)
    rc = _load().oracle_gemm(_ptr(a), a.strides[0], _ptr(sfa), sa[0], sa[1],
                             _ptr(b), b.strides[0], _ptr(sfb), sb[0], sb[1],
                             fmt, int(bool(b_per_row)), kgran, m, n, k, rp, R,
                             _ptr(d), n, dip, ldi)
    if rc != 0:
        raise ValueError("oracle_gemm: bad arguments")
    return round_output(d, out) if out != "f64" else d


def gemm_m_grouped_contiguous(a: np.ndarray, sfa: np.ndarray, b: np.ndarray, sfb: np.ndarray, fmt: int,
                              m_indices, out: str = "f64") -> np.ndarray:
    """M-grouped GEMM over the contiguous layout of "DeepGEMM Essentials"
    Parts 8-11 (m_grouped_gemm_fp8_fp8_bf16_nt_contiguous): row i of A is
    multiplied by expert e = m_indices[i]'s weights, D[i] = A[i] B[e]^T with
    A's 1x128 scales and expert e's own 128x128 block-scale grid (Part 10 casts
    every expert separately). Rows whose index is -1 are padding (Part 9) and
    stay NaN in the result; any other index outside [0, G) is an error.

    a: uint8 [m, k]; b: uint8 [G, n, k]; sfb: [G, ceil(n/128), ceil(k/128)]
    (float32, or int32 words when fmt == 2). Returns float64 [m, n]."""
    idx = np.asarray(m_indices).astype(np.int64).reshape(-1)
    m = a.shape[0]
    G, n, _ = b.shape
    assert idx.size == m and sfb.shape[0] == G
    if np.any((idx < -1) | (idx >= G)):
        raise ValueError("m_indices outside [-1, G)")
    d = np.full((m, n), np.nan)
    for e in range(G):
        rows = np.nonzero(idx == e)[0]
        if rows.size:
            d[rows] = gemm(a, sfa, b[e], sfb[e], fmt, rows=rows, out=out)
    return d
