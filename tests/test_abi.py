"""The C ABI boundary, without a GPU: libqlinear.so builds for sm_103a, loads,
exports every function include/qlinear.h declares, and rejects invalid
arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlinear.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\([^;{]*\)\s*;", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from quantised_linear_layers_gb300 import build
    path = build.build()
    return ctypes.CDLL(path), path


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fp8_cast_per_token", "fp8_cast_per_block", "gemm_fp8_nt_bf16", "gemm_fp8_wgrad_fp32",
                     "m_grouped_gemm_fp8_nt_bf16_contiguous", "ql_status_string", "ql_set_num_sms", "ql_get_num_sms", "ql_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    cdll, path = lib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"not exported: {missing}"
    for n in declared_functions():
        assert hasattr(cdll, n)


def test_library_built_for_sm103a_only():
    """The build passes exactly one -gencode, for sm_103a (the kernels' own
    binary version is checked at run time by a GPU test)."""
    from quantised_linear_layers_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.gpu
def test_kernels_run_as_sm103_binaries(lib):
    """cudaFuncGetAttributes(...).binaryVersion of the library's kernels, as
    the runtime reports it on the GPU: 103."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    cdll, _ = lib
    torch.cuda.init()
    assert cdll.ql_binary_version() == 103


def test_status_strings(lib):
    cdll, _ = lib
    cdll.ql_status_string.restype = ctypes.c_char_p
    assert cdll.ql_status_string(0) == b"QL_OK"
    for s in range(1, 6):
        assert cdll.ql_status_string(s).startswith(b"QL_ERR_")


def test_host_validation_rejects_before_cuda(lib):
    """These calls must return QL_ERR_INVALID_ARG from host checks alone."""
    from quantised_linear_layers_gb300 import ops
    ops.load_library()
    L = ops.load_library()
    p = ctypes.c_void_p(16)
    # gran_k 64 is not supported
    assert L.fp8_cast_per_token(p, 0, 4, 256, 256, 1, 64, 0, p, 256, 1, p, 2, 1, None) == 1
    # negative size
    assert L.fp8_cast_per_token(p, 0, -1, 256, 256, 1, 128, 0, p, 256, 1, p, 2, 1, None) == 1
    # unknown format, recip with UE8M0
    assert L.fp8_cast_per_token(p, 0, 4, 256, 256, 1, 128, 7, p, 256, 1, p, 2, 1, None) == 1
    assert L.fp8_cast_per_token(p, 0, 4, 256, 256, 1, 128, 0x101, p, 256, 1, p, 2, 1, None) == 1
    # bad dtype; null pointers
    assert L.fp8_cast_per_token(p, 9, 4, 256, 256, 1, 128, 0, p, 256, 1, p, 2, 1, None) == 1
    assert L.fp8_cast_per_token(None, 0, 4, 256, 256, 1, 128, 0, p, 256, 1, p, 2, 1, None) == 1
    # block cast: unknown format; recip with a UE8M0 format
    assert L.fp8_cast_per_block(p, 0, 4, 256, 256, 1, 3, p, 256, 1, p, 2, 1, None) == 1
    assert L.fp8_cast_per_block(p, 0, 4, 256, 256, 1, 0x102, p, 256, 1, p, 2, 1, None) == 1
    # dual per-token cast: null column output; row stride below n; recip with UE8M0; empty is a no-op
    T2 = L.fp8_cast_per_token_dual
    assert T2(p, 0, 4, 256, 256, 0, p, 256, p, 1, 4, None, 256, p, 1, 4, None) == 1
    assert T2(p, 0, 4, 256, 128, 0, p, 256, p, 1, 4, p, 256, p, 1, 4, None) == 1
    assert T2(p, 0, 4, 256, 256, 0x101, p, 256, p, 1, 4, p, 256, p, 1, 4, None) == 1
    assert T2(None, 0, 0, 256, 256, 0, None, 256, None, 1, 4, None, 256, None, 1, 4, None) == 0
    # dual block cast: missing second scale grid; unknown format; empty problem is a no-op
    D = L.fp8_cast_per_block_dual
    assert D(p, 0, 4, 256, 256, 1, 2, p, 256, 1, p, 2, 1, None, 1, 1, None) == 1
    assert D(p, 0, 4, 256, 256, 1, 3, p, 256, 1, p, 2, 1, p, 1, 1, None) == 1
    assert D(None, 0, 0, 256, 256, 1, 2, None, 256, 1, None, 2, 1, None, 1, 1, None) == 0
    # empty problems are no-ops (no CUDA call)
    assert L.fp8_cast_per_token(None, 0, 0, 256, 256, 1, 128, 0, None, 256, 1, None, 2, 1, None) == 0
    assert L.gemm_fp8_nt_bf16(None, 16, None, 1, 1, None, 16, None, 1, 1, 0, None, 16, 0, 16, 16, None, 0,
                              None) == 0
    # GEMM: bad format, null operands, short leading dimension
    assert L.gemm_fp8_nt_bf16(p, 32, p, 1, 1, p, 32, p, 1, 1, 5, p, 8, 4, 8, 32, None, 0, None) == 1
    assert L.gemm_fp8_nt_bf16(None, 32, p, 1, 1, p, 32, p, 1, 1, 0, p, 8, 4, 8, 32, None, 0, None) == 1
    assert L.gemm_fp8_nt_bf16(p, 16, p, 1, 1, p, 32, p, 1, 1, 0, p, 8, 4, 8, 32, None, 0, None) == 1
    # misaligned operand pointer / leading dimension
    q = ctypes.c_void_p(24)
    assert L.gemm_fp8_nt_bf16(q, 32, p, 1, 1, p, 32, p, 1, 1, 0, p, 8, 4, 8, 32, None, 0, None) == 3
    assert L.gemm_fp8_nt_bf16(p, 40, p, 1, 1, p, 32, p, 1, 1, 0, p, 8, 4, 8, 32, None, 0, None) == 3
    # grouped GEMM: m not a multiple of the 128-row alignment, no experts, no index vector, k == 0
    G = L.m_grouped_gemm_fp8_nt_bf16_contiguous
    assert G(p, 32, p, 1, 1, p, 32, p, 1, 1, 1, 0, p, 8, p, 2, 100, 8, 32, None) == 1
    assert G(p, 32, p, 1, 1, p, 32, p, 1, 1, 1, 0, p, 8, p, 0, 128, 8, 32, None) == 1
    assert G(p, 32, p, 1, 1, p, 32, p, 1, 1, 1, 0, p, 8, None, 2, 128, 8, 32, None) == 1
    assert G(p, 32, p, 1, 1, p, 32, p, 1, 1, 1, 0, p, 8, p, 2, 128, 8, 0, None) == 2
    assert G(None, 32, None, 1, 1, None, 32, None, 1, 1, 1, 0, None, 8, None, 2, 0, 8, 32, None) == 0
    assert L.ql_get_m_alignment_for_contiguous_layout() == 128
    # host pipeline: workspace too small, chunk_rows 0, unknown format (host checks only)
    H = L.ql_cast_gemm_host
    assert H(p, 64, p, 64, p, 1, 1, 0, p, 64, 64, 64, 64, 16, p, 10, None) == 1
    assert H(p, 64, p, 64, p, 1, 1, 0, p, 64, 64, 64, 64, 0, p, 1 << 30, None) == 1
    assert H(p, 64, p, 64, p, 1, 1, 7, p, 64, 64, 64, 64, 16, p, 1 << 30, None) == 1
    assert L.ql_cast_gemm_host_workspace_size(64, 64, 16, 0) > 0
    # GEMM with E4M3 output: group 64, unknown format, recip with UE8M0, no scale buffer, k == 0
    F = L.gemm_fp8_nt_fp8out
    assert F(p, 32, p, 1, 1, p, 32, p, 1, 1, 0, p, 32, p, 1, 1, 64, 0, 4, 8, 32, None) == 1
    assert F(p, 32, p, 1, 1, p, 32, p, 1, 1, 0, p, 32, p, 1, 1, 128, 5, 4, 8, 32, None) == 1
    assert F(p, 32, p, 1, 1, p, 32, p, 1, 1, 0, p, 32, p, 1, 1, 128, 0x101, 4, 8, 32, None) == 1
    assert F(p, 32, p, 1, 1, p, 32, p, 1, 1, 0, p, 32, None, 1, 1, 128, 0, 4, 8, 32, None) == 1
    assert F(p, 32, p, 1, 1, p, 32, p, 1, 1, 0, p, 32, p, 1, 1, 128, 0, 4, 8, 0, None) == 2
    assert L.ql_set_gemm_block_n(48) == 1
    assert L.ql_set_wait_limit_ms(0) == 1


def test_ops_fail_loudly_without_library(tmp_path):
    from quantised_linear_layers_gb300 import ops
    import quantised_linear_layers_gb300.ops as mod
    saved = mod._lib
    mod._lib = None
    try:
        with pytest.raises(RuntimeError, match="not found"):
            ops.load_library(str(tmp_path / "missing.so"))
    finally:
        mod._lib = saved
