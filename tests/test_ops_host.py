"""Host-side marshalling of the Python binding, on CPU: scale-tensor shapes
and the M-major TMA-aligned layout of "DeepGEMM Essentials" Part 5 (scales
transposed, the M extent padded so every column starts on 16 bytes), packed
UE8M0 word counts (four exponents per int32 along K), and argument checks that
raise before any library call."""
import pytest
import torch

from quantised_linear_layers_gb300 import ops


@pytest.mark.parametrize("n,gran,fmt,cols", [
    (4096, 128, ops.SF_FP32, 32), (4096, 32, ops.SF_UE8M0, 128),
    (4096, 32, ops.SF_PACKED_UE8M0, 32), (4096, 128, ops.SF_PACKED_UE8M0, 8),
    (1000, 128, ops.SF_FP32, 8), (1000, 128, ops.SF_PACKED_UE8M0, 2),
    (1000, 32, ops.SF_PACKED_UE8M0, 8), (7168, 128, ops.SF_PACKED_UE8M0, 14),
    (1, 128, ops.SF_PACKED_UE8M0, 1), (512, 128, ops.SF_FP32, 4),
])
def test_scale_columns(n, gran, fmt, cols):
    assert ops.sf_shape(n, gran, fmt) == cols


@pytest.mark.parametrize("m", [1, 3, 4, 7, 8, 129, 4096])
@pytest.mark.parametrize("fmt", [ops.SF_FP32, ops.SF_PACKED_UE8M0])
def test_mn_major_scales_are_tma_aligned(m, fmt):
    cols = 5
    s = ops.empty_sf(m, cols, fmt, "cpu", mn_major=True)
    assert s.shape == (m, cols)
    assert s.dtype == (torch.int32 if fmt == ops.SF_PACKED_UE8M0 else torch.float32)
    ld = -(-m // 4) * 4
    assert s.stride() == (1, ld)
    assert (s.stride(1) * s.element_size()) % 16 == 0
    r = ops.empty_sf(m, cols, fmt, "cpu")
    assert r.shape == (m, cols) and r.stride() == (cols, 1)


def test_mn_major_scales_of_zero_rows():
    s = ops.empty_sf(0, 3, ops.SF_FP32, "cpu", mn_major=True)
    assert s.shape == (0, 3)


def test_arguments_checked_before_the_library():
    a = torch.zeros((64, 256), dtype=torch.float8_e4m3fn)
    b = torch.zeros((128, 256), dtype=torch.float8_e4m3fn)
    sa = torch.ones((64, 2))
    sb = torch.ones((1, 2))
    with pytest.raises(ValueError):           # K differs
        ops.gemm_fp8_nt_bf16(a, sa, torch.zeros((128, 128), dtype=torch.float8_e4m3fn), sb)
    with pytest.raises(ValueError):           # K not contiguous
        ops.gemm_fp8_nt_bf16(a.t().contiguous().t(), sa, b, sb)
    with pytest.raises(TypeError):            # not an E4M3 tensor
        ops.gemm_fp8_nt_bf16(a.to(torch.bfloat16), sa, b, sb)
    with pytest.raises(ValueError):           # accumulate needs an existing output
        ops.gemm_fp8_wgrad_fp32(a, sa, b, sa, accumulate=True)
    with pytest.raises(ValueError):
        ops.fp8_cast_per_token(torch.zeros(8), 128)
    with pytest.raises(TypeError):
        ops._dtype_code(torch.zeros(4, dtype=torch.float16))
