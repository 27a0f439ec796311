"""CPU oracle for the fine-grained-scaled FP8 linear layer.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product path (the CUDA library
and its Python binding) never does. It shares no code with the CUDA path.

The arithmetic lives in plain C (``qlinear_oracle.c``); this package compiles
it with gcc and exposes numpy-level wrappers.
"""
from .oracle import (  # noqa: F401
    SF_FP32, SF_UE8M0, SF_PACKED_UE8M0, BF16, F32,
    build, round_output, e4m3_encode, e4m3_decode, cast_per_token, cast_per_block, gemm,
    gemm_m_grouped_contiguous,
    overflow_count, reset_overflow_count, num_threads, set_num_threads,
)
