// Per-group FP8 scale and quantisation arithmetic shared by the casts and by
// the GEMM epilogue that writes E4M3 output ("DeepGEMM Essentials:
// High-Performance FP8 Matrix Multiplication" Part 3; UE8M0 options of
// "deep-gemm: fused per-token FP8 cast in Triton (fused_per_token_cast_to_fp8),
// version 3"). One definition, so a fused cast is bit-identical to the cast
// kernels.
//
//   amax is clamped below at the float nearest 1e-4
//   fp32 scales : s = amax / 448 and f = 448 / amax, both correctly rounded
//                 (or f = 1 / s with the recip-of-scale option)
//   UE8M0       : s rounded up to a power of two: E = biased exponent of s,
//                 plus one if s has any mantissa bit; f = 2^(127 - E) exactly
//   data        : E4M3 round-to-nearest-even of fl32(x * f), sign kept
#pragma once

#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ql {

constexpr int kSfFp32 = 0, kSfUe8m0 = 1, kSfPacked = 2;

// Scale (as stored), factor and UE8M0 exponent byte of one group from its amax.
template <int FMT, bool RECIP>
__device__ __forceinline__ void group_scale(float amax, float& s_store, float& f, uint32_t& ebyte) {
    const float a = fmaxf(amax, 1e-4f);          // 1e-4f is the float nearest 1e-4
    const float s = __fdiv_rn(a, 448.0f);
    if constexpr (FMT == kSfFp32) {
        s_store = s;
        f = RECIP ? __fdiv_rn(1.0f, s) : __fdiv_rn(448.0f, a);
        ebyte = 0;
    } else {
        const uint32_t b = __float_as_uint(s);   // s is a positive normal float
        const uint32_t E = ((b >> 23) & 0xFFu) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
        s_store = __uint_as_float(E << 23);
        f = __uint_as_float((254u - E) << 23);   // 2^(127 - E)
        ebyte = E;
    }
}

// Lane-wise max of two pairs of bf16 values (exact; a NaN operand yields the
// other operand, as fmaxf does).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two fp32 values to two E4M3 bytes (lo -> low byte), round to nearest even.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float f) {
    return e4m3x2(__fmul_rn(a, f), __fmul_rn(b, f)) | (e4m3x2(__fmul_rn(c, f), __fmul_rn(d, f)) << 16);
}

}  // namespace ql
