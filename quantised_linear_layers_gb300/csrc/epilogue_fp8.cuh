// GEMM epilogue that writes E4M3 output with per-token scales: the cast of
// "DeepGEMM Essentials: High-Performance FP8 Matrix Multiplication" Part 3
// applied to the GEMM's bf16 output inside the GEMM, so the next layer's
// operand never makes a round trip through HBM in bf16 (the maintainer's
// advice in "[Help] Starter script for nn.Linear for fwd,bwd": fuse the cast
// and scaling into the previous kernel's output to save HBM bandwidth).
// The values cast are the bf16-rounded accumulators, exactly what
// the bf16-output GEMM would store, and the per-group arithmetic is that of
// quant.cuh, so the result equals the cast kernel applied to the bf16 GEMM
// output, bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gemm.cuh"
#include "quant.cuh"

namespace ql {

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Row `row`, columns [col0, col0 + 128) (col0 a multiple of 128) of D from
// the 128 fp32 accumulators acc[0..127]: E4M3 bytes into p.d (row stride
// p.ldd bytes) and one scale per GRAN-wide group into p.dsf (fp32 at
// [row*dsm + g*dsg], or for packed UE8M0 byte g%4 of int32 word
// [row*dsm + (g/4)*dsg]; the owner of the last group zeroes the word's pad
// bytes). Columns at or past n are not stored. With STAGED the bytes go to
// the 128-byte shared-memory row `srow` instead, 16-byte chunk k at
// k ^ swz (the 128-byte swizzle of a TMA tile store that the caller issues),
// and the scales are stored only when `row_ok`.
template <int GRAN, bool STAGED = false>
__device__ __forceinline__ void store_row_e4m3(const float* acc, int64_t row, int64_t col0, const GemmParams& p,
                                               uint8_t* srow = nullptr, int swz = 0, bool row_ok = true) {
    constexpr int NG = 128 / GRAN;
    uint8_t* drow = static_cast<uint8_t*>(p.d) + row * p.ldd;
    const int64_t G = (p.n + GRAN - 1) / GRAN;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        const int64_t c0 = col0 + gi * GRAN;
        if (c0 < p.n) {
            // accumulators of columns at or past n are exactly zero (their B
            // rows are zero-filled), so they cannot raise the amax
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < GRAN; ++e) amax = fmaxf(amax, fabsf(bf16_round(acc[gi * GRAN + e])));
            float s, f;
            uint32_t eb;
            if (p.dfmt == kSfFp32) {
                if (p.drecip) group_scale<kSfFp32, true>(amax, s, f, eb);
                else group_scale<kSfFp32, false>(amax, s, f, eb);
            } else {
                group_scale<kSfUe8m0, false>(amax, s, f, eb);
            }
#pragma unroll
            for (int j = 0; j < GRAN; j += 16) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float* a = acc + gi * GRAN + j + 4 * q;
                    w[q] = quant4(bf16_round(a[0]), bf16_round(a[1]), bf16_round(a[2]), bf16_round(a[3]), f);
                }
                const int64_t c = c0 + j;
                if constexpr (STAGED) {
                    *reinterpret_cast<uint4*>(srow + ((((gi * GRAN + j) >> 4) ^ swz) << 4)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                } else if (p.vec_store && c + 16 <= p.n) {
                    if (QL_IN(p.bnd, 2, drow + c, 16)) *reinterpret_cast<uint4*>(drow + c) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (c + e < p.n && QL_IN(p.bnd, 2, drow + c + e, 1))
                            drow[c + e] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
                }
            }
            const int64_t g = c0 / GRAN;
            if (!row_ok) continue;
            if (p.dfmt != kSfPacked) {
                float* sp = static_cast<float*>(p.dsf) + row * p.dsm + g * p.dsg;
                if (QL_IN(p.bnd, 3, sp, 4)) *sp = s;
            } else {
                uint8_t* wb = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(p.dsf) + row * p.dsm + (g / 4) * p.dsg);
                if (QL_IN(p.bnd, 3, wb, 4)) {
                    wb[g % 4] = static_cast<uint8_t>(eb);
                    if (g == G - 1)
                        for (int z = static_cast<int>(g % 4) + 1; z < 4; ++z) wb[z] = 0;
                }
            }
        }
    }
}

// The 128 columns of one epilogue thread, group width chosen at run time.
__device__ __forceinline__ void store_row_e4m3_any(const float* acc, int64_t row, int64_t col0,
                                                   const GemmParams& p) {
    if (p.dgran == 32) store_row_e4m3<32>(acc, row, col0, p);
    else store_row_e4m3<128>(acc, row, col0, p);
}

// The same into a staged 128-byte row (see store_row_e4m3).
__device__ __forceinline__ void stage_row_e4m3_any(const float* acc, int64_t row, int64_t col0, const GemmParams& p,
                                                   uint8_t* srow, int swz, bool row_ok) {
    if (p.dgran == 32) store_row_e4m3<32, true>(acc, row, col0, p, srow, swz, row_ok);
    else store_row_e4m3<128, true>(acc, row, col0, p, srow, swz, row_ok);
}

}  // namespace ql
