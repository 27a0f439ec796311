// Helpers of the CUDA-core promotion GEMMs (fp32 scales): scale decoding,
// packed fp32x2 arithmetic and tensor-memory reads of accumulator columns.
//
// The promotion itself ("[Help] Starter script for nn.Linear for fwd,bwd",
// maintainer's reply; "DeepGEMM Essentials: High-Performance FP8 Matrix
// Multiplication" Part 6): after the tensor core has summed one 128-wide K
// block into tensor memory, the partial product P_kb is read into registers
// and acc += (sa[row, kb] * sb(col, kb)) * P_kb, once per K block.
#pragma once

#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"

namespace ql {

// Scale of row `row_off` (element offset of the row in the scale tensor) and
// K block `kb`: an fp32 value (fmt 0/1) or one byte of a packed UE8M0 word
// (fmt 2: four K blocks per int32, block kb in byte kb % 4), as 2^(e - 127).
// In bounds-checked builds the read is checked against span `si` of `bnd`.
__device__ __forceinline__ float decode_scale(const void* base, int fmt, int64_t row_off, int kb, int64_t sk,
                                              const Bounds& bnd, int si) {
    if (fmt != 2) {
        const float* q = static_cast<const float*>(base) + row_off + kb * sk;
        return QL_IN(bnd, si, q, 4) ? __ldg(q) : 0.0f;
    }
    const uint32_t* q = static_cast<const uint32_t*>(base) + row_off + (kb >> 2) * sk;
    const uint32_t w = QL_IN(bnd, si, q, 4) ? __ldg(q) : 0u;
    const uint32_t e = (w >> (8 * (kb & 3))) & 0xFFu;
    return __uint_as_float(e ? (e << 23) : 0x00400000u);   // 2^(e-127)
}

__device__ __forceinline__ uint64_t pack2(float a, float b) {
    return static_cast<uint64_t>(__float_as_uint(a)) | (static_cast<uint64_t>(__float_as_uint(b)) << 32);
}

// acc2 = p2 * s2 + acc2 on two fp32 lanes at once
__device__ __forceinline__ void fma2(uint64_t& acc2, uint64_t p2, uint64_t s2) {
    asm volatile("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2) : "l"(p2), "l"(s2));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a2, uint64_t b2) {
    uint64_t r;
    asm volatile("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a2), "l"(b2));
    return r;
}

// Reads N (16, 32 or 64) consecutive fp32 accumulator columns of this warp's
// 32 TMEM lanes and waits for them.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&v)[N]) {
    if constexpr (N == 16) {
        tmem_ld_32x32b_x16(taddr, v);
    } else if constexpr (N == 32) {
        tmem_ld_32x32b_x32(taddr, v);
    } else {
        static_assert(N == 64, "16, 32 or 64 columns");
        tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld_32x32b_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
    }
    tmem_wait_ld(v);
}

// One arrive on `bar` for the whole (converged) warp, by its lane 0.
__device__ __forceinline__ void mbar_arrive_lane0(uint64_t* bar, int lane) {
    if (lane == 0) mbar_arrive(bar);
}

// Bounded wait whose outcome is the same for every lane of the warp (the
// .sync.aligned tensor-memory loads that follow need a converged warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl)) != 0;
}

}  // namespace ql
