// GEMM output through shared memory and TMA tile stores.
//
// The GEMM's epilogue warps hold one output row per lane (the 32x32b TMEM
// load shape: lane l of a warp owns row l of its 32-row quarter). Stored
// directly, every warp store touches 32 rows with half-filled sectors; staged
// instead through a small per-warp buffer, each 32-row block leaves by one TMA
// tile store of whole lines, and the same copy can add into an fp32 D in L2
// (the accumulate form of the weight gradient's fp32 main grad).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace ql {

// Writes one warp's 32 rows (lane l holds the CPT fp32 accumulators of row l,
// columns x0 .. x0+CPT of D, rows y0 .. y0+32) through the warp's staging
// buffer `stg` of 32 rows x RB bytes: CW = RB / element-size columns per copy,
// as bf16 (rounded to nearest even) or fp32. Chunk k (16 bytes) of row l sits
// at k ^ (l & 7) under the 128-byte swizzle (RB = 128), at k ^ ((l >> 1) & 3)
// under the 64-byte swizzle (RB = 64), and unswizzled otherwise (RB = 112,
// whose pitch already spreads 8 consecutive rows over all banks); `tmap` must
// describe D with a [32 x CW] box and the matching swizzle. Lane 0 waits until
// the previous copy has read the buffer before it is rewritten and issues the
// copies (TMA store, or TMA reduce-add when `add`); rows and columns outside D
// are dropped by the copy. The caller waits for the copies to complete
// (bulk_wait_all) before the buffer is released.
template <int CPT, int RB, bool OUT_F32>
__device__ __forceinline__ void tma_store_warp_rows(const float* acc, uint8_t* stg, const CUtensorMap* tmap,
                                                    int64_t x0, int32_t y0, bool add) {
    constexpr int ES = OUT_F32 ? 4 : 2;
    constexpr int CW = RB / ES;
    static_assert(RB % 16 == 0 && CPT % CW == 0, "whole 16-byte chunks, whole copies");
    const int lane = static_cast<int>(threadIdx.x & 31);
#pragma unroll
    for (int c = 0; c < CPT; c += CW) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int k = 0; k < RB / 16; ++k) {
            uint4 v;
            if constexpr (OUT_F32) {
                v = make_uint4(__float_as_uint(acc[c + 4 * k]), __float_as_uint(acc[c + 4 * k + 1]),
                               __float_as_uint(acc[c + 4 * k + 2]), __float_as_uint(acc[c + 4 * k + 3]));
            } else {
                const float* a8 = acc + c + 8 * k;
                __nv_bfloat162 h0 = __floats2bfloat162_rn(a8[0], a8[1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(a8[2], a8[3]);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(a8[4], a8[5]);
                __nv_bfloat162 h3 = __floats2bfloat162_rn(a8[6], a8[7]);
                v = make_uint4(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                               *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3));
            }
            uint32_t pos;
            if constexpr (RB == 128) pos = static_cast<uint32_t>((k ^ (lane & 7)) << 4);
            else if constexpr (RB == 64) pos = static_cast<uint32_t>((k ^ ((lane >> 1) & 3)) << 4);
            else pos = static_cast<uint32_t>(k << 4);
            *reinterpret_cast<uint4*>(stg + lane * RB + pos) = v;
        }
        fence_proxy_async_smem();     // the buffer's bytes are visible to the copy (async proxy)
        __syncwarp();
        if (lane == 0) {
            const int32_t x = static_cast<int32_t>(x0 + c);
            if (OUT_F32 && add) tma_reduce_add_2d(tmap, stg, x, y0);
            else tma_store_2d(tmap, stg, x, y0);
            bulk_commit_group();
        }
    }
}

}  // namespace ql
