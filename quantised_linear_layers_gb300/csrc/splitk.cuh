// The partial-sum exchange of the split-K GEMMs (a thread-block cluster of S
// CTAs, each summing a contiguous range of the K blocks of one 128 x 128 output
// tile): the S fp32 partial tiles are added through distributed shared memory,
// with no global scratch.
//
// Each CTA owns a slice of 128/S columns. Every CTA writes its partial of the
// other slices into staging blocks and the TMA engine copies each (one bulk
// copy per slice, of the tile's rows inside A only) into the owner's receive
// area, completing on the owner's mbarrier; the owner adds the S partials in
// rank order and writes bf16. Staging and receive areas reuse the operand
// ring, idle once every CTA of the cluster has passed the cluster barrier
// that follows its last MMA.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"
#include "gemm.cuh"

namespace ql {
namespace splitk {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kMathThreads = 256;
constexpr int kThreads = 384;
constexpr int kColsPerThread = BN / 2;          // an epilogue thread's columns (its column half)
constexpr int kRecvBytes = BM * BN * 4;         // S receive blocks of [128][128/S] fp32
// then, per column half, room for two staging blocks of [128][64] fp32
constexpr int kExchangeBytes = kRecvBytes + 4 * BM * (BN / 2) * 4;

// Byte offset of 16-byte chunk c of row r in a [128][sw] fp32 block: chunks
// are XOR-swizzled by the row's low three bits, so a warp's 32 consecutive
// rows touching the same logical chunk spread over all banks.
__device__ __forceinline__ uint32_t xchg_off(int r, int c, int sw) {
    return static_cast<uint32_t>(r * sw * 4 + ((c ^ (r & 7)) << 4));
}

// Geometry of one CTA's part in the exchange.
struct Exchange {
    uint8_t* ring;          // the idle operand ring (receive blocks, then staging)
    uint64_t* rbar;         // armed for (S - 1) * copy_bytes before the cluster barrier
    int rank, split, sw;
    uint32_t slice_bytes, copy_bytes;
};

__device__ __forceinline__ Exchange make_exchange(uint8_t* ring, uint64_t* rbar, const GemmParams& p, int mb) {
    Exchange x;
    x.ring = ring;
    x.rbar = rbar;
    x.split = static_cast<int>(cluster_nctarank());
    x.rank = static_cast<int>(cluster_ctarank());
    x.sw = BN / x.split;
    x.slice_bytes = static_cast<uint32_t>(BM * x.sw * 4);
    // only the tile's rows inside A travel: rows are contiguous in a slice block
    const int64_t rows_left = p.m - static_cast<int64_t>(mb) * BM;
    x.copy_bytes = static_cast<uint32_t>((rows_left < BM ? rows_left : BM) * x.sw * 4);
    return x;
}

// The epilogue threads' part, after the cluster barrier that follows every
// CTA's last MMA. accb: the fp32 bits of this thread's 64 partial columns
// (column half wg, tile row r_local); ok: they are valid (no wait ran out).
// Uses named barriers 1, 2 (one per column half) and 3 (all epilogue threads).
__device__ __forceinline__ void exchange_and_store(const uint32_t (&accb)[kColsPerThread], bool ok, const Exchange& x,
                                                   int wg, int r_local, int mb, int nb, const GemmParams& p,
                                                   const WaitCtl& ctl) {
    constexpr int CPT = kColsPerThread;
    uint8_t* recv = x.ring;
    // this half's staging blocks (one per remote slice, at most two)
    uint8_t* stage = x.ring + kRecvBytes + wg * 2 * x.slice_bytes;
    const int lg = __ffs(x.sw) - 1;
    const int first_slice = (wg * CPT) >> lg;
    if (ok) {
        // own slice straight into recv[rank], the others into staging[slice - first_slice]
#pragma unroll
        for (int c4 = 0; c4 < CPT / 4; ++c4) {
            const int col = wg * CPT + c4 * 4;
            const int j = col >> lg;
            const int cc = (col - (j << lg)) >> 2;
            uint8_t* blk = (j == x.rank) ? recv + x.rank * x.slice_bytes : stage + (j - first_slice) * x.slice_bytes;
            *reinterpret_cast<uint4*>(blk + xchg_off(r_local, cc, x.sw)) =
                make_uint4(accb[c4 * 4], accb[c4 * 4 + 1], accb[c4 * 4 + 2], accb[c4 * 4 + 3]);
        }
        fence_proxy_async_smem();     // staging visible to the bulk copies (async proxy)
    }
    named_bar_sync(1 + wg, 128);
    if (ok && (threadIdx.x & 127) == 0) {
        const int nsl = CPT >> lg;                    // slices in this half (1 or 2)
        for (int i = 0; i < nsl; ++i) {
            const int j = first_slice + i;
            if (j == x.rank) continue;
            bulk_copy_to_cluster(mapa_shared(recv + x.rank * x.slice_bytes, static_cast<uint32_t>(j)),
                                 stage + i * x.slice_bytes, x.copy_bytes, mapa_shared(x.rbar, static_cast<uint32_t>(j)));
        }
        bulk_commit_group();
    }
    named_bar_sync(3, kMathThreads);                  // own slice complete
    const bool got = ok && __all_sync(0xffffffffu, mbar_wait(x.rbar, 0, ctl)) != 0;   // the other CTAs' partials arrived
    if (got) {
        const int t = threadIdx.x - (kThreads - kMathThreads);
        const int row = t & (BM - 1), part = t >> 7;
        const int cpp = x.sw >> 3;                    // 16-byte chunks per thread: sw/4 over two parts
        const int64_t grow = static_cast<int64_t>(mb) * BM + row;
        if (grow < p.m) {
            __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.d) + grow * p.ldd;
            for (int c = part * cpp; c < (part + 1) * cpp; c += 2) {
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
                for (int s = 0; s < x.split; ++s) {
                    const uint8_t* blk = recv + s * x.slice_bytes;
                    const float4 v0 = *reinterpret_cast<const float4*>(blk + xchg_off(row, c, x.sw));
                    const float4 v1 = *reinterpret_cast<const float4*>(blk + xchg_off(row, c + 1, x.sw));
                    acc[0] += v0.x; acc[1] += v0.y; acc[2] += v0.z; acc[3] += v0.w;
                    acc[4] += v1.x; acc[5] += v1.y; acc[6] += v1.z; acc[7] += v1.w;
                }
                const int64_t col = static_cast<int64_t>(nb) * BN + x.rank * x.sw + c * 4;
                if (p.vec_store && col + 8 <= p.n) {
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(acc[0], acc[1]);
                    __nv_bfloat162 h1 = __floats2bfloat162_rn(acc[2], acc[3]);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[4], acc[5]);
                    __nv_bfloat162 h3 = __floats2bfloat162_rn(acc[6], acc[7]);
                    uint4 u;
                    u.x = *reinterpret_cast<uint32_t*>(&h0);
                    u.y = *reinterpret_cast<uint32_t*>(&h1);
                    u.z = *reinterpret_cast<uint32_t*>(&h2);
                    u.w = *reinterpret_cast<uint32_t*>(&h3);
                    if (QL_IN(p.bnd, 2, drow + col, 16)) *reinterpret_cast<uint4*>(drow + col) = u;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (col + e < p.n && QL_IN(p.bnd, 2, drow + col + e, 2)) drow[col + e] = __float2bfloat16_rn(acc[e]);
                }
            }
        }
    }
    // the staging blocks must stay until the copies out of them have read them
    if ((threadIdx.x & 127) == 0) bulk_wait_read_all();
}

}  // namespace splitk
}  // namespace ql
