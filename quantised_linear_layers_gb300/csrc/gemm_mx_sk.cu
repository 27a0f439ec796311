// Split-K block-scaled FP8 GEMM for few output tiles (small M) on sm_103a.
//
// Same product as gemm_mx.cu ("DeepGEMM Essentials: High-Performance FP8
// Matrix Multiplication" Parts 1 and 6, RHS scales read row-wise per "[Help]
// Starter script for nn.Linear for fwd,bwd"), with UE8M0 scales promoted by
// the tensor core's block-scaled MMA:
//
//   D[i,j] = sum_kb 2^(ea[i,kb]-127) * 2^(eb(j,kb)-127) * sum_{k in kb} A[i,k] B[j,k]
//
// When M is small (a decode batch: M = 64 or 128 with N = 4096, K = 7168)
// there are too few output tiles to give every SM one, and each SM would
// stream a long K loop through a pipeline whose depth, not HBM, sets the
// rate. Here the K blocks of one 128 x 128 tile are split over a thread-block
// cluster of S CTAs (S = 2 or 4, one CTA per SM): CTA r accumulates K blocks
// [r*KB/S, (r+1)*KB/S) in its own tensor memory. The S partial tiles are then
// summed through distributed shared memory with no global scratch: each CTA
// owns a slice of 128/S columns; every CTA writes its fp32 partial of slice j
// into a staging buffer and the TMA engine copies it (one bulk copy per
// slice, of the tile's rows inside A only: half the bytes at M = 64) into CTA
// j's receive area, completing on CTA j's mbarrier; CTA j adds the S partials
// and writes bf16. Staging and receive areas reuse the operand
// ring, idle once every CTA of the cluster has passed the cluster barrier that
// follows its last MMA.
//
// Roles per CTA (384 threads), as in gemm_mx.cu:
//   warp 0      TMA producer over the CTA's K range.
//   warp 1      MMA issuer: per K group (four K blocks sharing one packed
//               exponent word) tcgen05.cp of the exponents, then the
//               block-scaled MMAs of the group's K blocks inside the range.
//   warps 2-3   scale loaders (packed words, or exponents of fp32 powers of two).
//   warps 4-11  epilogue: accumulator -> registers -> staging / own slice,
//               bulk copies to the other CTAs, reduction and store of the
//               CTA's own slice.
// Every wait is bounded, and the one cluster barrier is reached by every
// thread of every CTA whatever happened before.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "splitk.cuh"

namespace ql {
namespace {

constexpr int kThreads = 384;
constexpr int kMathThreads = 256;
constexpr int BM = 128;
constexpr int BK = 128;
constexpr int BN = 128;
constexpr int kSfSlots = 8;

struct SkCfg {
    static constexpr int kStageA = BM * BK;
    static constexpr int kStageB = BN * BK;
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr int kStages = 6;
    static constexpr int kSfCols = 8;                       // A exponents 4 + B exponents 4
    static constexpr int kSfColBase = BN;
    static constexpr int kTmemCols = 256;
    static constexpr int kSlotWords = BM + 128;
    static constexpr int kColsPerThread = BN / 2;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kStageA;
    static constexpr int kOffSf = kOffB + kStages * kStageB;
    static constexpr int kOffBar = kOffSf + kSfSlots * kSlotWords * 4;
    static constexpr int kNumBars = 2 * kStages + 1 + 2 * kSfSlots + 2 + 1 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    // the partial exchange (splitk.cuh) reuses the operand ring
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(BN + 2 * kSfCols <= kTmemCols, "tensor memory budget");
    static_assert(splitk::kExchangeBytes <= kOffSf, "exchange fits in the operand ring");
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl)) != 0;
}

// Exponent words of K group g for R scale rows (as gemm_mx.cu): packed words
// read directly, or the exponent fields of four fp32 powers of two gathered.
template <int R>
__device__ __forceinline__ void exp_words(const void* base, int fmt, const int64_t (&row_off)[R],
                                          const bool (&valid)[R], int g, int64_t sk, int num_kb, uint32_t (&w)[R],
                                          const Bounds& bnd, int si) {
    if (fmt == 2) {
#pragma unroll
        for (int r = 0; r < R; ++r)
        {
            const uint32_t* q = static_cast<const uint32_t*>(base) + row_off[r] + g * sk;
            w[r] = (valid[r] && QL_IN(bnd, si, q, 4)) ? __ldg(q) : 0u;
        }
        return;
    }
    uint32_t bits[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j)
        {
            const float* q = static_cast<const float*>(base) + row_off[r] + (4 * g + j) * sk;
            bits[r][j] = (valid[r] && 4 * g + j < num_kb && QL_IN(bnd, si, q, 4)) ? __float_as_uint(__ldg(q)) : 0u;
        }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        w[r] = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) w[r] |= ((bits[r][j] >> 23) & 0xFFu) << (8 * j);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_sk_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      const GemmParams p) {
    using C = SkCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    uint32_t* sSf = reinterpret_cast<uint32_t*>(smem + C::kOffSf);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* sfull = tfull + 1;
    uint64_t* sempty = sfull + kSfSlots;
    uint64_t* sftfree = sempty + kSfSlots;      // [2]: TMEM scale stage free again
    uint64_t* done_bar = sftfree + 2;
    uint64_t* rbar = done_bar + 1;              // partials of the other CTAs received
    uint32_t* tmem_base_sm = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = static_cast<int>(cluster_nctarank());
    const int rank = static_cast<int>(cluster_ctarank());
    const int tile = static_cast<int>(cluster_id_x());
    const int mb = tile % p.tiles_m, nb = tile / p.tiles_m;
    const int kb0 = static_cast<int>((static_cast<int64_t>(rank) * p.num_kb) / split);
    const int kb1 = static_cast<int>((static_cast<int64_t>(rank + 1) * p.num_kb) / split);
    const int g0 = kb0 / 4, g1 = (kb1 + 3) / 4;      // K groups touching [kb0, kb1)
    const splitk::Exchange xchg = splitk::make_exchange(smem, rbar, p, mb);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(tfull, 1);
        for (int s = 0; s < kSfSlots; ++s) { mbar_init(&sfull[s], 32); mbar_init(&sempty[s], 1); }
        mbar_init(&sftfree[0], 1);
        mbar_init(&sftfree[1], 1);
        mbar_init(done_bar, 1);
        mbar_init(rbar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // armed before the cluster barrier that precedes any copy into this CTA
        mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(split - 1) * xchg.copy_bytes);
    }
    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        // This CTA's weight tiles into L2 while the previous kernel finishes
        // (B does not depend on it): all of its K range, so the whole weight
        // streams from HBM at once instead of a smem ring's depth at a time;
        // at most 64 MB over the grid, well inside L2.
        const int pf_cap = static_cast<int>((64u << 20) / (gridDim.x * static_cast<unsigned>(BN * BK)));
        const int pf = pf_cap > C::kStages ? pf_cap : C::kStages;
        for (int kb = kb0; kb < kb1 && kb < kb0 + pf; ++kb) tma_prefetch_l2_2d(&tmap_b, kb * BK, nb * BN);
    }
    if (warp == 1) { tmem_alloc(tmem_base_sm, C::kTmemCols); tmem_relinquish(); }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_sm;
    pdl_wait_prior();            // inputs of the previous kernel are complete from here on
    const WaitCtl ctl{abort_flag, p.dev_status, p.wait_limit_ns};
    const int num_kb = p.num_kb;

    if (warp < 4) {
        regs_dealloc<104>();  // 128 x 104 + 256 x 200 = 384 x 168 registers
        if (warp == 0) {
            if (elect_one()) {
                uint32_t it = 0;
                bool ok = true;
                for (int kb = kb0; kb < kb1 && !p.stall_producer; ++kb, ++it) {
                    const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, ctl)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                    tma_load_2d(sA + s * C::kStageA, &tmap_a, &full[s], kb * BK, mb * BM);
                    tma_load_2d(sB + s * C::kStageB, &tmap_b, &full[s], kb * BK, nb * BN);
                }
                if (!ok) {
                    const uint32_t first = it > (uint32_t)C::kStages ? it - C::kStages : 0u;
                    for (uint32_t j = first; j < it; ++j)
                        mbar_wait_drain(&full[j % C::kStages], (j / C::kStages) & 1u, p.wait_limit_ns);
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            if (elect_one()) {
                uint32_t it = 0;
                bool ok = true;
                const uint32_t d_tmem = tmem_base;
                for (int kg = g0; kg < g1 && ok; ++kg) {
                    const uint32_t gi = static_cast<uint32_t>(kg - g0);
                    const uint32_t slot = gi % kSfSlots, sph = (gi / kSfSlots) & 1u;
                    const uint32_t st = gi & 1u;
                    if (!mbar_wait(&sfull[slot], sph, ctl)) { ok = false; break; }
                    if (!mbar_wait(&sftfree[st], ((gi >> 1) & 1u) ^ 1u, ctl)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t sf_col = tmem_base + C::kSfColBase + st * C::kSfCols;
                    const uint32_t* slot_ptr = sSf + slot * C::kSlotWords;
                    tmem_cp_32x128b_warpx4(sf_col, rows16_desc(smem_addr(slot_ptr)));
                    tmem_cp_32x128b_warpx4(sf_col + 4, rows16_desc(smem_addr(slot_ptr + BM)));
                    for (int kbi = 0; kbi < 4; ++kbi) {
                        const int kb = kg * 4 + kbi;
                        if (kb < kb0) continue;
                        if (kb >= kb1) break;
                        const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                        if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                        tc_fence_after_sync();
                        const uint64_t adesc = sw128_kmajor_desc(smem_addr(sA + s * C::kStageA));
                        const uint64_t bdesc = sw128_kmajor_desc(smem_addr(sB + s * C::kStageB));
                        const uint32_t idesc = idesc_mxf8_ue8m0(BM, BN, kbi, kbi);
#pragma unroll
                        for (int k4 = 0; k4 < BK / 32; ++k4)
                            mma_mxf8_block_scaled(d_tmem, adesc + 2 * k4, bdesc + 2 * k4, idesc, sf_col, sf_col + 4,
                                                  (kb > kb0 || k4 > 0) ? 1u : 0u);
                        mma_commit(&empty[s]);
                        ++it;
                    }
                    if (!ok) break;
                    mma_commit(&sempty[slot]);
                    mma_commit(&sftfree[st]);
                }
                if (ok) mma_commit(tfull);
                mma_commit(done_bar);
                mbar_wait_drain(done_bar, 0, p.wait_limit_ns);
            }
            __syncwarp();
        } else {
            // scale loaders: warps 2 and 3 take alternate runs of K groups
            // (four groups per run for packed words), all loads of a run issued
            // before any is stored; line r of the 128-row chunk holds the words
            // of rows r, 32+r, 64+r, 96+r (tcgen05.cp's four-quarter layout)
            constexpr int R = 4;
            const uint32_t mine = static_cast<uint32_t>(warp - 2);
            const int run_len = (p.fmt == 2) ? R : 1;
            const int64_t nblocks_b = (p.n + 127) / 128;
            const int64_t m0 = static_cast<int64_t>(mb) * BM;
            int64_t offa[4], offb[1];
            bool vala[4], valb[1];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t row = m0 + 32 * q + lane;
                vala[q] = row < p.m;
                offa[q] = row * p.sam;
            }
            valb[0] = lane == 0 && nb < nblocks_b;           // the tile's one 128x128 block row of B
            offb[0] = static_cast<int64_t>(nb) * p.sbn;
            uint32_t gi = 0, run = 0;
            bool ok = true;
            for (int kg0 = g0; kg0 < g1 && ok; kg0 += run_len, ++run) {
                const int cnt = g1 - kg0 < run_len ? g1 - kg0 : run_len;
                if ((run & 1u) != mine) { gi += cnt; continue; }
                uint32_t wa[R][4], wb[R][1];
                if (p.fmt == 2) {
#pragma unroll
                    for (int j = 0; j < R; ++j) {
                        const bool in = j < cnt;
                        bool va[4], vb[1];
#pragma unroll
                        for (int q = 0; q < 4; ++q) va[q] = vala[q] && in;
                        vb[0] = valb[0] && in;
                        exp_words<4>(p.sfa, 2, offa, va, kg0 + j, p.sak, num_kb, wa[j], p.bnd, 0);
                        exp_words<1>(p.sfb, 2, offb, vb, kg0 + j, p.sbk, num_kb, wb[j], p.bnd, 1);
                    }
                } else {
                    exp_words<4>(p.sfa, p.fmt, offa, vala, kg0, p.sak, num_kb, wa[0], p.bnd, 0);
                    exp_words<1>(p.sfb, p.fmt, offb, valb, kg0, p.sbk, num_kb, wb[0], p.bnd, 1);
                }
                for (int j = 0; j < cnt; ++j) {
                    const uint32_t gj = gi + j;
                    const uint32_t slot = gj % kSfSlots, ph = (gj / kSfSlots) & 1u;
                    if (!warp_wait(&sempty[slot], ph ^ 1u, ctl)) { ok = false; break; }
                    uint32_t* dst = sSf + slot * C::kSlotWords;
                    *reinterpret_cast<uint4*>(dst + lane * 4) = make_uint4(wa[j][0], wa[j][1], wa[j][2], wa[j][3]);
                    const uint32_t wbc = __shfl_sync(0xffffffffu, wb[j][0], 0);
                    *reinterpret_cast<uint4*>(dst + BM + lane * 4) = make_uint4(wbc, wbc, wbc, wbc);
                    fence_proxy_async_smem();   // visible to tcgen05.cp (async proxy)
                    mbar_arrive(&sfull[slot]);
                }
                gi += cnt;
            }
        }
        cluster_sync_all();     // see the epilogue: every thread of the cluster passes it once
    } else {
        regs_alloc<200>();
        constexpr int CPT = C::kColsPerThread;       // 64 accumulator columns per thread
        const int wg = (warp - 4) >> 2;               // column half
        const int q = warp & 3;                       // TMEM lane quarter
        const int r_local = q * 32 + lane;            // accumulator row in the tile
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const bool ok = warp_wait(tfull, 0, ctl);
        uint32_t accb[CPT];
        if (ok) {
            tc_fence_after_sync();
            const uint32_t tcol = tmem_base + lane_base + wg * CPT;
            tmem_ld_32x32b_x32(tcol, *reinterpret_cast<uint32_t(*)[32]>(&accb[0]));
            tmem_ld_32x32b_x32(tcol + 32, *reinterpret_cast<uint32_t(*)[32]>(&accb[32]));
            tmem_wait_ld(accb);
        }
        tc_fence_before_sync();
        // every CTA's MMAs have finished: every operand ring of the cluster is idle
        cluster_sync_all();
        splitk::exchange_and_store(accb, ok, xchg, wg, r_local, mb, nb, p, ctl);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace

// Cluster size for a split-K launch of this shape: 4 or 2 CTAs per 128 x 128
// tile when tiles x S fit on the SMs with at least two K blocks per CTA; 1
// when no split applies.
int choose_split_k(int64_t m, int64_t n, int64_t k, int num_sms) {
    const int64_t tiles = ((m + BM - 1) / BM) * ((n + BN - 1) / BN);
    const int64_t kbs = (k + BK - 1) / BK;
    if (tiles * 4 <= num_sms && kbs >= 8) return 4;
    if (tiles * 2 <= num_sms && kbs >= 4) return 2;
    return 1;
}

cudaError_t launch_gemm_mx_sk(const GemmLaunch& L, GemmParams p, int split, cudaStream_t st) {
    using Cf = SkCfg;
    if (split != 2 && split != 4) return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    if (!encode_kmajor_map(&ta, L.a, L.m, L.k, L.lda, BM)) return cudaErrorInvalidValue;
    if (!encode_kmajor_map(&tb, L.b, L.n, L.k, L.ldb, BN)) return cudaErrorInvalidValue;
    p.tiles_m = static_cast<int>((L.m + BM - 1) / BM);
    p.tiles_n = static_cast<int>((L.n + BN - 1) / BN);
    const int tiles = p.tiles_m * p.tiles_n;
    auto kern = gemm_mx_sk_kernel;
    if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), Cf::kSmemBytes); e != cudaSuccess) return e;
    return launch_gemm_kernel(kern, static_cast<unsigned>(tiles * split), static_cast<unsigned>(split), Cf::kSmemBytes,
                              st, ta, tb, p);
}

}  // namespace ql
