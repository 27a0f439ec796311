// Split-K FP8 GEMM with CUDA-core promotion (fp32 scales) for few output
// tiles (small M) on sm_103a.
//
// The product of gemm.cu's promotion kernel ("DeepGEMM Essentials:
// High-Performance FP8 Matrix Multiplication" Parts 1 and 6, RHS scales read
// row-wise per "[Help] Starter script for nn.Linear for fwd,bwd"):
//
//   D[i,j] = sum_kb (sa[i,kb] * sb[j/128,kb]) * P_kb[i,j],  P_kb = sum_{k in kb} A[i,k] B[j,k]
//
// with any fp32 scales. With M = 64 or 128 (a decode batch against N = 4096, K
// = 7168) there are 32 tiles of 128 x 128; on one SM each they would walk all
// 56 K blocks, a pipeline whose per-K-block hand-offs, not HBM, set the rate.
// Here the K blocks of one tile are split over a thread-block cluster of S = 2
// or 4 CTAs: CTA r promotes K blocks [r*KB/S, (r+1)*KB/S) into its own fp32
// registers, and the S partial tiles are then summed in rank order through
// distributed shared memory (splitk.cuh) and written as bf16.
//
// Roles per CTA (384 threads):
//   warp 0      TMA producer over the CTA's K range (A and B boxes of 128 x 128).
//   warp 1      MMA issuer: per K block four kind::f8f6f4 MMAs (K = 32 each)
//               into a fresh tensor-memory stage (four stages of 128 columns).
//   warps 2-3   scale loaders: runs of four K blocks, one shared-memory slot
//               per run (the rows' sa, the tile's sb).
//   warps 4-11  math: per K block the partial product (tcgen05.ld), one arrive
//               per warp releases the stage, acc += (sa*sb)*P with fp32 FMAs;
//               then the cluster exchange and the bf16 store of the CTA's slice.
// Every wait is bounded, and the one cluster barrier is reached by every
// thread of every CTA whatever happened before.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "promote.cuh"
#include "splitk.cuh"

namespace ql {
namespace {

constexpr int kThreads = splitk::kThreads;
constexpr int BM = splitk::BM;
constexpr int BN = splitk::BN;
constexpr int BK = 128;
constexpr int kRun = 4;          // K blocks per scale slot
constexpr int kSlots = 4;

struct PskCfg {
    static constexpr int kStageA = BM * BK;
    static constexpr int kStageB = BN * BK;
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr int kStages = 6;
    static constexpr int kTmemStages = 4;                  // 4 x 128 columns: all of tensor memory
    static constexpr int kSlotFloats = BM + 4;             // one K block: 128 row scales, the tile's B scale
    static constexpr int kRunFloats = kRun * kSlotFloats;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kStageA;
    static constexpr int kOffScale = kOffB + kStages * kStageB;
    static constexpr int kOffBar = kOffScale + kSlots * kRunFloats * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kTmemStages + 2 * kSlots + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;      // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(splitk::kExchangeBytes <= kOffScale, "exchange fits in the operand ring");
};

__global__ void __launch_bounds__(kThreads, 1)
    gemm_prom_sk_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const GemmParams p) {
    using C = PskCfg;
    constexpr int CPT = splitk::kColsPerThread;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + C::kTmemStages;
    uint64_t* sfull = tempty + C::kTmemStages;
    uint64_t* sempty = sfull + kSlots;
    uint64_t* done_bar = sempty + kSlots;
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
    const int nkb = kb1 - kb0;
    const splitk::Exchange xchg = splitk::make_exchange(smem, rbar, p, mb);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        // the math warps release stages and scale slots one arrive per warp
        for (int s = 0; s < C::kTmemStages; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], splitk::kMathThreads / 32); }
        for (int s = 0; s < kSlots; ++s) { mbar_init(&sfull[s], 32); mbar_init(&sempty[s], splitk::kMathThreads / 32); }
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
        // this CTA's weight tiles into L2 while the previous kernel finishes
        // (B does not depend on it): all of its K range, at most 64 MB over the grid
        const int pf_cap = static_cast<int>((64u << 20) / (gridDim.x * static_cast<unsigned>(BN * BK)));
        const int pf = pf_cap > C::kStages ? pf_cap : C::kStages;
        for (int kb = kb0; kb < kb1 && kb < kb0 + pf; ++kb) tma_prefetch_l2_2d(&tmap_b, kb * BK, nb * BN);
    }
    if (warp == 1) { tmem_alloc(tmem_base_sm, 512); tmem_relinquish(); }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_sm;
    pdl_wait_prior();            // inputs of the previous kernel are complete from here on
    const WaitCtl ctl{abort_flag, p.dev_status, p.wait_limit_ns};

    if (warp < 4) {
        regs_dealloc<88>();   // 128 x 88 + 256 x 208 = 384 x 168 registers
        if (warp == 0) {
            // ---------------- TMA producer ----------------
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
                    // drain: every stage whose load was issued completes its phase
                    const uint32_t first = it > (uint32_t)C::kStages ? it - C::kStages : 0u;
                    for (uint32_t j = first; j < it; ++j)
                        mbar_wait_drain(&full[j % C::kStages], (j / C::kStages) & 1u, p.wait_limit_ns);
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ---------------- MMA issuer ----------------
            if (elect_one()) {
                const uint32_t idesc = idesc_e4m3_f32(BM, BN);
                bool ok = true;
                for (int i = 0; i < nkb && ok; ++i) {
                    const uint32_t ts = i % C::kTmemStages, tph = (i / C::kTmemStages) & 1u;
                    if (!mbar_wait(&tempty[ts], tph ^ 1u, ctl)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t s = i % C::kStages, ph = (i / C::kStages) & 1u;
                    if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint64_t adesc = sw128_kmajor_desc(smem_addr(sA + s * C::kStageA));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_addr(sB + s * C::kStageB));
                    const uint32_t d_tmem = tmem_base + ts * BN;
#pragma unroll
                    for (int k4 = 0; k4 < BK / 32; ++k4)
                        mma_e4m3(d_tmem, adesc + 2 * k4, bdesc + 2 * k4, idesc, k4 > 0 ? 1u : 0u);
                    mma_commit(&empty[s]);
                    mma_commit(&tfull[ts]);
                }
                // every MMA has completed before tensor memory is freed
                mma_commit(done_bar);
                mbar_wait_drain(done_bar, 0, p.wait_limit_ns);
            }
            __syncwarp();
        } else {
            // ---------------- scale loaders ----------------
            // Warps 2 and 3 take alternate runs of four K blocks, one slot per
            // run; all loads of a run are issued before any is stored.
            const uint32_t mine = static_cast<uint32_t>(warp - 2);
            const int64_t m0 = static_cast<int64_t>(mb) * BM;
            const bool b_ok = nb < (p.n + 127) / 128;
            uint32_t run = 0;
            bool ok = true;
            for (int i0 = 0; i0 < nkb && ok; i0 += kRun, ++run) {
                const int cnt = nkb - i0 < kRun ? nkb - i0 : kRun;
                if ((run & 1u) != mine) continue;
                float va[kRun][4], vb[kRun];
#pragma unroll
                for (int j = 0; j < kRun; ++j) {
                    const int kb = kb0 + i0 + j;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int64_t row = m0 + lane + 32 * r;
                        va[j][r] = (j < cnt && row < p.m) ? decode_scale(p.sfa, p.fmt, row * p.sam, kb, p.sak, p.bnd, 0) : 0.0f;
                    }
                    vb[j] = (j < cnt && lane == 0 && b_ok)
                                ? decode_scale(p.sfb, p.fmt, static_cast<int64_t>(nb) * p.sbn, kb, p.sbk, p.bnd, 1)
                                : 0.0f;
                }
                const uint32_t slot = run % kSlots, ph = (run / kSlots) & 1u;
                if (!warp_wait(&sempty[slot], ph ^ 1u, ctl)) { ok = false; break; }
                float* dst = sScale + slot * C::kRunFloats;
#pragma unroll
                for (int j = 0; j < kRun; ++j) {
                    if (j >= cnt) break;
#pragma unroll
                    for (int r = 0; r < 4; ++r) dst[j * C::kSlotFloats + lane + 32 * r] = va[j][r];
                    if (lane == 0) dst[j * C::kSlotFloats + BM] = vb[j];
                }
                mbar_arrive(&sfull[slot]);
            }
        }
        cluster_sync_all();     // see the math warps: every thread of the cluster passes it once
    } else {
        regs_alloc<208>();
        // ---------------- math: promotion, then the cluster exchange ----------------
        const int wg = (warp - 4) >> 2;          // column half
        const int q = warp & 3;                  // TMEM lane quarter
        const int r_local = q * 32 + lane;       // accumulator row in the tile
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        float acc[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
        bool ok = true;
        uint32_t run = 0;
        for (int i = 0; i < nkb; ++i) {
            const int jr = i % kRun;
            const uint32_t slot = run % kSlots, sph = (run / kSlots) & 1u;
            const bool slot_end = jr == kRun - 1 || i == nkb - 1;
            if (jr == 0 && !warp_wait(&sfull[slot], sph, ctl)) { ok = false; break; }
            const float* src = sScale + slot * C::kRunFloats + jr * C::kSlotFloats;
            const float sab = src[r_local] * src[BM];
            const uint32_t ts = i % C::kTmemStages, tph = (i / C::kTmemStages) & 1u;
            if (!warp_wait(&tfull[ts], tph, ctl)) { ok = false; break; }
            tc_fence_after_sync();
            uint32_t v[CPT];
            tmem_load_cols<CPT>(tmem_base + lane_base + ts * BN + wg * CPT, v);
            // read: one arrive per warp releases the stage to the MMA issuer
            tc_fence_before_sync();
            __syncwarp();
            mbar_arrive_lane0(&tempty[ts], lane);
            // one fp32 FMA per element (single rounding)
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[j] = fmaf(__uint_as_float(v[j]), sab, acc[j]);
            if (slot_end) {
                __syncwarp();
                mbar_arrive_lane0(&sempty[slot], lane);
                ++run;
            }
        }
        uint32_t accb[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) accb[j] = __float_as_uint(acc[j]);
        ok = __all_sync(0xffffffffu, ok) != 0;
        tc_fence_before_sync();
        // every CTA's MMAs have finished: every operand ring of the cluster is idle
        cluster_sync_all();
        splitk::exchange_and_store(accb, ok, xchg, wg, r_local, mb, nb, p, ctl);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace

cudaError_t launch_gemm_prom_sk(const GemmLaunch& L, GemmParams p, int split, cudaStream_t st) {
    using Cf = PskCfg;
    if (split != 2 && split != 4) return cudaErrorInvalidValue;
    if (L.a_mn || L.b_mn || L.out_f32 || L.out_fp8 || L.m_indices != nullptr) return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    if (!encode_kmajor_map(&ta, L.a, L.m, L.k, L.lda, BM)) return cudaErrorInvalidValue;
    if (!encode_kmajor_map(&tb, L.b, L.n, L.k, L.ldb, BN)) return cudaErrorInvalidValue;
    p.tiles_m = static_cast<int>((L.m + BM - 1) / BM);
    p.tiles_n = static_cast<int>((L.n + BN - 1) / BN);
    const int tiles = p.tiles_m * p.tiles_n;
    auto kern = gemm_prom_sk_kernel;
    if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), Cf::kSmemBytes); e != cudaSuccess) return e;
    return launch_gemm_kernel(kern, static_cast<unsigned>(tiles * split), static_cast<unsigned>(split), Cf::kSmemBytes,
                              st, ta, tb, p);
}

}  // namespace ql
