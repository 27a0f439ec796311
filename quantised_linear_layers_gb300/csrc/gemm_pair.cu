// Block-scaled FP8 GEMM with fp32 scales on CTA pairs: the tensor cores of
// two SMs (tcgen05 cta_group::2) and promotion on the CUDA cores.
//
// The product of "DeepGEMM Essentials: High-Performance FP8 Matrix
// Multiplication" Parts 1, 6 (gemm_fp8_fp8_bf16_nt) and 12-13
// (wgrad_gemm_fp8_fp8_fp32_nt), RHS scales read row-wise per "[Help] Starter
// script for nn.Linear for fwd,bwd" (maintainer's reply):
//
//   D[i,j] = sum_kb sa[i,kb] * sb(j,kb) * P_kb[i,j],  P_kb = sum_{k in kb} A[i,k] B[j,k]
//
// with sa and sb arbitrary fp32 values, so every 128-wide K block's partial
// product leaves the tensor core and is scaled and summed on the CUDA cores.
//
// Why pairs: a 128 x 256 tile on one SM pulls 48 KB of operands from L2 per
// K block; a 256 x 256 tile on a CTA pair runs one MMA stream issued by the
// leader CTA over both SMs' shared memory: A is split along M (each CTA loads
// its 128 rows) and B along N (each CTA loads 128 of the 256 rows), so each
// SM pulls 32 KB per K block for the same work.
//
// Measured standing (GB300, fp32 scales, L2 flushed): it matches the
// single-SM promotion kernel but does not beat it (8192 x 8192 x 7168: 429 us
// against 421 us), so it runs only when requested (ql_set_gemm_path(5)).
// Throw-away ablations located the limit: without the FMAs the pair kernel
// takes 300 us, without the FMAs and the partial-product loads 298 us, and
// without the scale loads as well the skeleton of copies, MMAs and hand-offs
// still takes about 273 us, 730 cycles per K block against 549 for the MMAs.
// The two 256-column accumulator stages that fill tensor memory make the MMA
// of K block kb+2 wait until both CTAs' math warps have read kb, and the
// commit -> read -> release -> issue round trip (about 900 cycles) is longer
// than one K block's MMAs. 128-column tiles (four stages) measured slower
// (547 us): their operand traffic per flop is the single-SM kernel's again.
// The peer CTA's release is a relaxed remote arrive: with release semantics
// at cluster scope it waited on the thread's outstanding memory operations and
// the kernel ran at half speed (842 us).
//
// Roles (384 threads per CTA, one CTA per SM, clusters of 2):
//   warp 0      TMA producer in each CTA: its A rows and B rows of each K
//               block; both CTAs' copies complete on the leader's "full"
//               barrier, armed by the leader for the pair's bytes.
//   warp 1      leader: tensor memory owner and MMA issuer; per K block four
//               cta_group::2 kind::f8f6f4 MMAs (K = 32 each) into a fresh
//               tensor-memory stage (two stages of 256 columns), commits
//               multicast to both CTAs (operand stage free, partial product
//               ready).
//   warps 2-3   scale loaders in each CTA: sa of its 128 rows and sb of the
//               tile's columns per K block into its own shared-memory ring.
//   warps 4-11  math in each CTA: thread (quarter q, lane l) owns row
//               32q + l of the CTA's 128 and 128 of the 256 columns; per K
//               block it reads the partial product (tcgen05.ld), the warp
//               releases the stage to the leader (one arrive), and it
//               promotes acc += (sa*sb) * P with fp32 FMAs; after
//               the last K block the rows leave through shared memory and
//               TMA tile stores.
// Every wait is bounded in time; on a time-out the CTA raises the device
// status word and both CTAs drain their copies and MMAs before tensor memory
// is freed (the exit protocol of the block-scaled pair kernel).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"
#include "epilogue_tma.cuh"
#include "gemm.cuh"
#include "promote.cuh"

namespace ql {
namespace {

constexpr int kThreads = 384;
constexpr int kMathThreads = 256;
constexpr int kMathWarps = kMathThreads / 32;
constexpr int BM = 128;         // rows of A per CTA (256 per pair)
constexpr int BK = 128;         // K block = scale granularity
constexpr int kScaleSlots = 16;   // K blocks of scales ahead of the math (global-load latency)

// BN: columns of D per pair tile (128 or 256); each CTA loads BN / 2 rows of
// B and holds all BN columns of its 128 rows in tensor memory, in 512 / BN
// stages (all of tensor memory).
template <int BN, bool PER_ROW_B, bool OUT_F32>
struct PairCfg {
    static constexpr int BNH = BN / 2;
    static constexpr int kTmemStages = 512 / BN;
    static constexpr int kStageA = BM * BK;
    static constexpr int kStageB = BNH * BK;
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr int kSbPerSlot = PER_ROW_B ? BN : 4;
    static constexpr int kSlotFloats = BM + kSbPerSlot;
    static constexpr int kCPT = BN / 2;                 // columns per math thread
    // staged output: one 32-row x 64-byte buffer (64-byte swizzle) per math warp
    static constexpr int kOutWarpBytes = 32 * 64;
    static constexpr int kFixed = kScaleSlots * kSlotFloats * 4 + 256 + 8 * kOutWarpBytes + 2048;
    static constexpr int kStages = (8 * kStageBytes + kFixed <= 232448) ? 8 : ((6 * kStageBytes + kFixed <= 232448) ? 6 : 5);
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kStageA;
    static constexpr int kOffScale = kOffB + kStages * kStageB;
    static constexpr int kOffBar = kOffScale + kScaleSlots * kSlotFloats * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kTmemStages + 2 * kScaleSlots + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffStage = ((kOffMisc + 16 + 1023) / 1024) * 1024;
    static constexpr int kSmemBytes = kOffStage + 8 * kOutWarpBytes + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kStageB % 1024 == 0 && kStageA % 1024 == 0, "stages stay 1024-byte aligned");
};

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mb, int& nb) {
    const int group_size = p.group_m * p.tiles_n;
    const int group = t / group_size;
    const int first_m = group * p.group_m;
    const int rem = p.tiles_m - first_m;
    const int gm = rem < p.group_m ? rem : p.group_m;
    const int w = t - group * group_size;
    mb = first_m + w % gm;
    nb = w / gm;
}

template <int BN, bool PER_ROW_B, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_d, const GemmParams p) {
    using C = PairCfg<BN, PER_ROW_B, OUT_F32>;
    constexpr int BNH = C::BNH;
    constexpr int kTmemStages = C::kTmemStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;                       // leader: both CTAs' copies landed
    uint64_t* empty = full + C::kStages;         // stage free (multicast commit)
    uint64_t* tfull = empty + C::kStages;        // partial product ready (multicast commit)
    uint64_t* tempty = tfull + kTmemStages;      // leader: both CTAs' math warps read it
    uint64_t* sfull = tempty + kTmemStages;      // this CTA's scale slot written
    uint64_t* sempty = sfull + kScaleSlots;      // this CTA's scale slot read
    uint64_t* done_bar = sempty + kScaleSlots;   // leader: every MMA completed
    uint32_t* tmem_base_sm = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(num_clusters_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        // the math warps release stages and scale slots one arrive per warp
        for (int s = 0; s < kTmemStages; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], 2 * kMathWarps); }
        for (int s = 0; s < kScaleSlots; ++s) { mbar_init(&sfull[s], 32); mbar_init(&sempty[s], kMathWarps); }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        *peer_issued = 0;
        fence_mbar_init();
    }
    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        // the first tile's first weight tiles (this CTA's half) into L2 while the
        // previous kernel finishes
        if (cid < p.tiles_m * p.tiles_n) {
            int mb0, nb0;
            tile_coords(cid, p, mb0, nb0);
            const int brow0 = nb0 * BN + static_cast<int>(rank) * BNH;
            for (int kb = 0; kb < p.num_kb && kb < C::kStages; ++kb) {
                if (p.b_mn) tma_prefetch_l2_2d(&tmap_b, brow0, kb * BK);
                else tma_prefetch_l2_2d(&tmap_b, kb * BK, brow0);
            }
        }
    }
    if (warp == 1) { tmem_alloc_pair(tmem_base_sm, 512); tmem_relinquish_pair(); }
    tc_fence_before_sync();
    cluster_sync_all();          // barriers of both CTAs initialised before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_sm;
    pdl_wait_prior();            // inputs of the previous kernel are complete from here on

    const WaitCtl ctl{abort_flag, p.dev_status, p.wait_limit_ns};
    const int num_tiles = p.tiles_m * p.tiles_n;     // pair tiles of 256 x 256
    const int num_kb = p.num_kb;
    uint32_t issued = 0;                         // stages this CTA's producer issued

    if (warp < 4) {
        regs_dealloc<88>();   // 128 x 88 + 256 x 208 = 384 x 168 registers
        if (warp == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            if (elect_one()) {
                uint32_t it = 0;
                bool ok = true;
                const uint32_t leader_full0 = mapa_shared(&full[0], 0);
                for (int t = cid; t < num_tiles && ok && !p.stall_producer; t += ncl) {
                    int mb, nb;
                    tile_coords(t, p, mb, nb);
                    const int a_row = mb * 2 * BM + static_cast<int>(rank) * BM;
                    const int b_row = nb * BN + static_cast<int>(rank) * BNH;
                    for (int kb = 0; kb < num_kb; ++kb, ++it) {
                        const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                        if (!mbar_wait(&empty[s], ph ^ 1u, ctl)) { ok = false; break; }
                        uint8_t* a_dst = sA + s * C::kStageA;
                        uint8_t* b_dst = sB + s * C::kStageB;
                        if (leader) {
                            mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
                            if (p.a_mn) tma_load_2d(a_dst, &tmap_a, &full[s], a_row, kb * BK);
                            else tma_load_2d(a_dst, &tmap_a, &full[s], kb * BK, a_row);
                            if (p.b_mn) tma_load_2d(b_dst, &tmap_b, &full[s], b_row, kb * BK);
                            else tma_load_2d(b_dst, &tmap_b, &full[s], kb * BK, b_row);
                        } else {
                            const uint32_t fb = leader_full0 + s * 8u;
                            if (p.a_mn) tma_load_2d_pair(a_dst, &tmap_a, fb, a_row, kb * BK);
                            else tma_load_2d_pair(a_dst, &tmap_a, fb, kb * BK, a_row);
                            if (p.b_mn) tma_load_2d_pair(b_dst, &tmap_b, fb, b_row, kb * BK);
                            else tma_load_2d_pair(b_dst, &tmap_b, fb, kb * BK, b_row);
                        }
                    }
                }
                issued = it;
                if (!leader) st_shared_cluster(mapa_shared(const_cast<uint32_t*>(peer_issued), 0), it);
            }
            issued = __reduce_max_sync(0xffffffffu, issued);   // every lane knows the count
        } else if (warp == 1) {
            if (leader) {
                // ---------------- MMA issuer for the pair ----------------
                if (elect_one()) {
                    const uint32_t idesc = idesc_e4m3_f32(2 * BM, BN) | idesc_mn_bits(p.a_mn, p.b_mn);
                    const uint64_t astep = k32_step(p.a_mn), bstep = k32_step(p.b_mn);
                    uint32_t it = 0;
                    bool ok = true;
                    for (int t = cid; t < num_tiles && ok; t += ncl) {
                        for (int kb = 0; kb < num_kb; ++kb, ++it) {
                            const uint32_t ts = it % kTmemStages, tph = (it / kTmemStages) & 1u;
                            if (!mbar_wait_cluster(&tempty[ts], tph ^ 1u, ctl)) { ok = false; break; }
                            tc_fence_after_sync();
                            const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                            if (!mbar_wait_cluster(&full[s], ph, ctl)) { ok = false; break; }
                            tc_fence_after_sync();
                            const uint64_t adesc = sw128_desc(smem_addr(sA + s * C::kStageA), p.a_mn);
                            const uint64_t bdesc = sw128_desc(smem_addr(sB + s * C::kStageB), p.b_mn);
                            const uint32_t d_tmem = tmem_base + ts * BN;
#pragma unroll
                            for (int k4 = 0; k4 < BK / 32; ++k4)
                                mma_e4m3_pair(d_tmem, adesc + astep * k4, bdesc + bstep * k4, idesc, k4 > 0 ? 1u : 0u);
                            mma_commit_pair_multicast(&empty[s], 0x3);
                            mma_commit_pair_multicast(&tfull[ts], 0x3);
                        }
                    }
                    // every MMA has completed before tensor memory is freed
                    mma_commit_pair_multicast(done_bar, 0x1);
                    mbar_wait_drain(done_bar, 0, p.wait_limit_ns);
                }
            }
            __syncwarp();
        } else {
            // ---------------- scale loaders (both CTAs) ----------------
            // Warps 2 and 3 take alternate runs of K blocks (four, or two when B
            // has a scale per row); all loads of a run are issued before any is
            // stored, so a run costs one memory round trip.
            constexpr int kRun = PER_ROW_B ? 2 : 4;
            constexpr int kSbLoads = PER_ROW_B ? BN / 32 : 1;
            const uint32_t mine = static_cast<uint32_t>(warp - 2);
            uint32_t g = 0, run = 0;
            bool ok = true;
            const int64_t nblocks_b = (p.n + 127) / 128;
            for (int t = cid; t < num_tiles && ok; t += ncl) {
                int mb, nb;
                tile_coords(t, p, mb, nb);
                const int64_t m0 = static_cast<int64_t>(mb) * 2 * BM + rank * BM;
                const int64_t n0 = static_cast<int64_t>(nb) * BN;
                for (int kb0 = 0; kb0 < num_kb; kb0 += kRun, ++run) {
                    const int cnt = num_kb - kb0 < kRun ? num_kb - kb0 : kRun;
                    if ((run & 1u) != mine) { g += cnt; continue; }
                    float va[kRun][4], vb[kRun][kSbLoads];
#pragma unroll
                    for (int j = 0; j < kRun; ++j) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int64_t row = m0 + lane + 32 * i;
                            va[j][i] = (j < cnt && row < p.m) ? decode_scale(p.sfa, p.fmt, row * p.sam, kb0 + j, p.sak, p.bnd, 0)
                                                              : 0.0f;
                        }
#pragma unroll
                        for (int i = 0; i < kSbLoads; ++i) {
                            float v = 0.0f;
                            if (j < cnt) {
                                if constexpr (PER_ROW_B) {
                                    const int64_t col = n0 + lane + 32 * i;
                                    if (col < p.n) v = decode_scale(p.sfb, p.fmt, col * p.sbn, kb0 + j, p.sbk, p.bnd, 1);
                                } else {
                                    const int64_t r = n0 / 128 + lane;
                                    if (lane < (BN + 127) / 128 && r < nblocks_b)
                                        v = decode_scale(p.sfb, p.fmt, r * p.sbn, kb0 + j, p.sbk, p.bnd, 1);
                                }
                            }
                            vb[j][i] = v;
                        }
                    }
                    for (int j = 0; j < cnt; ++j) {
                        const uint32_t gj = g + j;
                        const uint32_t slot = gj % kScaleSlots, ph = (gj / kScaleSlots) & 1u;
                        if (!warp_wait(&sempty[slot], ph ^ 1u, ctl)) { ok = false; break; }
                        float* dst = sScale + slot * C::kSlotFloats;
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = va[j][i];
                        if constexpr (PER_ROW_B) {
#pragma unroll
                            for (int i = 0; i < kSbLoads; ++i) dst[BM + lane + 32 * i] = vb[j][i];
                        } else {
                            if (lane < (BN + 127) / 128) dst[BM + lane] = vb[j][0];
                        }
                        mbar_arrive(&sfull[slot]);
                    }
                    if (!ok) break;
                    g += cnt;
                }
            }
        }
    } else {
        regs_alloc<208>();
        // ---------------- math (both CTAs): promotion + epilogue ----------------
        constexpr int CPT = C::kCPT;
        const int wg = (warp - 4) >> 2;          // column half
        const int q = warp & 3;                  // TMEM lane quarter
        const int r_local = q * 32 + lane;       // accumulator row in this CTA's 128
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const bool vec_store = p.vec_store != 0;
        const uint32_t leader_tempty0 = mapa_shared(&tempty[0], 0);
        float acc[CPT];
        uint32_t g = 0;
        bool ok = true;
        for (int t = cid; t < num_tiles && ok; t += ncl) {
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const int64_t row = static_cast<int64_t>(mb) * 2 * BM + rank * BM + r_local;
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
            for (int kb = 0; kb < num_kb; ++kb, ++g) {
                const uint32_t slot = g % kScaleSlots, sph = (g / kScaleSlots) & 1u;
                const uint32_t ts = g % kTmemStages, tph = (g / kTmemStages) & 1u;
                if (!warp_wait(&sfull[slot], sph, ctl)) { ok = false; break; }
                const float* src = sScale + slot * C::kSlotFloats;
                const float sa = src[r_local];
                if (!warp_wait(&tfull[ts], tph, ctl)) { ok = false; break; }
                tc_fence_after_sync();
                const uint32_t tcol = tmem_base + lane_base + ts * BN + wg * CPT;
                constexpr int U = 64;                 // columns per TMEM read round
#pragma unroll
                for (int c0 = 0; c0 < CPT; c0 += U) {
                    uint32_t v[U];
                    tmem_load_cols<U>(tcol + c0, v);
                    if (c0 + U == CPT) {
                        // last read of this stage: once every lane's loads are
                        // complete, one arrive per warp releases it to the
                        // leader; the peer's is relaxed, since it publishes no
                        // memory writes (a release at cluster scope would wait
                        // for all of the thread's outstanding memory operations)
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if (leader) mbar_arrive(&tempty[ts]);
                            else mbar_arrive_remote_relaxed(leader_tempty0 + ts * 8u);
                        }
                    }
                    // one fp32 FMA per element (single rounding); the packed
                    // f32x2 form retires the same 32 FMAs per clock per SMSP
                    // and would need the accumulators paired and unpaired
                    if constexpr (!PER_ROW_B) {
                        const float sab = sa * src[BM + ((BN == 256) ? wg : 0)];
#pragma unroll
                        for (int j = 0; j < U; ++j) acc[c0 + j] = fmaf(__uint_as_float(v[j]), sab, acc[c0 + j]);
                    } else {
                        const float* sbp = src + BM + wg * CPT + c0;
#pragma unroll
                        for (int j = 0; j < U; ++j) acc[c0 + j] = fmaf(__uint_as_float(v[j]), sa * sbp[j], acc[c0 + j]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[slot]);
            }
            if (!ok) break;
            // ---------------- epilogue ----------------
            const int64_t col0 = static_cast<int64_t>(nb) * BN + wg * CPT;
            if (p.tma_d) {
                // this warp's 32 rows through its staging buffer and TMA tile
                // stores (rows and columns outside D are dropped by the copy)
                uint8_t* stg = smem + C::kOffStage + (warp - 4) * C::kOutWarpBytes;
                const int32_t y = static_cast<int32_t>(static_cast<int64_t>(mb) * 2 * BM + rank * BM + q * 32);
                tma_store_warp_rows<CPT, 64, OUT_F32>(acc, stg, &tmap_d, col0, y, p.accumulate != 0);
                continue;
            }
            if (row < p.m) {
                if constexpr (!OUT_F32) {
                    __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.d) + row * p.ldd;
#pragma unroll
                    for (int j = 0; j < CPT; j += 8) {
                        const int64_t c = col0 + j;
                        if (vec_store && c + 8 <= p.n) {
                            uint4 u;
                            __nv_bfloat162 h0 = __floats2bfloat162_rn(acc[j], acc[j + 1]);
                            __nv_bfloat162 h1 = __floats2bfloat162_rn(acc[j + 2], acc[j + 3]);
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[j + 4], acc[j + 5]);
                            __nv_bfloat162 h3 = __floats2bfloat162_rn(acc[j + 6], acc[j + 7]);
                            u.x = *reinterpret_cast<uint32_t*>(&h0);
                            u.y = *reinterpret_cast<uint32_t*>(&h1);
                            u.z = *reinterpret_cast<uint32_t*>(&h2);
                            u.w = *reinterpret_cast<uint32_t*>(&h3);
                            if (QL_IN(p.bnd, 2, drow + c, 16)) *reinterpret_cast<uint4*>(drow + c) = u;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (c + e < p.n && QL_IN(p.bnd, 2, drow + c + e, 2)) drow[c + e] = __float2bfloat16_rn(acc[j + e]);
                        }
                    }
                } else {
                    float* drow = static_cast<float*>(p.d) + row * p.ldd;
#pragma unroll
                    for (int j = 0; j < CPT; j += 4) {
                        const int64_t c = col0 + j;
                        if (vec_store && c + 4 <= p.n) {
                            if (!QL_IN(p.bnd, 2, drow + c, 16)) continue;
                            float4 o = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                            if (p.accumulate) {
                                const float4 old = *reinterpret_cast<const float4*>(drow + c);
                                o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
                            }
                            *reinterpret_cast<float4*>(drow + c) = o;
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (c + e < p.n && QL_IN(p.bnd, 2, drow + c + e, 4))
                                    drow[c + e] = p.accumulate ? drow[c + e] + acc[j + e] : acc[j + e];
                        }
                    }
                }
            }
        }
        // the staged tiles' copies are complete before the buffers go away
        if (p.tma_d && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    cluster_sync_all();          // every role of both CTAs has stopped issuing
    // Drain every copy of the last kStages stages either CTA issued. After a
    // time-out the two producers may have stopped at different stages: a stage
    // only the peer issued is armed now for the peer's bytes, and a stage only
    // the leader issued gives up the peer's share it was armed for.
    if (leader && warp == 0 && lane == 0) {
        const uint32_t it_l = issued, it_p = *peer_issued;
        const uint32_t hi = it_l > it_p ? it_l : it_p;
        const uint32_t lo = hi > static_cast<uint32_t>(C::kStages) ? hi - C::kStages : 0u;
        for (uint32_t j = lo; j < hi; ++j) {
            const uint32_t s = j % C::kStages, ph = (j / C::kStages) & 1u;
            if (j >= it_l) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            else if (j >= it_p) mbar_complete_tx(&full[s], C::kStageBytes);
            mbar_wait_drain(&full[s], ph, p.wait_limit_ns);
        }
    }
    __syncwarp();
    cluster_sync_all();          // no copy, MMA or remote arrive of either CTA is still in flight
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

template <int BN, bool PER_ROW_B, bool OUT_F32>
cudaError_t launch_pair_t(const GemmLaunch& L, GemmParams p, cudaStream_t st, int num_sms) {
    using Cf = PairCfg<BN, PER_ROW_B, OUT_F32>;
    constexpr int BNH = Cf::BNH;
    CUtensorMap ta, tb;
    if (!(L.a_mn ? encode_kmajor_map(&ta, L.a, L.k, L.m, L.lda, BK) : encode_kmajor_map(&ta, L.a, L.m, L.k, L.lda, BM)))
        return cudaErrorInvalidValue;
    if (!(L.b_mn ? encode_kmajor_map(&tb, L.b, L.k, L.n, L.ldb, BK) : encode_kmajor_map(&tb, L.b, L.n, L.k, L.ldb, BNH)))
        return cudaErrorInvalidValue;
    // bf16 / fp32 output through TMA tile stores when D's rows start and end 16-byte aligned
    CUtensorMap td = {};
    p.tma_d = 0;
    constexpr int es = OUT_F32 ? 4 : 2;
    // a TMA store may write a row's last 16-byte chunk whole, so D's rows must end on one
    if ((reinterpret_cast<uintptr_t>(L.d) & 15u) == 0 && L.ldd > 0 && (L.ldd * es) % 16 == 0 && (L.n * es) % 16 == 0 &&
        encode_2d_map(&td, L.d, OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, L.m, L.n,
                      L.ldd * es, 32, 64 / es, /*swizzle=*/64))
        p.tma_d = 1;
    p.tiles_m = static_cast<int>((L.m + 2 * BM - 1) / (2 * BM));
    p.tiles_n = static_cast<int>((L.n + BN - 1) / BN);
    const int tiles = p.tiles_m * p.tiles_n;
    int pairs = num_sms / 2;
    if (pairs < 1) pairs = 1;
    if (tiles < pairs) pairs = tiles;
    auto kern = gemm_fp8_pair_kernel<BN, PER_ROW_B, OUT_F32>;
    if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), Cf::kSmemBytes); e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a persistent grid of no more pairs than can be resident at once
    const int max_pairs = max_active_clusters(reinterpret_cast<const void*>(kern), cfg);
    if (pairs > max_pairs) pairs = max_pairs;
    return launch_gemm_kernel(kern, static_cast<unsigned>(2 * pairs), 2, Cf::kSmemBytes, st, ta, tb, td, p);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmLaunch& L, const GemmParams& p, cudaStream_t st, int num_sms) {
    if (L.out_f32) return launch_pair_t<256, true, true>(L, p, st, num_sms);
    return launch_pair_t<256, false, false>(L, p, st, num_sms);
}

}  // namespace ql
