// Block-scaled FP8 GEMM on CTA pairs (tcgen05 cta_group::2) for UE8M0 scales.
//
// Same product as gemm_mx.cu ("DeepGEMM Essentials: High-Performance FP8
// Matrix Multiplication" Parts 1, 6, 12-13; RHS scales read row-wise per
// "[Help] Starter script for nn.Linear for fwd,bwd"), computed on 256 x 256
// tiles by a cluster of two CTAs on neighbouring SMs. The pair's tensor cores
// run one MMA stream issued by the leader CTA: A is split along M (each CTA
// holds its 128 rows) and B along N (each CTA holds 128 of the 256 columns'
// rows), so a pipeline stage is 32 KB per SM instead of 48 KB for a 128 x 256
// tile on one SM. That halves the B bytes each SM pulls from L2 and leaves room
// for six stages in flight.
//
// Roles (384 threads per CTA, one CTA per SM, clusters of 2):
//   warp 0      TMA producer in each CTA: its A rows and B rows of each
//               128-wide K block. Both CTAs' copies complete on the leader's
//               "full" barrier, which the leader arms for the pair's bytes.
//   warp 1      leader: MMA issuer (tcgen05.cp of the exponents, then 4 x 4
//               block-scaled cta_group::2 MMAs per K group); commits are
//               multicast to both CTAs.
//   warps 2-3   exponent loaders in each CTA (as in gemm_mx.cu) for its A rows
//               and all 256 B rows (each CTA's tensor memory holds the B
//               exponents of the whole tile), arriving on the leader's barrier.
//   warps 4-11  epilogue in each CTA: its 128 rows x 256 columns of D.
// Exit: a cluster barrier; then the leader drains every copy either CTA
// issued (balancing stages that only one side armed or issued, after a
// time-out); a second cluster barrier; then tensor memory is freed.
//
// Tile width: 256 columns leave room in tensor memory (512 columns) for one
// fp32 accumulator beside the exponents, so the next tile's MMAs wait until
// both epilogues have read the last one out. 224-column tiles fit two
// accumulators (at columns 0 and 256) and the exponents (at 480): the MMAs of
// tile t+1 run while the epilogues drain tile t. The 224-wide form is the
// default; 256 remains for the E4M3-output epilogue (whole 128-column groups
// per thread) and for MN-major B (one 128-byte swizzle atom per CTA).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"
#include "epilogue_fp8.cuh"
#include "epilogue_tma.cuh"
#include "gemm.cuh"

namespace ql {
namespace {

constexpr int kThreads = 384;
constexpr int kMathThreads = 256;
constexpr int BM = 128;      // rows of A per CTA (256 per pair)
constexpr int BK = 128;
constexpr int kSfSlots = 8;

// BN: columns of D per pair (256 or 224); each CTA holds BN / 2 rows of B.
// OUT_BYTES: element size of a D that leaves through shared memory and TMA
// tile stores (1: E4M3, 2: bf16, 4: fp32; 0: stored directly). Each epilogue warp owns
// one buffer of 32 rows x kCW columns (rows of 128 bytes with the 128-byte
// swizzle, or 112 bytes unswizzled, whose pitch already spreads 8 consecutive
// rows over all banks); the operand ring gives up a stage when the buffers do
// not fit beside six.
template <int BN, int OUT_BYTES = 0>
struct Mx2Cfg {
    static constexpr int BNH = BN / 2;
    static constexpr int kStageA = BM * BK;
    static constexpr int kStageB = BNH * BK;
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr bool kStageOut = OUT_BYTES != 0;
    static constexpr int kCW = OUT_BYTES == 4 ? 32 : (OUT_BYTES == 1 ? 128 : ((BN / 2) % 64 == 0 ? 64 : 56));
    static constexpr int kRB = kCW * (OUT_BYTES == 0 ? 2 : OUT_BYTES);               // bytes per staged row
    static constexpr bool kOutSwizzle = kRB == 128;
    static constexpr int kOutWarpBytes = 32 * kRB;
    static constexpr int kSfbChunks = 2;         // all B rows of the tile (up to 256) in each CTA
    // six operand stages unless the output buffers leave room for five only:
    // bytes besides the ring (exponent slots, barriers for two accumulators, misc)
    static constexpr int kFixedBytes = kSfSlots * (BM + 128 * kSfbChunks) * 4 + (2 * 2 + 2 * kSfSlots + 3) * 8 + 16;
    static constexpr int kStages =
        ((6 * (kStageBytes + 16) + kFixedBytes + 1023) / 1024) * 1024 + (kStageOut ? 8 * kOutWarpBytes : 0) + 1024 <=
                232448
            ? 6
            : 5;
    static constexpr int kSfCols = 4 + 4 * kSfbChunks;
    static constexpr int kTmemCols = 512;
    static constexpr int kAccStride = 256;       // accumulator stages start on 256-column boundaries
    static constexpr int kAccStages = (kAccStride + BN + 2 * kSfCols <= kTmemCols) ? 2 : 1;
    static constexpr int kSfColBase = (kAccStages - 1) * kAccStride + BN;
    static constexpr int kSlotWords = BM + 128 * kSfbChunks;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kStageA;
    static constexpr int kOffSf = kOffB + kStages * kStageB;
    static constexpr int kOffBar = kOffSf + kSfSlots * kSlotWords * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kAccStages + 2 * kSfSlots + 2 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffStage = kStageOut ? ((kOffMisc + 16 + 1023) / 1024) * 1024 : kOffMisc + 16;
    static constexpr int kSmemBytes = kOffStage + (kStageOut ? 8 * kOutWarpBytes : 0) + 1024;
    static_assert(BN % 32 == 0 && BN <= 256, "pair tile width");
    static_assert(!kStageOut || (BN / 2) % kCW == 0, "staged output takes whole chunks");
    static_assert(kRB % 16 == 0 && (!kOutSwizzle || kRB == 128), "16-byte chunks per staged row");
    static_assert(kStageB % 1024 == 0, "B stages stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kSfColBase + 2 * kSfCols <= kTmemCols, "tensor memory budget");
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

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl)) != 0;
}

// Exponent words of K group g for R scale rows (see gemm_mx.cu).
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

template <int BN, bool PER_ROW_B, bool OUT_F32, bool OUT_FP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx2_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const GemmParams p) {
    using C = Mx2Cfg<BN, OUT_FP8 ? 1 : (OUT_F32 ? 4 : 2)>;
    constexpr int BNH = C::BNH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    uint32_t* sSf = reinterpret_cast<uint32_t*>(smem + C::kOffSf);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;                       // leader: both CTAs' copies landed
    uint64_t* empty = full + C::kStages;         // stage free (multicast commit)
    uint64_t* tfull = empty + C::kStages;        // [kAccStages] accumulator ready (multicast commit)
    uint64_t* tempty = tfull + C::kAccStages;    // [kAccStages] leader: both epilogues drained it
    uint64_t* sfull = tempty + C::kAccStages;    // leader: both CTAs' exponent slots written
    uint64_t* sempty = sfull + kSfSlots;         // exponent slot free (multicast commit)
    uint64_t* sftfree = sempty + kSfSlots;       // leader: TMEM exponent stage free
    uint64_t* done_bar = sftfree + 2;
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
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *peer_issued = 0;
        for (int s = 0; s < C::kAccStages; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], 2 * kMathThreads);
        }
        for (int s = 0; s < kSfSlots; ++s) { mbar_init(&sfull[s], 64); mbar_init(&sempty[s], 1); }
        mbar_init(&sftfree[0], 1);
        mbar_init(&sftfree[1], 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
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
            for (int kb = 0; kb < p.num_kb && kb < C::kStages; ++kb) {
                const int brow0 = nb0 * BN + static_cast<int>(rank) * BNH;
                if (p.b_mn) tma_prefetch_l2_2d(&tmap_b, brow0, kb * BK);
                else tma_prefetch_l2_2d(&tmap_b, kb * BK, brow0);
            }
        }
    }
    if (warp == 1) { tmem_alloc_pair(tmem_base_sm, C::kTmemCols); tmem_relinquish_pair(); }
    tc_fence_before_sync();
    cluster_sync_all();          // barriers of both CTAs initialised before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_sm;
    pdl_wait_prior();            // inputs of the previous kernel are complete from here on

    const WaitCtl ctl{abort_flag, p.dev_status, p.wait_limit_ns};
    const int num_tiles = p.tiles_m * p.tiles_n;     // pair tiles of 256 x 256
    const int num_kb = p.num_kb;
    const int num_groups = (num_kb + 3) / 4;
    uint32_t issued = 0;                         // stages this CTA's producer issued

    if (warp < 4) {
        regs_dealloc<136>();  // 128 x 136 + 256 x 184 = 384 x 168 registers
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
                        if (leader) {
                            mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
                            if (p.a_mn) tma_load_2d(sA + s * C::kStageA, &tmap_a, &full[s], a_row, kb * BK);
                            else tma_load_2d(sA + s * C::kStageA, &tmap_a, &full[s], kb * BK, a_row);
                            if (p.b_mn) tma_load_2d(sB + s * C::kStageB, &tmap_b, &full[s], b_row, kb * BK);
                            else tma_load_2d(sB + s * C::kStageB, &tmap_b, &full[s], kb * BK, b_row);
                        } else {
                            if (p.a_mn) tma_load_2d_pair(sA + s * C::kStageA, &tmap_a, leader_full0 + s * 8u, a_row, kb * BK);
                            else tma_load_2d_pair(sA + s * C::kStageA, &tmap_a, leader_full0 + s * 8u, kb * BK, a_row);
                            if (p.b_mn) tma_load_2d_pair(sB + s * C::kStageB, &tmap_b, leader_full0 + s * 8u, b_row, kb * BK);
                            else tma_load_2d_pair(sB + s * C::kStageB, &tmap_b, leader_full0 + s * 8u, kb * BK, b_row);
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
                    uint32_t it = 0, g = 0, tc = 0;
                    bool ok = true;
                    for (int t = cid; t < num_tiles && ok; t += ncl, ++tc) {
                        const uint32_t as = tc % C::kAccStages, aph = (tc / C::kAccStages) & 1u;
                        if (!mbar_wait_cluster(&tempty[as], aph ^ 1u, ctl)) { ok = false; break; }
                        tc_fence_after_sync();
                        const uint32_t d_tmem = tmem_base + as * C::kAccStride;
                        for (int kg = 0; kg < num_groups && ok; ++kg, ++g) {
                            const uint32_t slot = g % kSfSlots, sph = (g / kSfSlots) & 1u;
                            const uint32_t st = g & 1u;
                            if (!mbar_wait_cluster(&sfull[slot], sph, ctl)) { ok = false; break; }
                            if (!mbar_wait(&sftfree[st], ((g >> 1) & 1u) ^ 1u, ctl)) { ok = false; break; }
                            tc_fence_after_sync();
                            const uint32_t sf_col = tmem_base + C::kSfColBase + st * C::kSfCols;
                            const uint32_t* slot_ptr = sSf + slot * C::kSlotWords;
                            tmem_cp_pair_32x128b_warpx4(sf_col, rows16_desc(smem_addr(slot_ptr)));
#pragma unroll
                            for (int c = 0; c < C::kSfbChunks; ++c)
                                tmem_cp_pair_32x128b_warpx4(sf_col + 4 + 4 * c,
                                                            rows16_desc(smem_addr(slot_ptr + BM + 128 * c)));
                            for (int kbi = 0; kbi < 4; ++kbi) {
                                const int kb = kg * 4 + kbi;
                                if (kb >= num_kb) break;
                                const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                                if (!mbar_wait_cluster(&full[s], ph, ctl)) { ok = false; break; }
                                tc_fence_after_sync();
                                const uint64_t adesc = sw128_desc(smem_addr(sA + s * C::kStageA), p.a_mn);
                                const uint64_t bdesc = sw128_desc(smem_addr(sB + s * C::kStageB), p.b_mn);
                                const uint32_t idesc =
                                    idesc_mxf8_ue8m0(2 * BM, BN, kbi, kbi) | idesc_mn_bits(p.a_mn, p.b_mn);
                                const uint64_t astep = k32_step(p.a_mn), bstep = k32_step(p.b_mn);
#pragma unroll
                                for (int k4 = 0; k4 < BK / 32; ++k4)
                                    mma_mxf8_block_scaled_pair(d_tmem, adesc + astep * k4, bdesc + bstep * k4, idesc,
                                                               sf_col, sf_col + 4, (kb > 0 || k4 > 0) ? 1u : 0u);
                                mma_commit_pair_multicast(&empty[s], 0x3);
                                ++it;
                            }
                            if (!ok) break;
                            mma_commit_pair_multicast(&sempty[slot], 0x3);
                            mma_commit_pair_multicast(&sftfree[st], 0x1);
                        }
                        if (!ok) break;
                        mma_commit_pair_multicast(&tfull[as], 0x3);
                    }
                    mma_commit_pair_multicast(done_bar, 0x1);
                    mbar_wait_drain(done_bar, 0, p.wait_limit_ns);
                }
            }
            __syncwarp();
        } else {
            // ---------------- exponent loaders (both CTAs) ----------------
            // a word per B row when B has per-row exponents or when the tile's
            // rows do not start on a 128-row block (224-wide tiles)
            constexpr bool kRowWords = PER_ROW_B || (BN % 128 != 0);
            constexpr int R = kRowWords ? 2 : 4;
            constexpr int NB = kRowWords ? 4 * C::kSfbChunks : C::kSfbChunks;
            const uint32_t mine = static_cast<uint32_t>(warp - 2);
            const int run_len = (p.fmt == 2) ? R : 1;
            const uint32_t leader_sfull0 = mapa_shared(&sfull[0], 0);
            uint32_t g = 0, run = 0;
            bool ok = true;
            const int64_t nblocks_b = (p.n + 127) / 128;
            for (int t = cid; t < num_tiles && ok; t += ncl) {
                int mb, nb;
                tile_coords(t, p, mb, nb);
                const int64_t a_row = static_cast<int64_t>(mb) * 2 * BM + rank * BM;
                const int64_t b_row0 = static_cast<int64_t>(nb) * BN;
                for (int kg0 = 0; kg0 < num_groups; kg0 += run_len, ++run) {
                    const int cnt = num_groups - kg0 < run_len ? num_groups - kg0 : run_len;
                    if ((run & 1u) != mine) { g += cnt; continue; }
                    uint32_t wa[R][4], wb[R][NB];
                    int64_t offa[4], offb[NB];
                    bool vala[4], valb[NB];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t row = a_row + 32 * q + lane;
                        vala[q] = row < p.m;
                        offa[q] = row * p.sam;
                    }
#pragma unroll
                    for (int i = 0; i < NB; ++i) {
                        if constexpr (kRowWords) {
                            const int64_t row = b_row0 + 32 * i + lane;    // chunk i/4, quarter i%4
                            valb[i] = row < p.n && 32 * i + lane < BN;
                            offb[i] = PER_ROW_B ? row * p.sbn : (row / 128) * p.sbn;
                        } else {
                            const int64_t r = b_row0 / 128 + i;            // chunk i: one block word
                            valb[i] = r < nblocks_b;
                            offb[i] = r * p.sbn;
                        }
                    }
                    if (p.fmt == 2) {
#pragma unroll
                        for (int j = 0; j < R; ++j) {
                            const bool in = j < cnt;
                            bool va[4], vb[NB];
#pragma unroll
                            for (int q = 0; q < 4; ++q) va[q] = vala[q] && in;
#pragma unroll
                            for (int i = 0; i < NB; ++i) vb[i] = valb[i] && in;
                            exp_words<4>(p.sfa, 2, offa, va, kg0 + j, p.sak, num_kb, wa[j], p.bnd, 0);
                            exp_words<NB>(p.sfb, 2, offb, vb, kg0 + j, p.sbk, num_kb, wb[j], p.bnd, 1);
                        }
                    } else {
                        exp_words<4>(p.sfa, p.fmt, offa, vala, kg0, p.sak, num_kb, wa[0], p.bnd, 0);
                        exp_words<NB>(p.sfb, p.fmt, offb, valb, kg0, p.sbk, num_kb, wb[0], p.bnd, 1);
                    }
                    for (int j = 0; j < cnt; ++j) {
                        const uint32_t gj = g + j;
                        const uint32_t slot = gj % kSfSlots, ph = (gj / kSfSlots) & 1u;
                        if (!warp_wait(&sempty[slot], ph ^ 1u, ctl)) { ok = false; break; }
                        uint32_t* dst = sSf + slot * C::kSlotWords;
                        *reinterpret_cast<uint4*>(dst + lane * 4) = make_uint4(wa[j][0], wa[j][1], wa[j][2], wa[j][3]);
#pragma unroll
                        for (int c = 0; c < C::kSfbChunks; ++c) {
                            uint4 v;
                            if constexpr (kRowWords) {
                                v = make_uint4(wb[j][4 * c], wb[j][4 * c + 1], wb[j][4 * c + 2], wb[j][4 * c + 3]);
                            } else {
                                v = make_uint4(wb[j][c], wb[j][c], wb[j][c], wb[j][c]);
                            }
                            *reinterpret_cast<uint4*>(dst + BM + 128 * c + lane * 4) = v;
                        }
                        fence_proxy_async_smem();   // visible to tcgen05.cp (async proxy)
                        if (leader) mbar_arrive(&sfull[slot]);
                        else mbar_arrive_remote(leader_sfull0 + slot * 8u);
                    }
                    if (!ok) break;
                    g += cnt;
                }
            }
        }
    } else {
        regs_alloc<184>();
        // ---------------- epilogue (both CTAs): 128 rows x 256 columns ----------------
        constexpr int CPT = BN / 2;
        const int wg = (warp - 4) >> 2;
        const int q = warp & 3;
        const int r_local = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const bool vec_store = p.vec_store != 0;
        const uint32_t leader_tempty0 = mapa_shared(&tempty[0], 0);
        uint32_t tc = 0;
        for (int t = cid; t < num_tiles; t += ncl, ++tc) {
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const uint32_t as = tc % C::kAccStages, aph = (tc / C::kAccStages) & 1u;
            if (!warp_wait(&tfull[as], aph, ctl)) break;
            tc_fence_after_sync();
            uint32_t accb[CPT];
            const uint32_t tcol = tmem_base + lane_base + as * C::kAccStride + wg * CPT;
            if constexpr (CPT % 32 == 0) {
#pragma unroll
                for (int c0 = 0; c0 < CPT; c0 += 32)
                    tmem_ld_32x32b_x32(tcol + c0, *reinterpret_cast<uint32_t(*)[32]>(&accb[c0]));
            } else {
                // 16-column loads, each starting on a 16-column boundary
#pragma unroll
                for (int c0 = 0; c0 < CPT; c0 += 16)
                    tmem_ld_32x32b_x16(tcol + c0, *reinterpret_cast<uint32_t(*)[16]>(&accb[c0]));
            }
            tmem_wait_ld(accb);            // one wait for all loads
            float* acc = reinterpret_cast<float*>(accb);
            tc_fence_before_sync();
            if (leader) mbar_arrive(&tempty[as]);
            else mbar_arrive_remote(leader_tempty0 + as * 8u);
            const int64_t row = static_cast<int64_t>(mb) * 2 * BM + rank * BM + r_local;
            const int64_t col0 = static_cast<int64_t>(nb) * BN + wg * CPT;
            if constexpr (C::kStageOut) {
                if (p.tma_d) {
                    // D rows through this warp's staging buffer and TMA tile stores
                    uint8_t* stg = smem + C::kOffStage + (warp - 4) * C::kOutWarpBytes;
                    const int32_t y = static_cast<int32_t>(static_cast<int64_t>(mb) * 2 * BM + rank * BM + q * 32);
                    if constexpr (OUT_FP8) {
                        // E4M3 bytes staged (one 128-byte row per lane), scales stored directly
                        static_assert(CPT == 128, "E4M3 output needs 128 columns per thread");
                        if (lane == 0) bulk_wait_read_all();     // the previous copy has read the buffer
                        __syncwarp();
                        stage_row_e4m3_any(acc, row, col0, p, stg + lane * 128, lane & 7, row < p.m);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmap_d, stg, static_cast<int32_t>(col0), y);
                            bulk_commit_group();
                        }
                    } else {
                        tma_store_warp_rows<CPT, C::kRB, OUT_F32>(acc, stg, &tmap_d, col0, y, p.accumulate != 0);
                    }
                    continue;
                }
            }
            if (row < p.m) {
                if constexpr (OUT_FP8) {
                    store_row_e4m3_any(acc, row, col0, p);
                } else if constexpr (!OUT_F32) {
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
        if constexpr (C::kStageOut) {
            // the staged tiles' copies are complete before the buffers go away
            if (p.tma_d && lane == 0) bulk_wait_all();
            __syncwarp();
        }
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
        tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
}

template <int BN, bool PER_ROW_B, bool OUT_F32, bool OUT_FP8 = false>
cudaError_t launch_mx2_t(const GemmLaunch& L, GemmParams p, cudaStream_t st, int num_sms) {
    using Cf = Mx2Cfg<BN, OUT_FP8 ? 1 : (OUT_F32 ? 4 : 2)>;
    constexpr int BNH = Cf::BNH;
    CUtensorMap ta, tb;
    if (!(L.a_mn ? encode_kmajor_map(&ta, L.a, L.k, L.m, L.lda, BK) : encode_kmajor_map(&ta, L.a, L.m, L.k, L.lda, BM)))
        return cudaErrorInvalidValue;
    if (!(L.b_mn ? encode_kmajor_map(&tb, L.b, L.k, L.n, L.ldb, BK) : encode_kmajor_map(&tb, L.b, L.n, L.k, L.ldb, BNH)))
        return cudaErrorInvalidValue;
    // E4M3 / bf16 / fp32 output through TMA tile stores when D's rows start and end 16-byte aligned
    CUtensorMap td = {};
    p.tma_d = 0;
    if constexpr (Cf::kStageOut) {
        constexpr int es = OUT_FP8 ? 1 : (OUT_F32 ? 4 : 2);
        const CUtensorMapDataType dt = OUT_FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                               : (OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
        // a TMA store may write a row's last 16-byte chunk whole, so D's rows must end on one
        if ((reinterpret_cast<uintptr_t>(L.d) & 15u) == 0 && L.ldd > 0 && (L.ldd * es) % 16 == 0 &&
            (L.n * es) % 16 == 0 &&
            encode_2d_map(&td, L.d, dt, L.m, L.n, L.ldd * es, 32, Cf::kCW, Cf::kOutSwizzle ? 128 : 0))
            p.tma_d = 1;
    }
    p.tiles_m = static_cast<int>((L.m + 2 * BM - 1) / (2 * BM));
    p.tiles_n = static_cast<int>((L.n + BN - 1) / BN);
    const int tiles = p.tiles_m * p.tiles_n;
    int pairs = num_sms / 2;
    if (pairs < 1) pairs = 1;
    if (tiles < pairs) pairs = tiles;
    auto kern = gemm_mx2_kernel<BN, PER_ROW_B, OUT_F32, OUT_FP8>;
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
    if (pairs > max_pairs) {
        pairs = max_pairs;
        cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    }
    return launch_gemm_kernel(kern, cfg.gridDim.x, 2, Cf::kSmemBytes, st, ta, tb, td, p);
}

}  // namespace

cudaError_t launch_gemm_mx2(const GemmLaunch& L, const GemmParams& p, cudaStream_t st, int num_sms) {
    if (L.out_fp8) return launch_mx2_t<256, false, false, true>(L, p, st, num_sms);
    if (L.b_mn) {
        if (L.out_f32) return launch_mx2_t<256, true, true>(L, p, st, num_sms);
        return launch_mx2_t<256, false, false>(L, p, st, num_sms);
    }
    if (L.out_f32) return launch_mx2_t<256, true, true>(L, p, st, num_sms);
    return launch_mx2_t<224, false, false>(L, p, st, num_sms);
}

}  // namespace ql
