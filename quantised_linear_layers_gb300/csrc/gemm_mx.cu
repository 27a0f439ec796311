// Block-scaled FP8 GEMM for UE8M0 (power-of-two) scales on sm_103a.
//
// Same product as the promotion kernel in gemm.cu ("DeepGEMM Essentials:
// High-Performance FP8 Matrix Multiplication" Parts 1, 6, 12-13; RHS scales
// read row-wise per "[Help] Starter script for nn.Linear for fwd,bwd"):
//
//   D[i,j] = sum_kb 2^(ea[i,kb]-127) * 2^(eb(j,kb)-127) * sum_{k in kb} A[i,k] B[j,k]
//
// When every scale is a power of two the per-K-block promotion can be done by
// the tensor core itself: tcgen05.mma.kind::mxf8f6f4.block_scale multiplies
// each 32-wide K slice by one UE8M0 scale per row of A and per row of B, read
// from tensor memory. A 128-wide K block is four such slices with the same
// exponent byte, so the whole K loop accumulates in one TMEM accumulator and
// the math warps touch it once per tile.
//
// Roles (384 threads, one persistent CTA per SM):
//   warp 0      TMA producer (as in gemm.cu).
//   warp 1      MMA issuer: per group of four K blocks, tcgen05.cp copies the
//               group's exponents (one int32 word per row: four K-block bytes)
//               from shared to tensor memory, then issues 4 x 4 block-scaled
//               MMAs selecting byte kb % 4 through the scale IDs.
//   warps 2-3   scale loaders: per K group, one packed word per row of A and
//               per row of B (B's 128x128 block exponent, loaded once and
//               repeated over its 128 rows; wgrad: B's own per-row exponents),
//               several groups per memory round trip, stored in the order
//               tcgen05.cp's four-quarter layout expects: row 32q + r of a
//               128-row chunk goes to 16-byte line r, word q.
//   warps 4-11  epilogue: after a tile's last MMA, read the fp32 accumulator
//               out of TMEM into registers, release TMEM, convert and store
//               while the MMA warp already runs the next tile.
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
constexpr int BM = 128;
constexpr int BK = 128;
constexpr int kSfSlots = 8;          // shared-memory scale ring (K groups)

// OUT_BYTES: element size of a D that leaves through shared memory and TMA
// tile stores (2: bf16, 4: fp32; 0: stored directly). Each epilogue warp owns a
// 2 KB buffer of 32 rows x 64 bytes in the 64-byte swizzle (32 bf16 or 16 fp32
// columns per copy), which fits beside every tile width's operand ring.
template <int BN, int OUT_BYTES = 0>
struct MxCfg {
    static constexpr int kStageA = BM * BK;
    static constexpr int kStageB = BN * BK;
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr int kStages = (BN == 256) ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int kAccStages = BN == 256 ? 1 : 2;
    static constexpr int kSfbChunks = (BN + 127) / 128;
    static constexpr int kSfCols = 4 + 4 * kSfbChunks;     // per TMEM scale stage
    static constexpr int kSfColBase = kAccStages * BN;
    static constexpr int kTmemColsUsed = kSfColBase + 2 * kSfCols;
    static constexpr int kTmemCols = kTmemColsUsed <= 64 ? 64 : (kTmemColsUsed <= 128 ? 128 : (kTmemColsUsed <= 256 ? 256 : 512));
    static constexpr int kSlotWords = BM + 128 * kSfbChunks;
    static constexpr int kColsPerThread = BN / 2;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kStageA;
    static constexpr int kOffSf = kOffB + kStages * kStageB;
    static constexpr int kOffBar = kOffSf + kSfSlots * kSlotWords * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kAccStages + 2 * kSfSlots + 2 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kCW = OUT_BYTES == 0 ? 1 : 64 / OUT_BYTES;          // columns per copy
    static constexpr bool kStageOut = OUT_BYTES != 0 && (BN / 2) % kCW == 0;
    static constexpr int kOutWarpBytes = 32 * 64;
    static constexpr int kOffStage = kStageOut ? ((kOffMisc + 16 + 1023) / 1024) * 1024 : kOffMisc + 16;
    static constexpr int kSmemBytes = kOffStage + (kStageOut ? 8 * kOutWarpBytes : 0) + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kTmemColsUsed <= 512, "tensor memory budget");
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

// Exponent words of K group g for R scale rows at once (row r at element
// offset row_off[r]): fmt 2 reads the packed int32 word; fmt 1 (fp32 powers
// of two) gathers the exponent fields of the group's four K blocks. Every
// global load is issued before any is used, so a call costs one memory round
// trip. K blocks past num_kb contribute byte 0.
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
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_d, const GemmParams p) {
    using C = MxCfg<BN, OUT_FP8 ? 0 : (OUT_F32 ? 4 : 2)>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    uint32_t* sSf = reinterpret_cast<uint32_t*>(smem + C::kOffSf);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + C::kAccStages;
    uint64_t* sfull = tempty + C::kAccStages;
    uint64_t* sempty = sfull + kSfSlots;
    uint64_t* sftfree = sempty + kSfSlots;      // [2]: TMEM scale stage free again
    uint64_t* done_bar = sftfree + 2;
    uint32_t* tmem_base_sm = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int s = 0; s < C::kAccStages; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], kMathThreads); }
        for (int s = 0; s < kSfSlots; ++s) { mbar_init(&sfull[s], 32); mbar_init(&sempty[s], 1); }
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
        // the first tile's first weight tiles into L2 while the previous kernel finishes
        if (p.m_indices == nullptr && static_cast<int>(blockIdx.x) < p.tiles_m * p.tiles_n) {
            int mb0, nb0;
            tile_coords(blockIdx.x, p, mb0, nb0);
            for (int kb = 0; kb < p.num_kb && kb < C::kStages; ++kb) {
                if (p.b_mn) tma_prefetch_l2_2d(&tmap_b, nb0 * BN, kb * BK);
                else tma_prefetch_l2_2d(&tmap_b, kb * BK, nb0 * BN);
            }
        }
    }
    if (warp == 1) { tmem_alloc(tmem_base_sm, C::kTmemCols); tmem_relinquish(); }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_sm;
    pdl_wait_prior();            // inputs of the previous kernel are complete from here on

    const WaitCtl ctl{abort_flag, p.dev_status, p.wait_limit_ns};
    const int num_tiles = p.tiles_m * p.tiles_n;
    const int num_kb = p.num_kb;
    const int num_groups = (num_kb + 3) / 4;

    if (warp < 4) {
        regs_dealloc<136>();  // 128 x 136 + 256 x 184 = 384 x 168 registers
        if (warp == 0) {
            if (elect_one()) {
                uint32_t it = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < num_tiles && ok && !p.stall_producer; t += gridDim.x) {
                    int mb, nb;
                    tile_coords(t, p, mb, nb);
                    const int e = tile_expert(p, mb, false);
                    if (e < 0) continue;
                    const int brow = static_cast<int>(e * p.b_group_rows) + nb * BN;
                    for (int kb = 0; kb < num_kb; ++kb, ++it) {
                        const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                        if (!mbar_wait(&empty[s], ph ^ 1u, ctl)) { ok = false; break; }
                        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                        if (p.a_mn) tma_load_2d(sA + s * C::kStageA, &tmap_a, &full[s], mb * BM, kb * BK);
                        else tma_load_2d(sA + s * C::kStageA, &tmap_a, &full[s], kb * BK, mb * BM);
                        if (p.b_mn) tma_load_2d(sB + s * C::kStageB, &tmap_b, &full[s], brow, kb * BK);
                        else tma_load_2d(sB + s * C::kStageB, &tmap_b, &full[s], kb * BK, brow);
                    }
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
                uint32_t it = 0, g = 0, tc = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                    int mb, nb;
                    tile_coords(t, p, mb, nb);
                    if (tile_expert(p, mb, false) < 0) continue;
                    const uint32_t as = tc % C::kAccStages, aph = (tc / C::kAccStages) & 1u;
                    ++tc;
                    if (!mbar_wait(&tempty[as], aph ^ 1u, ctl)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + as * BN;
                    for (int kg = 0; kg < num_groups && ok; ++kg, ++g) {
                        const uint32_t slot = g % kSfSlots, sph = (g / kSfSlots) & 1u;
                        const uint32_t st = g & 1u;
                        if (!mbar_wait(&sfull[slot], sph, ctl)) { ok = false; break; }
                        // the MMAs of group g-2 have finished reading this TMEM scale stage
                        if (!mbar_wait(&sftfree[st], ((g >> 1) & 1u) ^ 1u, ctl)) { ok = false; break; }
                        tc_fence_after_sync();
                        const uint32_t sf_col = tmem_base + C::kSfColBase + st * C::kSfCols;
                        const uint32_t* slot_ptr = sSf + slot * C::kSlotWords;
                        tmem_cp_32x128b_warpx4(sf_col, rows16_desc(smem_addr(slot_ptr)));
#pragma unroll
                        for (int c = 0; c < C::kSfbChunks; ++c)
                            tmem_cp_32x128b_warpx4(sf_col + 4 + 4 * c, rows16_desc(smem_addr(slot_ptr + BM + 128 * c)));
                        for (int kbi = 0; kbi < 4; ++kbi) {
                            const int kb = kg * 4 + kbi;
                            if (kb >= num_kb) break;
                            const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                            if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                            tc_fence_after_sync();
                            const uint64_t adesc = sw128_desc(smem_addr(sA + s * C::kStageA), p.a_mn);
                            const uint64_t bdesc = sw128_desc(smem_addr(sB + s * C::kStageB), p.b_mn);
                            const uint32_t idesc = idesc_mxf8_ue8m0(BM, BN, kbi, kbi) | idesc_mn_bits(p.a_mn, p.b_mn);
                            const uint64_t astep = k32_step(p.a_mn), bstep = k32_step(p.b_mn);
#pragma unroll
                            for (int k4 = 0; k4 < BK / 32; ++k4)
                                mma_mxf8_block_scaled(d_tmem, adesc + astep * k4, bdesc + bstep * k4, idesc, sf_col,
                                                      sf_col + 4, (kb > 0 || k4 > 0) ? 1u : 0u);
                            mma_commit(&empty[s]);
                            ++it;
                        }
                        if (!ok) break;
                        mma_commit(&sempty[slot]);
                        mma_commit(&sftfree[st]);
                    }
                    if (!ok) break;
                    mma_commit(&tfull[as]);
                }
                mma_commit(done_bar);
                mbar_wait_drain(done_bar, 0, p.wait_limit_ns);
            }
            __syncwarp();
        } else {
            // scale loaders: warps 2 and 3 take alternate runs of K groups. A run
            // is four groups when the exponents are packed (two when B has a
            // word per row), else one group (four loads per word); all loads of
            // a run are issued before any is stored, so a run costs one memory
            // round trip. Line r of a 128-row chunk holds the words of rows
            // r, 32+r, 64+r, 96+r.
            constexpr int R = PER_ROW_B ? 2 : 4;
            constexpr int NB = PER_ROW_B ? 4 * C::kSfbChunks : 1;
            const uint32_t mine = static_cast<uint32_t>(warp - 2);
            const int run_len = (p.fmt == 2) ? R : 1;
            uint32_t g = 0, run = 0;
            bool ok = true;
            const int64_t nblocks_b = (p.n + 127) / 128;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int mb, nb;
                tile_coords(t, p, mb, nb);
                const int e = tile_expert(p, mb, false);
                if (e < 0) continue;
                const int64_t m0 = static_cast<int64_t>(mb) * BM, n0 = static_cast<int64_t>(nb) * BN;
                const int64_t sb_off = e * p.sbg;
                for (int kg0 = 0; kg0 < num_groups; kg0 += run_len, ++run) {
                    const int cnt = num_groups - kg0 < run_len ? num_groups - kg0 : run_len;
                    if ((run & 1u) != mine) { g += cnt; continue; }
                    uint32_t wa[R][4], wb[R][NB];
                    int64_t offa[4], offb[NB];
                    bool vala[4], valb[NB];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t row = m0 + 32 * q + lane;
                        vala[q] = row < p.m;
                        offa[q] = row * p.sam;
                    }
#pragma unroll
                    for (int i = 0; i < NB; ++i) {
                        if constexpr (PER_ROW_B) {
                            const int64_t row = n0 + 32 * i + lane;        // chunk i/4, quarter i%4
                            valb[i] = row < p.n;
                            offb[i] = sb_off + row * p.sbn;
                        } else {
                            const int64_t r = n0 / 128 + lane;             // one block word per chunk
                            valb[i] = lane < C::kSfbChunks && r < nblocks_b;
                            offb[i] = sb_off + r * p.sbn;
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
                            if constexpr (PER_ROW_B) {
                                v = make_uint4(wb[j][4 * c], wb[j][4 * c + 1], wb[j][4 * c + 2], wb[j][4 * c + 3]);
                            } else {
                                const uint32_t wbc = __shfl_sync(0xffffffffu, wb[j][0], c);
                                v = make_uint4(wbc, wbc, wbc, wbc);
                            }
                            *reinterpret_cast<uint4*>(dst + BM + 128 * c + lane * 4) = v;
                        }
                        fence_proxy_async_smem();   // visible to tcgen05.cp (async proxy)
                        mbar_arrive(&sfull[slot]);
                    }
                    if (!ok) break;
                    g += cnt;
                }
            }
        }
    } else {
        regs_alloc<184>();
        // ---------------- epilogue warpgroups ----------------
        constexpr int CPT = C::kColsPerThread;
        constexpr int U = CPT < 32 ? CPT : 32;
        const int wg = (warp - 4) >> 2;
        const int q = warp & 3;
        const int r_local = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const bool vec_store = p.vec_store != 0;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const int e = tile_expert(p, mb, threadIdx.x == kThreads - kMathThreads);
            if (e < 0) continue;
            const int64_t row = static_cast<int64_t>(mb) * BM + r_local;
            const bool store_row = row < p.m && (wg != 0 ? row_in_expert_quiet(p, row, e) : row_in_expert(p, row, e));
            const uint32_t as = tc % C::kAccStages, aph = (tc / C::kAccStages) & 1u;
            ++tc;
            if (!warp_wait(&tfull[as], aph, ctl)) break;
            tc_fence_after_sync();
            uint32_t accb[CPT];
            const uint32_t tcol = tmem_base + lane_base + as * BN + wg * CPT;
#pragma unroll
            for (int c0 = 0; c0 < CPT; c0 += U) {
                if constexpr (U == 16) tmem_ld_32x32b_x16(tcol + c0, *reinterpret_cast<uint32_t(*)[16]>(&accb[c0]));
                else tmem_ld_32x32b_x32(tcol + c0, *reinterpret_cast<uint32_t(*)[32]>(&accb[c0]));
            }
            tmem_wait_ld(accb);            // one wait for all loads
            float* acc = reinterpret_cast<float*>(accb);
            tc_fence_before_sync();
            mbar_arrive(&tempty[as]);
            const int64_t col0 = static_cast<int64_t>(nb) * BN + wg * CPT;
            if constexpr (C::kStageOut) {
                if (p.tma_d && __all_sync(0xffffffffu, store_row)) {
                    // all 32 rows of this warp are written: through its staging buffer
                    uint8_t* stg = smem + C::kOffStage + (warp - 4) * C::kOutWarpBytes;
                    const int32_t y = static_cast<int32_t>(static_cast<int64_t>(mb) * BM + q * 32);
                    tma_store_warp_rows<CPT, 64, OUT_F32>(acc, stg, &tmap_d, col0, y, p.accumulate != 0);
                    continue;
                }
            }
            if (store_row) {
                if constexpr (OUT_FP8) {
                    static_assert(CPT == 128, "E4M3 output needs 128 columns per thread");
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
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int BN, bool PER_ROW_B, bool OUT_F32, bool OUT_FP8 = false>
cudaError_t launch_mx_t(const GemmLaunch& L, GemmParams p, cudaStream_t st, int num_sms) {
    using Cf = MxCfg<BN, OUT_FP8 ? 0 : (OUT_F32 ? 4 : 2)>;
    CUtensorMap ta, tb;
    if (!(L.a_mn ? encode_kmajor_map(&ta, L.a, L.k, L.m, L.lda, BK) : encode_kmajor_map(&ta, L.a, L.m, L.k, L.lda, BM)))
        return cudaErrorInvalidValue;
    if (!(L.b_mn ? encode_kmajor_map(&tb, L.b, L.k, L.n, L.ldb, BK)
                 : encode_kmajor_map(&tb, L.b, L.n * (L.m_indices ? L.num_groups : 1), L.k, L.ldb, BN)))
        return cudaErrorInvalidValue;
    // bf16 / fp32 output through TMA tile stores when D's rows start and end 16-byte aligned
    CUtensorMap td = {};
    p.tma_d = 0;
    if constexpr (Cf::kStageOut) {
        constexpr int es = OUT_F32 ? 4 : 2;
        // a TMA store may write a row's last 16-byte chunk whole, so D's rows must end on one
        if ((reinterpret_cast<uintptr_t>(L.d) & 15u) == 0 && L.ldd > 0 && (L.ldd * es) % 16 == 0 &&
            (L.n * es) % 16 == 0 &&
            encode_2d_map(&td, L.d, OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, L.m,
                          L.n, L.ldd * es, 32, Cf::kCW, /*swizzle=*/64))
            p.tma_d = 1;
    }
    p.tiles_m = static_cast<int>((L.m + BM - 1) / BM);
    p.tiles_n = static_cast<int>((L.n + BN - 1) / BN);
    const int tiles = p.tiles_m * p.tiles_n;
    const int grid = tiles < num_sms ? tiles : num_sms;
    auto kern = gemm_mx_kernel<BN, PER_ROW_B, OUT_F32, OUT_FP8>;
    if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), Cf::kSmemBytes); e != cudaSuccess) return e;
    return launch_gemm_kernel(kern, static_cast<unsigned>(grid), 1, Cf::kSmemBytes, st, ta, tb, td, p);
}

template <bool PER_ROW_B, bool OUT_F32>
cudaError_t dispatch_mx(int bn, const GemmLaunch& L, const GemmParams& p, cudaStream_t st, int num_sms) {
    switch (bn) {
        case 256: return launch_mx_t<256, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
        case 128: return launch_mx_t<128, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
        case 64: return launch_mx_t<64, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
        default: return launch_mx_t<32, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
    }
}

}  // namespace

cudaError_t launch_gemm_mx(const GemmLaunch& L, const GemmParams& p, int bn, cudaStream_t st, int num_sms) {
    if (L.out_fp8) return launch_mx_t<256, false, false, true>(L, p, st, num_sms);
    if (L.out_f32) return dispatch_mx<true, true>(bn, L, p, st, num_sms);
    return dispatch_mx<false, false>(bn, L, p, st, num_sms);
}

}  // namespace ql
