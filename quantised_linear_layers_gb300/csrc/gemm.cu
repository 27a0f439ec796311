// Block-scaled FP8 GEMM for sm_103a: D = A * B^T.
//
// "DeepGEMM Essentials: High-Performance FP8 Matrix Multiplication" Parts 1, 6
// (gemm_fp8_fp8_bf16_nt) and 12-13 (wgrad_gemm_fp8_fp8_fp32_nt); scale
// semantics of "[Help] Starter script for nn.Linear for fwd,bwd" (maintainer's
// reply: one row (1, ceil(k/128)) of the RHS scale grid per 128-row block of B,
// used for all K blocks):
//
//   D[i,j] = sum_kb sa[i,kb] * sb(j,kb) * P_kb[i,j],  P_kb = sum_{k in kb} A[i,k] B[j,k]
//
// Design (one persistent CTA per SM, 12 warps):
//   warp 0      TMA producer: A tile [128 x 128 B] and B tile [BN x 128 B] per
//               128-wide K block into a STAGES-deep shared-memory ring
//               (128-byte swizzle).
//   warp 1      owns tensor memory; one elected lane issues four
//               tcgen05.mma.kind::f8f6f4 (K = 32 each) per K block into a fresh
//               TMEM accumulator stage, then commits to free the smem stage and
//               to publish the stage to the math warps.
//   warps 2-3   scale loaders: sa[128 rows] and sb (one value per 128-column
//               block, or one per column for wgrad) of each K block into a
//               shared-memory scale ring (any scale strides; packed UE8M0 is
//               decoded here), several K blocks per memory round trip.
//   warps 4-11  two math warpgroups: each thread owns one accumulator row and
//               BN/2 columns in registers; per K block it reads P_kb from TMEM
//               (tcgen05.ld) and promotes acc += (sa*sb) * P_kb with fp32
//               FMAs (packed f32x2 when every column has its own scale); after the last K block it writes bf16 (or fp32,
//               optionally accumulated) output.
// Tiles are 128 x BN (BN in {256,128,64,32}), visited in grouped raster order
// (GROUP_M m-blocks share each n-block sweep) for L2 reuse. Every wait is
// bounded in time; on a time-out the CTA raises the device status word,
// drains its own copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "bounds.cuh"
#include "common.cuh"
#include "epilogue_fp8.cuh"
#include "epilogue_tma.cuh"
#include "gemm.cuh"
#include "promote.cuh"

namespace ql {
// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

// cuTensorMapEncodeTiled from the driver, looked up once (thread-safe static).
static EncodeTiledFn get_encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return nullptr;
    }();
    return fn;
}

cudaError_t ensure_smem_attr(const void* kern, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kern, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({kern, dev});
    return e;
}

int max_active_clusters(const void* kern, const cudaLaunchConfig_t& cfg) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({kern, dev});
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = 1;
    cache[{kern, dev}] = n;
    return n;
}

bool encode_2d_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int64_t rows, int64_t cols,
                   int64_t row_stride_bytes, int box_rows, int box_cols, int swizzle) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                    : (swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};   // 128 bytes of K per row
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


namespace {

constexpr int kThreads = 384;
constexpr int kMathThreads = 256;
constexpr int BM = 128;
constexpr int BK = 128;         // K block = scale granularity
// Scale slots: with one B scale per 128 columns, a slot holds one loader run
// of 4 K blocks and the math warps wait on it and release it once per run, one
// arrive per warp; with a B scale per column (wgrad) a slot holds one K block
// and every math thread releases it.

// OUT_BYTES: element size of a D that leaves through shared memory and TMA
// tile stores (2: bf16, 4: fp32; 0: stored directly), one 2 KB buffer of 32
// rows x 64 bytes (64-byte swizzle) per epilogue warp.
template <int BN, bool PER_ROW_B, int OUT_BYTES = 0>
struct Cfg {
    static constexpr int kStageA = BM * BK;                  // bytes
    static constexpr int kStageB = BN * BK;
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr int kStages = (BN == 256) ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int kTmemStages = (512 / BN) < 4 ? (512 / BN) : 4;
    static constexpr int kTmemColsUsed = kTmemStages * BN;
    static constexpr int kTmemCols = kTmemColsUsed <= 32 ? 32 : (kTmemColsUsed <= 64 ? 64 : (kTmemColsUsed <= 128 ? 128 : (kTmemColsUsed <= 256 ? 256 : 512)));
    static constexpr int kSbPerSlot = PER_ROW_B ? BN : 4;
    static constexpr int kSlotFloats = BM + kSbPerSlot;      // one K block's scales
    static constexpr int kRun = PER_ROW_B ? 2 : 4;           // K blocks per loader run
    static constexpr int kSlotKb = PER_ROW_B ? 1 : kRun;     // K blocks per slot
    static constexpr int kScaleSlots = PER_ROW_B ? 8 : 4;
    static constexpr int kRunFloats = kSlotKb * kSlotFloats;
    static constexpr uint32_t kRelease = PER_ROW_B ? kMathThreads : kMathThreads / 32;   // arrives per release
    static constexpr int kColsPerThread = BN / 2;
    // shared memory layout (offsets from a 1024-aligned base)
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kStageA;
    static constexpr int kOffScale = kOffB + kStages * kStageB;
    static constexpr int kOffBar = kOffScale + kScaleSlots * kRunFloats * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kTmemStages + 2 * kScaleSlots + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr bool kStageOut = OUT_BYTES != 0 && (BN / 2) % (64 / (OUT_BYTES == 0 ? 1 : OUT_BYTES)) == 0;
    static constexpr int kOutWarpBytes = 32 * 64;
    static constexpr int kOffStage = kStageOut ? ((kOffMisc + 16 + 1023) / 1024) * 1024 : kOffMisc + 16;
    static constexpr int kSmemBytes = kOffStage + (kStageOut ? 8 * kOutWarpBytes : 0) + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kColsPerThread % 16 == 0, "columns per thread");
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

template <int BN, bool PER_ROW_B, bool OUT_F32, bool OUT_FP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const GemmParams p) {
    using C = Cfg<BN, PER_ROW_B, OUT_FP8 ? 0 : (OUT_F32 ? 4 : 2)>;
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
    uint64_t* sempty = sfull + C::kScaleSlots;
    uint64_t* done_bar = sempty + C::kScaleSlots;
    uint32_t* tmem_base_sm = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int s = 0; s < C::kTmemStages; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], C::kRelease); }
        for (int s = 0; s < C::kScaleSlots; ++s) { mbar_init(&sfull[s], 32); mbar_init(&sempty[s], C::kRelease); }
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

    if (warp < 4) {
        regs_dealloc<88>();   // 128 x 88 + 256 x 208 = 384 x 168 registers
        if (warp == 0) {
            // ---------------- TMA producer ----------------
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
                const uint32_t idesc = idesc_e4m3_f32(BM, BN) | idesc_mn_bits(p.a_mn, p.b_mn);
                const uint64_t astep = k32_step(p.a_mn), bstep = k32_step(p.b_mn);
                uint32_t it = 0, tc = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                    int mb, nb;
                    tile_coords(t, p, mb, nb);
                    if (tile_expert(p, mb, false) < 0) continue;
                    for (int kb = 0; kb < num_kb; ++kb, ++it, ++tc) {
                        const uint32_t ts = tc % C::kTmemStages, tph = (tc / C::kTmemStages) & 1u;
                        if (!mbar_wait(&tempty[ts], tph ^ 1u, ctl)) { ok = false; break; }
                        tc_fence_after_sync();
                        const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                        if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                        tc_fence_after_sync();
                        const uint64_t adesc = sw128_desc(smem_addr(sA + s * C::kStageA), p.a_mn);
                        const uint64_t bdesc = sw128_desc(smem_addr(sB + s * C::kStageB), p.b_mn);
                        const uint32_t d_tmem = tmem_base + ts * BN;
#pragma unroll
                        for (int k4 = 0; k4 < BK / 32; ++k4)
                            mma_e4m3(d_tmem, adesc + astep * k4, bdesc + bstep * k4, idesc, k4 > 0 ? 1u : 0u);
                        mma_commit(&empty[s]);
                        mma_commit(&tfull[ts]);
                    }
                }
                // all MMAs issued by this thread have completed before tensor memory is freed
                mma_commit(done_bar);
                mbar_wait_drain(done_bar, 0, p.wait_limit_ns);
            }
            __syncwarp();
        } else {
            // ---------------- scale loaders ----------------
            // Warps 2 and 3 take alternate runs of K blocks (four, or two when B
            // has a scale per row); all loads of a run are issued before any
            // is stored, so a run costs one memory round trip. A run fills one
            // slot (kSlotKb == kRun) or one slot per K block.
            constexpr int kRun = C::kRun;
            constexpr int kSbLoads = PER_ROW_B ? BN / 32 : 1;
            const uint32_t mine = static_cast<uint32_t>(warp - 2);
            uint32_t run = 0, g = 0;
            bool ok = true;
            const int64_t nblocks_b = (p.n + 127) / 128;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int mb, nb;
                tile_coords(t, p, mb, nb);
                const int e = tile_expert(p, mb, false);
                if (e < 0) continue;
                const int64_t m0 = static_cast<int64_t>(mb) * BM, n0 = static_cast<int64_t>(nb) * BN;
                const int64_t sb_off = e * p.sbg;
                for (int kb0 = 0; kb0 < num_kb; kb0 += kRun, ++run) {
                    const int cnt = num_kb - kb0 < kRun ? num_kb - kb0 : kRun;
                    if ((run & 1u) != mine) { g += cnt; continue; }
                    float va[kRun][4], vb[kRun][kSbLoads];
#pragma unroll
                    for (int j = 0; j < kRun; ++j) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int64_t row = m0 + lane + 32 * i;
                            va[j][i] = (j < cnt && row < p.m) ? decode_scale(p.sfa, p.fmt, row * p.sam, kb0 + j, p.sak, p.bnd, 0) : 0.0f;
                        }
#pragma unroll
                        for (int i = 0; i < kSbLoads; ++i) {
                            float v = 0.0f;
                            if (j < cnt) {
                                if constexpr (PER_ROW_B) {
                                    const int64_t col = n0 + lane + 32 * i;
                                    if (col < p.n) v = decode_scale(p.sfb, p.fmt, sb_off + col * p.sbn, kb0 + j, p.sbk, p.bnd, 1);
                                } else {
                                    const int64_t r = n0 / 128 + lane;
                                    if (lane < (BN + 127) / 128 && r < nblocks_b)
                                        v = decode_scale(p.sfb, p.fmt, sb_off + r * p.sbn, kb0 + j, p.sbk, p.bnd, 1);
                                }
                            }
                            vb[j][i] = v;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < kRun; ++j) {
                        if (j >= cnt) break;
                        // slot of this K block: the run's (per-run slots) or its own
                        const uint32_t u = C::kSlotKb == 1 ? g + j : run;
                        const uint32_t slot = u % C::kScaleSlots, ph = (u / C::kScaleSlots) & 1u;
                        if ((C::kSlotKb == 1 || j == 0) && !warp_wait(&sempty[slot], ph ^ 1u, ctl)) { ok = false; break; }
                        float* dst = sScale + slot * C::kRunFloats + (C::kSlotKb == 1 ? 0 : j) * C::kSlotFloats;
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = va[j][i];
                        if constexpr (PER_ROW_B) {
#pragma unroll
                            for (int i = 0; i < kSbLoads; ++i) dst[BM + lane + 32 * i] = vb[j][i];
                        } else {
                            if (lane < (BN + 127) / 128) dst[BM + lane] = vb[j][0];
                        }
                        if (C::kSlotKb == 1 || j == cnt - 1) mbar_arrive(&sfull[slot]);
                    }
                    if (!ok) break;
                    g += cnt;
                }
            }
        }
    } else {
        regs_alloc<208>();
        // ---------------- math warpgroups: promotion + epilogue ----------------
        constexpr int CPT = C::kColsPerThread;
        const int wg = (warp - 4) >> 2;          // column half
        const int q = warp & 3;                  // TMEM lane quarter
        const int r_local = q * 32 + lane;       // accumulator row in the tile
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const bool vec_store = p.vec_store != 0;
        float acc[CPT];
        uint32_t g = 0, run = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const int e = tile_expert(p, mb, threadIdx.x == kThreads - kMathThreads);
            if (e < 0) continue;
            const int64_t row = static_cast<int64_t>(mb) * BM + r_local;
            const bool store_row = row < p.m && (wg != 0 ? row_in_expert_quiet(p, row, e) : row_in_expert(p, row, e));
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
            for (int kb = 0; kb < num_kb; ++kb, ++g) {
                // the slot of this K block: its loader run's, or its own
                const int jr = C::kSlotKb == 1 ? 0 : kb % C::kSlotKb;
                const uint32_t u = C::kSlotKb == 1 ? g : run;
                const uint32_t slot = u % C::kScaleSlots, sph = (u / C::kScaleSlots) & 1u;
                const bool slot_end = C::kSlotKb == 1 || jr == C::kSlotKb - 1 || kb == num_kb - 1;
                const uint32_t ts = g % C::kTmemStages, tph = (g / C::kTmemStages) & 1u;
                if (jr == 0 && !warp_wait(&sfull[slot], sph, ctl)) { ok = false; break; }
                const float* src = sScale + slot * C::kRunFloats + jr * C::kSlotFloats;
                const float sa = src[r_local];
                if (!warp_wait(&tfull[ts], tph, ctl)) { ok = false; break; }
                tc_fence_after_sync();
                const uint32_t tcol = tmem_base + lane_base + ts * BN + wg * CPT;
                constexpr int U = CPT < 64 ? CPT : 64;     // columns per TMEM read round
                // one scale per 128 columns: one fp32 FMA per element (single
                // rounding); the packed f32x2 form retires the same 32 FMAs
                // per clock per SMSP and needs the accumulators paired and
                // unpaired around it (measured: 8192 x 8192 x 7168 439 -> 421 us)
                if constexpr (!PER_ROW_B) {
                    const float sab = sa * src[BM + ((BN == 256) ? wg : 0)];
#pragma unroll
                    for (int c0 = 0; c0 < CPT; c0 += U) {
                        uint32_t v[U];
                        tmem_load_cols<U>(tcol + c0, v);
                        if (c0 + U == CPT) {              // last read of this stage
                            tc_fence_before_sync();
                            __syncwarp();
                            mbar_arrive_lane0(&tempty[ts], lane);
                        }
#pragma unroll
                        for (int j = 0; j < U; ++j) acc[c0 + j] = fmaf(__uint_as_float(v[j]), sab, acc[c0 + j]);
                    }
                    if (slot_end) {
                        __syncwarp();
                        mbar_arrive_lane0(&sempty[slot], lane);
                        ++run;
                    }
                } else {
                    // a scale per column: (sa * sb) and the FMA, two elements
                    // per packed f32x2 instruction (half the instructions of
                    // the scalar form)
                    const uint64_t sa2 = pack2(sa, sa);
#pragma unroll
                    for (int c0 = 0; c0 < CPT; c0 += U) {
                        uint32_t v[U];
                        tmem_load_cols<U>(tcol + c0, v);
                        if (c0 + U == CPT) {
                            tc_fence_before_sync();
                            mbar_arrive(&tempty[ts]);
                        }
                        const float* sbp = src + BM + wg * CPT + c0;
#pragma unroll
                        for (int j = 0; j < U; j += 2) {
                            const uint64_t s2 = mul2(sa2, pack2(sbp[j], sbp[j + 1]));
                            uint64_t a2 = pack2(acc[c0 + j], acc[c0 + j + 1]);
                            fma2(a2, pack2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2);
                            acc[c0 + j] = __uint_as_float(static_cast<uint32_t>(a2));
                            acc[c0 + j + 1] = __uint_as_float(static_cast<uint32_t>(a2 >> 32));
                        }
                    }
                    mbar_arrive(&sempty[slot]);
                }
            }
            if (!ok) break;
            // ---------------- epilogue ----------------
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
cudaError_t launch_t(const GemmLaunch& L, GemmParams p, cudaStream_t st, int num_sms) {
    using Cf = Cfg<BN, PER_ROW_B, OUT_FP8 ? 0 : (OUT_F32 ? 4 : 2)>;
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
                          L.n, L.ldd * es, 32, 64 / es, /*swizzle=*/64))
            p.tma_d = 1;
    }
    p.tiles_m = static_cast<int>((L.m + BM - 1) / BM);
    p.tiles_n = static_cast<int>((L.n + BN - 1) / BN);
    const int tiles = p.tiles_m * p.tiles_n;
    int grid = tiles < num_sms ? tiles : num_sms;
    auto kern = gemm_fp8_kernel<BN, PER_ROW_B, OUT_F32, OUT_FP8>;
    if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), Cf::kSmemBytes); e != cudaSuccess) return e;
    return launch_gemm_kernel(kern, static_cast<unsigned>(grid), 1, Cf::kSmemBytes, st, ta, tb, td, p);
}

template <bool PER_ROW_B, bool OUT_F32>
cudaError_t dispatch_bn(int bn, const GemmLaunch& L, const GemmParams& p, cudaStream_t st, int num_sms) {
    switch (bn) {
        case 256: return launch_t<256, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
        case 128: return launch_t<128, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
        case 64: return launch_t<64, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
        default: return launch_t<32, PER_ROW_B, OUT_F32>(L, p, st, num_sms);
    }
}

}  // namespace

int choose_block_n(int64_t m, int64_t n, int num_sms) {
    const int64_t tm = (m + BM - 1) / BM;
    const int cands[4] = {256, 128, 64, 32};
    for (int i = 0; i < 4; ++i) {
        const int64_t tiles = tm * ((n + cands[i] - 1) / cands[i]);
        if (tiles >= num_sms) return cands[i];
    }
    return 32;
}

cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t st, int num_sms) {
    GemmParams p{};
    p.m = L.m;
    p.n = L.n;
    p.num_kb = static_cast<int>((L.k + BK - 1) / BK);
    p.sfa = L.sfa;
    p.sam = L.sam;
    p.sak = L.sak;
    p.sfb = L.sfb;
    p.sbn = L.sbn;
    p.sbk = L.sbk;
    p.fmt = L.fmt;
    p.d = L.d;
    p.ldd = L.ldd;
    p.accumulate = L.accumulate;
    p.group_m = 16;
    p.dev_status = L.dev_status;
    p.wait_limit_ns = L.wait_limit_ns;
    p.stall_producer = L.stall_producer;
    p.m_indices = L.m_indices;
    p.num_groups = L.m_indices ? L.num_groups : 1;
    p.b_group_rows = L.n;
    p.sbg = L.sbg;
    p.dsf = L.dsf;
    p.dsm = L.dsm;
    p.dsg = L.dsg;
    p.dgran = L.dgran;
    p.dfmt = L.dfmt;
    p.drecip = L.drecip;
    p.a_mn = L.a_mn ? 1 : 0;
    p.b_mn = L.b_mn ? 1 : 0;
    const int64_t es = L.out_fp8 ? 1 : (L.out_f32 ? 4 : 2);
    p.vec_store = ((reinterpret_cast<uintptr_t>(L.d) & 15u) == 0 && (L.ldd * es) % 16 == 0) ? 1 : 0;
    {
        // byte ranges of the buffers read or written with plain loads and stores
        const int64_t kscales = L.fmt == 2 ? (p.num_kb + 3) / 4 : p.num_kb;
        const int64_t brows = L.per_row_b ? L.n : (L.n + 127) / 128;
        const int64_t dg = L.dgran > 0 ? (L.n + L.dgran - 1) / L.dgran : 0;
        p.bnd.s[0] = span_of(L.sfa, 4, L.m, L.sam, kscales, L.sak);
        p.bnd.s[1] = span_of(L.sfb, 4, brows, L.sbn, kscales, L.sbk, L.m_indices ? L.num_groups : 1, L.sbg);
        p.bnd.s[2] = span_of(L.d, es, L.m, L.ldd, L.n, 1);
        p.bnd.s[3] = L.out_fp8 ? span_of(L.dsf, 4, L.m, L.dsm, L.dfmt == 2 ? (dg + 3) / 4 : dg, L.dsg) : Span{0, 0};
        p.bnd.s[4] = span_of(L.m_indices, 4, L.m, 1);
        p.bnd.status = L.dev_status;
    }
    const int bn = L.block_n > 0 ? L.block_n : choose_block_n(L.m, L.n, num_sms);
    // UE8M0 scales (fp32 powers of two or packed exponents): promotion by the
    // tensor core's block-scaled MMA unless the CUDA-core path is requested.
    const bool ue8m0 = L.fmt == 1 || L.fmt == 2;
    const bool grouped = L.m_indices != nullptr;   // the pair kernel's two M halves share one B
    // CUDA-core promotion (fp32 scales, or forced): on one SM per tile; path 5
    // runs it on CTA pairs (256 x 256 tiles), which measured no faster (its two
    // accumulator stages leave the promotion hand-off exposed), 6 forces the
    // single-SM kernel, 7 the split-K cluster form below.
    const bool promote = !ue8m0 || L.path == 1 || L.path == 5 || L.path == 6 || L.path == 7;
    if (promote && !grouped && !L.out_fp8 && L.path == 5) return launch_gemm_pair(L, p, st, num_sms);
    if (L.a_mn || L.b_mn) {
        // MN-major operands: one 128-byte swizzle atom of M / N per CTA, so
        // 128-column tiles on one SM, or the CTA pair (128 columns per CTA)
        if (!promote) {
            const int64_t pair_tiles = ((L.m + 255) / 256) * ((L.n + 255) / 256);
            if (L.path == 3 || (L.path == 0 && pair_tiles >= num_sms / 2)) return launch_gemm_mx2(L, p, st, num_sms);
            return launch_gemm_mx(L, p, 128, st, num_sms);
        }
        if (L.out_f32) return launch_t<128, true, true>(L, p, st, num_sms);
        return launch_t<128, false, false>(L, p, st, num_sms);
    }
    if (L.out_fp8) {
        // E4M3 output: 256-wide tiles, so every epilogue thread owns whole
        // 128-column groups of its row (pair, single-SM or promotion kernel)
        if (!promote) {
            const int64_t pair_tiles = ((L.m + 255) / 256) * ((L.n + 255) / 256);
            if (L.path == 3 || (L.path == 0 && pair_tiles >= num_sms / 2)) return launch_gemm_mx2(L, p, st, num_sms);
            return launch_gemm_mx(L, p, 256, st, num_sms);
        }
        return launch_t<256, false, false, true>(L, p, st, num_sms);
    }
    // CUDA-core promotion with too few 128 x 128 tiles to occupy the SMs (small
    // M) and a long K loop (16 K blocks or more): split-K over a cluster (path 7
    // forces it wherever a split applies). With fewer K blocks the cluster's
    // launch and exchange cost more than the split saves (128 x 256 x 512: 10.9
    // us on one SM per tile, 12.3 us split in two).
    if (promote && !grouped && !L.out_f32 && (L.path == 7 || (L.path == 0 && L.block_n == 0 && p.num_kb >= 16))) {
        const int split_p = choose_split_k(L.m, L.n, L.k, num_sms);
        if (split_p >= 2) return launch_gemm_prom_sk(L, p, split_p, st);
    }
    if (ue8m0 && L.path == 3 && !grouped) return launch_gemm_mx2(L, p, st, num_sms);
    const int split = (ue8m0 && !grouped && !L.out_f32) ? choose_split_k(L.m, L.n, L.k, num_sms) : 1;
    if (L.path == 4 && split >= 2) return launch_gemm_mx_sk(L, p, split, st);
    if (ue8m0 && L.path == 0 && !grouped && L.block_n == 0) {
        // CTA pairs (256 x 224 tiles for bf16 output, 256 x 256 for fp32)
        // when there is a tile for every pair of SMs; split-K over a cluster
        // when the 128 x 128 tiles are too few to occupy the SMs; CTA pairs
        // again down to a tile for every other pair (mid-size M: their larger
        // tiles read A and B fewer times than single-SM tiles narrow enough to
        // fill the SMs); else single-SM tiles.
        const int64_t bnp = L.out_f32 ? 256 : 224;
        const int64_t pair_tiles = ((L.m + 255) / 256) * ((L.n + bnp - 1) / bnp);
        if (pair_tiles >= num_sms / 2) return launch_gemm_mx2(L, p, st, num_sms);
        if (split >= 2) return launch_gemm_mx_sk(L, p, split, st);
        if (pair_tiles >= num_sms / 4) return launch_gemm_mx2(L, p, st, num_sms);
    }
    if (!promote) return launch_gemm_mx(L, p, bn, st, num_sms);
    if (L.out_f32) return dispatch_bn<true, true>(bn, L, p, st, num_sms);
    return dispatch_bn<false, false>(bn, L, p, st, num_sms);
}

}  // namespace ql
