// FP8 casts for sm_103a.
//
// Per-token cast ("DeepGEMM Essentials: High-Performance FP8 Matrix
// Multiplication" Part 3, options of "deep-gemm: fused per-token FP8 cast in
// Triton (fused_per_token_cast_to_fp8), version 3") and 128x128 block cast
// (Part 4). Each kernel reads its input once from HBM and writes E4M3 data and
// scales straight into the caller's (possibly strided) views.
//
// Arithmetic per group (bit-exact; quant.cuh): amax = max(|x|) in fp32
// (exact), then the scale, factor and E4M3 rounding of quant.cuh.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "bounds.cuh"
#include "cast.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "quant.cuh"

namespace ql {
namespace {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Two fp32 products at once (mul.rn.f32x2: each lane rounded to nearest even,
// subnormals kept, exactly as the scalar multiply).
__device__ __forceinline__ float2 mul_rn2(float2 a, float2 b) {
    const uint64_t a2 = static_cast<uint64_t>(__float_as_uint(a.x)) | (static_cast<uint64_t>(__float_as_uint(a.y)) << 32);
    const uint64_t b2 = static_cast<uint64_t>(__float_as_uint(b.x)) | (static_cast<uint64_t>(__float_as_uint(b.y)) << 32);
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a2), "l"(b2));
    return make_float2(__uint_as_float(static_cast<uint32_t>(r)), __uint_as_float(static_cast<uint32_t>(r >> 32)));
}

// quant4 (quant.cuh) with the four products taken two at a time.
__device__ __forceinline__ uint32_t quant4_pk(float a, float b, float c, float d, float f) {
    const float2 f2 = make_float2(f, f);
    const float2 p = mul_rn2(make_float2(a, b), f2), q = mul_rn2(make_float2(c, d), f2);
    return e4m3x2(p.x, p.y) | (e4m3x2(q.x, q.y) << 16);
}

// ---------------------------------------------------------------------------
// Row-contiguous per-token cast (x_stride_n == 1, out_stride_n == 1).
// One warp task = (row, chunk of 32*E elements); each lane owns E consecutive
// elements, E = 64 bytes of input (32 bf16 or 16 fp32: four 16-byte loads, all
// issued before use), so a group of G elements is G/E consecutive lanes and its
// amax is a shuffle reduction over them (none for bf16 with G = 32).
// ---------------------------------------------------------------------------
template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(256, 4) cast_rows_kernel(const T* __restrict__ x, int64_t m, int64_t n, int64_t ldx,
                                                        uint8_t* __restrict__ out, int64_t ldo,
                                                        void* __restrict__ sf, int64_t ssm, int64_t ssg,
                                                        int64_t chunks_per_row, int vec_in, int vec_out,
                                                        const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    constexpr int kElemsPerLane = 64 / sizeof(T);          // 32 (bf16) or 16 (fp32)
    constexpr int kChunk = 32 * kElemsPerLane;
    constexpr int kLanesPerGroup = GRAN / kElemsPerLane;   // 1, 2, 4 or 8
    constexpr int kVec = 16 / sizeof(T);                   // elements per 16-byte load
    constexpr int kLoads = kElemsPerLane / kVec;           // 4
    static_assert(kLanesPerGroup >= 1, "a lane's elements lie in one group");

    const int lane = threadIdx.x & 31;
    const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t total = m * chunks_per_row;
    const int64_t G = (n + GRAN - 1) / GRAN;

    for (int64_t task = warp_global; task < total; task += nwarps) {
        const int64_t row = task / chunks_per_row;
        const int64_t chunk = task - row * chunks_per_row;
        const int64_t e0 = chunk * kChunk + static_cast<int64_t>(lane) * kElemsPerLane;
        const T* xr = x + row * ldx;

        uint4 raw[kLoads];
#pragma unroll
        for (int l = 0; l < kLoads; ++l) {
            const int64_t e = e0 + l * kVec;
            if (vec_in && e + kVec <= n) {
                raw[l] = QL_IN(bnd, 0, xr + e, 16) ? __ldg(reinterpret_cast<const uint4*>(xr + e)) : make_uint4(0, 0, 0, 0);
            } else {
                union { uint4 u; T t[kVec]; } tmp;
#pragma unroll
                for (int i = 0; i < kVec; ++i)
                    tmp.t[i] = (e + i < n && QL_IN(bnd, 0, xr + e + i, sizeof(T))) ? xr[e + i] : T(0.0f);
                raw[l] = tmp.u;
            }
        }
        // |x| max (exact in the input type): packed bf16x2 or scalar fp32
        float amax = 0.0f;
        if constexpr (sizeof(T) == 2) {
            __nv_bfloat162 m2 = __float2bfloat162_rn(0.0f);
#pragma unroll
            for (int l = 0; l < kLoads; ++l) {
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[l]);
#pragma unroll
                for (int i = 0; i < 4; ++i) m2 = __hmax2(m2, __habs2(h[i]));
            }
            amax = fmaxf(__bfloat162float(m2.x), __bfloat162float(m2.y));
        } else {
#pragma unroll
            for (int l = 0; l < kLoads; ++l) {
                const float* t = reinterpret_cast<const float*>(&raw[l]);
#pragma unroll
                for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(t[i]));
            }
        }
#pragma unroll
        for (int off = 1; off < kLanesPerGroup; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

        float s, f;
        uint32_t ebyte;
        if constexpr (FMT == kSfFp32 && !RECIP && kLanesPerGroup >= 2) {
            // group_scale's two correctly rounded divisions, one per lane of
            // a pair inside the group (a / 448 on the even lane, 448 / a on
            // the odd one), exchanged by shuffle: same operations, one divide
            // per lane instead of two
            const float a = fmaxf(amax, 1e-4f);
            const bool odd = (lane & 1) != 0;
            const float qd = __fdiv_rn(odd ? 448.0f : a, odd ? a : 448.0f);
            s = __shfl_sync(0xffffffffu, qd, lane & ~1);
            f = __shfl_sync(0xffffffffu, qd, lane | 1);
            ebyte = 0;
        } else {
            group_scale<FMT, RECIP>(amax, s, f, ebyte);
        }

        if (e0 < n) {
            uint8_t* orow = out + row * ldo;
            uint32_t w[kElemsPerLane / 4];
#pragma unroll
            for (int q = 0; q < kElemsPerLane / 4; ++q) {
                const T* t = reinterpret_cast<const T*>(&raw[0]) + 4 * q;
                w[q] = quant4(to_f32(t[0]), to_f32(t[1]), to_f32(t[2]), to_f32(t[3]), f);
            }
            if (vec_out && e0 + kElemsPerLane <= n) {
#pragma unroll
                for (int q = 0; q < kElemsPerLane / 16; ++q)
                    if (QL_IN(bnd, 1, orow + e0 + 16 * q, 16))
                        *reinterpret_cast<uint4*>(orow + e0 + 16 * q) =
                            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < kElemsPerLane; ++i)
                    if (e0 + i < n && QL_IN(bnd, 1, orow + e0 + i, 1))
                        orow[e0 + i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
            }
        }

        const int64_t g = e0 / GRAN;
        if constexpr (FMT != kSfPacked) {
            float* sp = static_cast<float*>(sf) + row * ssm + g * ssg;
            if ((lane % kLanesPerGroup) == 0 && g < G && QL_IN(bnd, 2, sp, 4)) *sp = s;
        } else {
            // four consecutive groups per int32 word; groups past the last are 0
            constexpr int kWordLanes = 4 * kLanesPerGroup;  // 4 .. 32
            const uint32_t mine = (g < G) ? ebyte : 0u;
            const int base = (lane / kWordLanes) * kWordLanes;
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word |= __shfl_sync(0xffffffffu, mine, base + j * kLanesPerGroup) << (8 * j);
            int32_t* wp = static_cast<int32_t*>(sf) + row * ssm + (g / 4) * ssg;
            if ((lane % kWordLanes) == 0 && g < G && QL_IN(bnd, 2, wp, 4)) *wp = static_cast<int32_t>(word);
        }
    }
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Transposed per-token cast (x_stride_m == 1): logical row i is a column of the
// physical array P[j][i] = x[i + j*ldx], and its groups run along j.
// A warp owns 4V consecutive i (V = elements per 16-byte load) and walks kSub
// subtiles of 128 consecutive j. In a subtile, lane (jr = lane/4, ic = lane%4)
// loads rows j + 16*jr + l, l < 16, at columns i0 .. i0+V: 16 independent
// 16-byte loads per lane. For each of its V logical rows a lane then holds 16
// consecutive j, so a group's amax is a shuffle over the lanes of the same ic
// (three steps for 128-wide groups, one for 32), and the lane writes its 16
// output bytes with one 16-byte store (eight lanes fill 128 contiguous bytes of
// an output row). The 8 warps of a CTA sit side by side along i, so the CTA
// reads 8 x 64 contiguous bytes of every physical row it touches. Packed
// 128-wide groups take kSub = 4 subtiles per warp so that the warp itself owns
// whole int32 words.
// ---------------------------------------------------------------------------
template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(256, 1) cast_cols_kernel(const T* __restrict__ x, int64_t m, int64_t n, int64_t ldx,
                                                           uint8_t* __restrict__ out, int64_t ldo,
                                                           void* __restrict__ sf, int64_t ssm, int64_t ssg,
                                                           int vec_in, int vec_out, const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    constexpr int V = 16 / sizeof(T);          // 8 (bf16) or 4 (fp32)
    constexpr int WI = 4 * V;                  // logical rows per warp
    constexpr int WJ = 128;                    // group-axis extent of a subtile
    constexpr int kSub = (FMT == kSfPacked && GRAN == 128) ? 4 : 1;
    constexpr int kLaneSpan = GRAN / 16;       // lanes (along jr) per group: 2 or 8

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int jr = lane >> 2, ic = lane & 3;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * (8 * WI) + warp * WI + ic * V;   // lane's first column
    const int64_t jw = static_cast<int64_t>(blockIdx.y) * (kSub * WJ);                     // warp's first row
    const int64_t Gtot = (n + GRAN - 1) / GRAN;
    const bool full_cols = vec_in && i0 + V <= m;
    const bool leader = (jr % kLaneSpan) == 0;  // first lane of a group (per ic)

    uint32_t ebytes[V];                         // packed 128-groups: byte k of each word
#pragma unroll
    for (int c = 0; c < V; ++c) ebytes[c] = 0;

    for (int sub = 0; sub < kSub; ++sub) {
        const int64_t j0 = jw + sub * WJ + jr * 16;                          // lane's first row
        uint4 raw[16];
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            const int64_t j = j0 + l;
            if (j < n && full_cols) {
                const T* src = x + j * ldx + i0;
                raw[l] = QL_IN(bnd, 0, src, 16) ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
            } else {
                union { uint4 u; T t[V]; } tmp;
#pragma unroll
                for (int c = 0; c < V; ++c)
                    tmp.t[c] = (j < n && i0 + c < m && QL_IN(bnd, 0, x + j * ldx + i0 + c, sizeof(T)))
                                   ? x[j * ldx + i0 + c] : T(0.0f);
                raw[l] = tmp.u;
            }
        }
        float amax[V];
#pragma unroll
        for (int c = 0; c < V; ++c) amax[c] = 0.0f;
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            const T* t = reinterpret_cast<const T*>(&raw[l]);
#pragma unroll
            for (int c = 0; c < V; ++c) amax[c] = fmaxf(amax[c], fabsf(to_f32(t[c])));
        }
#pragma unroll
        for (int c = 0; c < V; ++c)
#pragma unroll
            for (int off = 4; off < 4 * kLaneSpan; off <<= 1)
                amax[c] = fmaxf(amax[c], __shfl_xor_sync(0xffffffffu, amax[c], off));

        const int64_t g = j0 / GRAN;             // this lane's group along j
#pragma unroll
        for (int c = 0; c < V; ++c) {
            float s, f;
            uint32_t ebyte;
            group_scale<FMT, RECIP>(amax[c], s, f, ebyte);
            const int64_t i = i0 + c;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const T* t0 = reinterpret_cast<const T*>(&raw[4 * q]);
                const T* t1 = reinterpret_cast<const T*>(&raw[4 * q + 1]);
                const T* t2 = reinterpret_cast<const T*>(&raw[4 * q + 2]);
                const T* t3 = reinterpret_cast<const T*>(&raw[4 * q + 3]);
                w[q] = quant4(to_f32(t0[c]), to_f32(t1[c]), to_f32(t2[c]), to_f32(t3[c]), f);
            }
            if (i < m && j0 < n) {
                uint8_t* orow = out + i * ldo;
                if (vec_out && j0 + 16 <= n) {
                    if (QL_IN(bnd, 1, orow + j0, 16))
                        *reinterpret_cast<uint4*>(orow + j0) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    for (int e = 0; e < 16; ++e)
                        if (j0 + e < n && QL_IN(bnd, 1, orow + j0 + e, 1))
                            orow[j0 + e] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
                }
            }
            if constexpr (FMT != kSfPacked) {
                float* sp = static_cast<float*>(sf) + i * ssm + g * ssg;
                if (leader && i < m && g < Gtot && QL_IN(bnd, 2, sp, 4)) *sp = s;
            } else if constexpr (GRAN == 32) {
                // the subtile's 128 rows are one word: groups of lanes jr = 0, 2, 4, 6
                const uint32_t mine = (g < Gtot) ? ebyte : 0u;
                uint32_t word = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) word |= __shfl_sync(0xffffffffu, mine, ic + 8 * k) << (8 * k);
                const int64_t g0 = (jw + sub * WJ) / GRAN;
                int32_t* wp = static_cast<int32_t*>(sf) + i * ssm + (g0 / 4) * ssg;
                if (jr == 0 && i < m && g0 < Gtot && QL_IN(bnd, 2, wp, 4)) *wp = static_cast<int32_t>(word);
            } else {
                ebytes[c] |= ((g < Gtot) ? ebyte : 0u) << (8 * sub);
            }
        }
    }
    if constexpr (FMT == kSfPacked && GRAN == 128) {
        const int64_t g0 = jw / GRAN;            // four groups: one word
#pragma unroll
        for (int c = 0; c < V; ++c) {
            const int64_t i = i0 + c;
            int32_t* wp = static_cast<int32_t*>(sf) + i * ssm + (g0 / 4) * ssg;
            if (jr == 0 && i < m && g0 < Gtot && QL_IN(bnd, 2, wp, 4)) *wp = static_cast<int32_t>(ebytes[c]);
        }
    }
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// TMA-staged transposed per-token cast (x_stride_m == 1, 16-byte-aligned
// rows). The physical array P[j][i] is read in boxes of 128 rows (j) x 128
// bytes (BI = 64 bf16 or 32 fp32 values of i) by one producer thread into a
// 4-stage shared-memory ring; two consumer warps each take 4V of the box's
// columns with the lane mapping of the register kernel below (lane jr, ic:
// rows 16*jr .. +16, columns V*ic .. +V), quantise, and store 16 bytes per
// logical row. A CTA walks a unit of four consecutive boxes along j of one
// column strip, so for packed 128-wide groups each lane owns whole words.
// Every wait is bounded; on a time-out the CTA records it and drains.
// ---------------------------------------------------------------------------
namespace cols_tma {
constexpr int kStages = 4;
constexpr int kRows = 128;                 // j per box
constexpr int kBoxBytes = kRows * 128;     // 16 KB
constexpr int kUnit = 4;                   // boxes per unit (512 rows)
constexpr int kThreads = 96;               // producer warp + 2 consumer warps
}  // namespace cols_tma

template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(96) cast_cols_tma_kernel(const __grid_constant__ CUtensorMap tmap, int64_t m,
                                                          int64_t n, uint8_t* __restrict__ out, int64_t ldo,
                                                          void* __restrict__ sf, int64_t ssm, int64_t ssg,
                                                          int vec_out, uint32_t* dev_status, uint64_t limit_ns,
                                                          const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    using namespace cols_tma;
    constexpr int V = 16 / sizeof(T);
    constexpr int BI = 128 / sizeof(T);        // columns per box
    constexpr int kLaneSpan = GRAN / 16;       // lanes (along jr) per group
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kStages * kBoxBytes);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t strips = (m + BI - 1) / BI;
    const int64_t jblocks = (n + kUnit * kRows - 1) / (kUnit * kRows);
    const int64_t units = strips * jblocks;
    const int64_t Gtot = (n + GRAN - 1) / GRAN;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 2); }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl ctl{abort_flag, dev_status, limit_ns};

    if (warp == 0) {
        // ---- producer ----
        if (lane == 0) {
            tma_prefetch_desc(&tmap);
            uint32_t it = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const int64_t strip = u % strips, jb = u / strips;
                for (int b = 0; b < kUnit; ++b, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, ctl)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], kBoxBytes);
                    tma_load_2d(ring + s * kBoxBytes, &tmap, &full[s], static_cast<int32_t>(strip * BI),
                                static_cast<int32_t>((jb * kUnit + b) * kRows));
                }
            }
            if (!ok) {
                const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
                for (uint32_t j = first; j < it; ++j) mbar_wait_drain(&full[j % kStages], (j / kStages) & 1u, limit_ns);
            }
        }
        __syncwarp();
    } else {
        // ---- consumers: warp c takes columns [c*4V, c*4V + 4V) of each box ----
        const int cw = warp - 1;
        const int jr = lane >> 2, ic = lane & 3;
        const bool leader = (jr % kLaneSpan) == 0;
        uint32_t it = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int64_t strip = u % strips, jb = u / strips;
            const int64_t i0 = strip * BI + cw * 4 * V + ic * V;
            uint32_t words[V];
#pragma unroll
            for (int c = 0; c < V; ++c) words[c] = 0;
            for (int b = 0; b < kUnit; ++b, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, ctl))) { ok = false; break; }
                const uint8_t* box = ring + s * kBoxBytes;
                uint4 raw[16];
#pragma unroll
                for (int l = 0; l < 16; ++l)
                    raw[l] = *reinterpret_cast<const uint4*>(box + (jr * 16 + l) * 128 + (cw * 4 * V + ic * V) * sizeof(T));
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                const int64_t j0 = (jb * kUnit + b) * kRows + jr * 16;
                float amax[V];
#pragma unroll
                for (int c = 0; c < V; ++c) amax[c] = 0.0f;
#pragma unroll
                for (int l = 0; l < 16; ++l) {
                    const T* t = reinterpret_cast<const T*>(&raw[l]);
#pragma unroll
                    for (int c = 0; c < V; ++c) amax[c] = fmaxf(amax[c], fabsf(to_f32(t[c])));
                }
#pragma unroll
                for (int c = 0; c < V; ++c)
#pragma unroll
                    for (int off = 4; off < 4 * kLaneSpan; off <<= 1)
                        amax[c] = fmaxf(amax[c], __shfl_xor_sync(0xffffffffu, amax[c], off));
                const int64_t g = j0 / GRAN;
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    float sc, f;
                    uint32_t ebyte;
                    group_scale<FMT, RECIP>(amax[c], sc, f, ebyte);
                    const int64_t i = i0 + c;
                    uint32_t w[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const T* t0 = reinterpret_cast<const T*>(&raw[4 * q]);
                        const T* t1 = reinterpret_cast<const T*>(&raw[4 * q + 1]);
                        const T* t2 = reinterpret_cast<const T*>(&raw[4 * q + 2]);
                        const T* t3 = reinterpret_cast<const T*>(&raw[4 * q + 3]);
                        w[q] = quant4(to_f32(t0[c]), to_f32(t1[c]), to_f32(t2[c]), to_f32(t3[c]), f);
                    }
                    if (i < m && j0 < n) {
                        uint8_t* orow = out + i * ldo;
                        if (vec_out && j0 + 16 <= n) {
                            if (QL_IN(bnd, 1, orow + j0, 16))
                                *reinterpret_cast<uint4*>(orow + j0) = make_uint4(w[0], w[1], w[2], w[3]);
                        } else {
                            for (int e = 0; e < 16; ++e)
                                if (j0 + e < n && QL_IN(bnd, 1, orow + j0 + e, 1))
                                    orow[j0 + e] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
                        }
                    }
                    if constexpr (FMT != kSfPacked) {
                        float* sp = static_cast<float*>(sf) + i * ssm + g * ssg;
                        if (leader && i < m && g < Gtot && QL_IN(bnd, 2, sp, 4)) *sp = sc;
                    } else if constexpr (GRAN == 32) {
                        const uint32_t mine = (g < Gtot) ? ebyte : 0u;
                        uint32_t word = 0;
#pragma unroll
                        for (int k = 0; k < 4; ++k) word |= __shfl_sync(0xffffffffu, mine, ic + 8 * k) << (8 * k);
                        const int64_t g0 = (jb * kUnit + b) * kRows / GRAN;
                        int32_t* wp = static_cast<int32_t*>(sf) + i * ssm + (g0 / 4) * ssg;
                        if (jr == 0 && i < m && g0 < Gtot && QL_IN(bnd, 2, wp, 4)) *wp = static_cast<int32_t>(word);
                    } else {
                        words[c] |= ((g < Gtot) ? ebyte : 0u) << (8 * b);
                    }
                }
            }
            if constexpr (FMT == kSfPacked && GRAN == 128) {
                if (ok) {
                    const int64_t g0 = jb * kUnit;
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        const int64_t i = i0 + c;
                        int32_t* wp = static_cast<int32_t*>(sf) + i * ssm + (g0 / 4) * ssg;
                        if (jr == 0 && i < m && g0 < Gtot && QL_IN(bnd, 2, wp, 4)) *wp = static_cast<int32_t>(words[c]);
                    }
                }
            }
        }
    }
    __syncthreads();
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Column-major per-token cast (x_stride_m == 1 and out_stride_m == 1): the
// logical row i is a column of the physical array P[j][i], and the cast's
// output is written in the same physical layout (Q[j][i]), e.g. dY [T, C]
// cast with 1x128 groups along T for the weight gradient, read by the GEMM as
// an MN-major operand, so nothing is transposed in memory. One CTA (16 warps)
// covers 128 physical rows (j) x 32*V columns (i), V = 8 bytes of input per
// lane; warp w takes rows 8w .. 8w+8 and lane l columns l*V .. l*V+V of each,
// so every load and store of a warp is one contiguous run of a physical row.
// Column amaxes are combined over the warps of a group through shared memory.
// 16 registers of input per thread keep two CTAs (32 warps) on each SM.
// ---------------------------------------------------------------------------
namespace colmajor {
constexpr int kWarps = 16;
constexpr int kRowsPerWarp = 8;
constexpr int kLaneBytes = 8;
}  // namespace colmajor

template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(512, 2) cast_colmajor_kernel(const T* __restrict__ x, int64_t m, int64_t n,
                                                               int64_t ldx, uint8_t* __restrict__ out, int64_t ldo,
                                                               void* __restrict__ sf, int64_t ssm, int64_t ssg,
                                                               int vec_in, int vec_out, const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    using namespace colmajor;
    constexpr int V = kLaneBytes / sizeof(T);       // columns per lane (4 bf16 or 2 fp32)
    constexpr int R = kRowsPerWarp;
    constexpr int WPG = GRAN / R;                   // warps per group (16 or 4)
    constexpr int NG = kWarps / WPG;                // groups per tile (1 or 4)
    __shared__ float red[kWarps][32][V + 1];
    __shared__ uint32_t ebuf[NG][32][V];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * 32 * V + lane * V;   // first logical row of this lane
    const int64_t jt = static_cast<int64_t>(blockIdx.y) * (kWarps * R);        // first physical row of the tile
    const int64_t j0 = jt + warp * R;
    const int64_t G = (n + GRAN - 1) / GRAN;

    uint2 raw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t j = j0 + r;
        const T* src = x + j * ldx + i0;
        if (j < n && vec_in && i0 + V <= m) {
            raw[r] = QL_IN(bnd, 0, src, 8) ? __ldg(reinterpret_cast<const uint2*>(src)) : make_uint2(0, 0);
        } else {
            T t[V];
#pragma unroll
            for (int c = 0; c < V; ++c) t[c] = (j < n && i0 + c < m && QL_IN(bnd, 0, src + c, sizeof(T))) ? src[c] : T(0.0f);
            raw[r] = *reinterpret_cast<const uint2*>(t);
        }
    }
    {
        float amax[V];
#pragma unroll
        for (int c = 0; c < V; ++c) amax[c] = 0.0f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const T* t = reinterpret_cast<const T*>(&raw[r]);
#pragma unroll
            for (int c = 0; c < V; ++c) amax[c] = fmaxf(amax[c], fabsf(to_f32(t[c])));
        }
#pragma unroll
        for (int c = 0; c < V; ++c) red[warp][lane][c] = amax[c];
    }
    __syncthreads();
    const int w0 = (warp / WPG) * WPG;              // first warp of this warp's group
    const int64_t g = (jt + w0 * R) / GRAN;         // this warp's group index along j
    const bool group_lead = warp == w0;
    float f[V];
#pragma unroll
    for (int c = 0; c < V; ++c) {
        float a = red[w0][lane][c];
#pragma unroll
        for (int w = 1; w < WPG; ++w) a = fmaxf(a, red[w0 + w][lane][c]);
        float sc;
        uint32_t eb;
        group_scale<FMT, RECIP>(a, sc, f[c], eb);
        const int64_t i = i0 + c;
        if constexpr (FMT != kSfPacked) {
            float* sp = static_cast<float*>(sf) + i * ssm + g * ssg;
            if (group_lead && i < m && g < G && QL_IN(bnd, 2, sp, 4)) *sp = sc;
        } else if constexpr (GRAN == 128) {
            uint8_t* word = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(sf) + i * ssm + (g / 4) * ssg);
            if (group_lead && i < m && g < G && QL_IN(bnd, 2, word, 4)) {
                word[g % 4] = static_cast<uint8_t>(eb);
                if (g == G - 1)
                    for (int z = static_cast<int>(g % 4) + 1; z < 4; ++z) word[z] = 0;
            }
        } else {
            if (group_lead) ebuf[warp / WPG][lane][c] = (g < G) ? eb : 0u;
        }
    }
    // quantise: row r of this lane -> V bytes at Q[j0 + r][i0 .. i0+V)
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t j = j0 + r;
        if (j >= n) break;
        const T* t = reinterpret_cast<const T*>(&raw[r]);
        uint8_t* dst = out + j * ldo + i0;
        uint32_t w = e4m3x2(__fmul_rn(to_f32(t[0]), f[0]), __fmul_rn(to_f32(t[1]), f[1]));
        if constexpr (V == 4)
            w |= e4m3x2(__fmul_rn(to_f32(t[2]), f[2]), __fmul_rn(to_f32(t[3]), f[3])) << 16;
        if (vec_out && i0 + V <= m) {
            if (QL_IN(bnd, 1, dst, V)) {
                if constexpr (V == 4) *reinterpret_cast<uint32_t*>(dst) = w;
                else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w);
            }
        } else {
#pragma unroll
            for (int c = 0; c < V; ++c)
                if (i0 + c < m && QL_IN(bnd, 1, dst + c, 1)) dst[c] = static_cast<uint8_t>(w >> (8 * c));
        }
    }
    if constexpr (FMT == kSfPacked && GRAN == 32) {
        // the four 32-row groups of the tile make one word per logical row
        __syncthreads();
        if (warp == 0) {
            const int64_t gw = jt / 32;                // first group of the tile (a multiple of 4)
#pragma unroll
            for (int c = 0; c < V; ++c) {
                const int64_t i = i0 + c;
                int32_t* wp = static_cast<int32_t*>(sf) + i * ssm + (gw / 4) * ssg;
                if (i < m && gw < G && QL_IN(bnd, 2, wp, 4)) {
                    const uint32_t word = ebuf[0][lane][c] | (ebuf[1][lane][c] << 8) | (ebuf[2][lane][c] << 16) |
                                          (ebuf[3][lane][c] << 24);
                    *wp = static_cast<int32_t>(word);
                }
            }
        }
    }
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Column-major per-token cast, one warp per column chunk (x_stride_m == 1,
// out_stride_m == 1, 16-byte-aligned physical rows): the same operation as
// cast_colmajor_kernel. One producer thread streams stages of 128 physical
// rows (j) x 256 bytes, each two 128-byte-wide boxes loaded with the 128-byte
// swizzle, into a 4-stage shared-memory ring. Each of the 16 consumer warps
// owns one 16-byte column chunk of a stage (8 bf16 or 4 fp32 logical rows i)
// over all 128 physical rows: lane l holds rows l, l+32, l+64 and l+96, which
// the swizzle spreads over all banks. A 1 x GRAN group along j is one quarter
// (GRAN 32) or all four quarters (GRAN 128) of the lanes' rows, so its column
// amax is one warp reduction: redux.sync max on the float bits, which order as
// the values do because every partial amax is a non-negative, non-NaN float
// (each starts at 0 and fmaxf drops NaN). A warp releases the stage once its
// bytes are in registers and computes its scales without waiting for any
// other warp. For bf16 input with a 16-byte-aligned output, the E4M3 rows go
// through a double-buffered 128 x 128-byte output tile (128-byte swizzle) that
// one store thread writes back with a TMA tile store, so every write is a
// full line; otherwise each lane stores its 8 or 4 bytes per row directly.
// Persistent CTAs walk the stages row band by row band; every wait is bounded.
// ---------------------------------------------------------------------------
namespace colmajor_sw {
constexpr int kStages = 4;
constexpr int kRows = 128;                     // physical rows (j) per stage
constexpr int kHalfBytes = kRows * 128;        // one 128-byte-wide box, 16 KB
constexpr int kStageBytes = 2 * kHalfBytes;
constexpr int kOutBytes = kRows * 128;         // E4M3 output tile of a bf16 stage
constexpr int kConsumerWarps = 16;             // 2 boxes x 8 chunks of 16 bytes
constexpr int kThreads = 32 * (2 + kConsumerWarps);   // producer, consumers, store warp
constexpr int kSmemBytes = kStages * kStageBytes + 2 * kOutBytes + 1024 + (2 * kStages + 4) * 8 + 16;
}  // namespace colmajor_sw

template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(colmajor_sw::kThreads, 1)
    cast_colmajor_sw_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap omap,
                            int64_t m, int64_t n, uint8_t* __restrict__ out, int64_t ldo, void* __restrict__ sf,
                            int64_t ssm, int64_t ssg, int vec_out, int tma_out, uint32_t* dev_status,
                            uint64_t limit_ns, const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    using namespace colmajor_sw;
    static_assert(GRAN == 32 || GRAN == 128, "groups of 32 or 128 rows");
    constexpr int E = 16 / sizeof(T);              // columns (logical rows i) per warp
    constexpr int BH = 128 / sizeof(T);            // columns per box
    constexpr int BI = 2 * BH;                     // columns per stage
    constexpr int QPG = GRAN / 32;                 // row quarters per 1 x GRAN group
    constexpr int NGS = 4 / QPG;                   // groups per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* obuf = ring + kStages * kStageBytes;                  // [2][128 rows x 128 bytes], swizzled
    uint64_t* full = reinterpret_cast<uint64_t*>(obuf + 2 * kOutBytes);
    uint64_t* empty = full + kStages;
    uint64_t* ofull = empty + kStages;                               // output tile written by all warps
    uint64_t* oempty = ofull + 2;                                    // output tile read by its TMA store
    volatile int* abort_flag = reinterpret_cast<volatile int*>(oempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t strips = (m + BI - 1) / BI;
    const int64_t bands = (n + kRows - 1) / kRows;
    const int64_t units = strips * bands;
    const int64_t G = (n + GRAN - 1) / GRAN;
    const bool tile_out = sizeof(T) == 2 && tma_out != 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kConsumerWarps); }
        for (int b = 0; b < 2; ++b) { mbar_init(&ofull[b], kConsumerWarps); mbar_init(&oempty[b], 1); }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl ctl{abort_flag, dev_status, limit_ns};

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmap);
            uint32_t it = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++it) {
                const int64_t band = u / strips, strip = u % strips;
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, ctl)) { ok = false; break; }
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                const int32_t x0 = static_cast<int32_t>(strip * BI), y0 = static_cast<int32_t>(band * kRows);
                tma_load_2d(ring + s * kStageBytes, &tmap, &full[s], x0, y0);
                tma_load_2d(ring + s * kStageBytes + kHalfBytes, &tmap, &full[s], x0 + BH, y0);
            }
            if (!ok) {
                const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
                for (uint32_t j = first; j < it; ++j) mbar_wait_drain(&full[j % kStages], (j / kStages) & 1u, limit_ns);
            }
        }
        __syncwarp();
    } else if (warp == kConsumerWarps + 1) {
        if (tile_out && lane == 0) {
            uint32_t it = 0;
            for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++it) {
                const int64_t band = u / strips, strip = u % strips;
                const uint32_t b = it & 1u;
                if (!mbar_wait(&ofull[b], (it >> 1) & 1u, ctl)) break;
                tma_store_2d(&omap, obuf + b * kOutBytes, static_cast<int32_t>(strip * BI),
                             static_cast<int32_t>(band * kRows));
                bulk_commit_group();
                bulk_wait_read_but_one();                    // the previous tile has been read
                if (it > 0) mbar_arrive(&oempty[b ^ 1u]);
            }
            bulk_wait_all();
        }
        __syncwarp();
    } else {
        const int cw = warp - 1;
        const int half = cw >> 3, chunk = cw & 7;
        // byte offset of this lane's 16-byte chunk within a 128-byte swizzled row
        // (rows l + 32q share l & 7, so one offset serves all four quarters)
        const uint32_t col_off = static_cast<uint32_t>((chunk ^ (lane & 7)) << 4);
        // (group, column) pairs of one stage; lane l turns pair l % NP into its scale
        constexpr int NP = NGS * E;
        static_assert(32 % NP == 0, "pairs divide the warp");
        const int pl = lane % NP, p_gi = pl / E, p_e = pl % E;
        int64_t band = blockIdx.x / strips, strip = blockIdx.x % strips;
        uint32_t it = 0;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++it) {
            if (it > 0) {
                strip += gridDim.x;
                while (strip >= strips) { strip -= strips; ++band; }
            }
            const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, ctl))) break;
            const uint8_t* box = ring + s * kStageBytes + half * kHalfBytes;
            uint4 raw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                raw[q] = *reinterpret_cast<const uint4*>(box + (lane + 32 * q) * 128 + col_off);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);

            const int64_t i0 = strip * BI + half * BH + chunk * E;   // first logical row of this warp
            // this lane's |x| maxima per (group, column) as non-negative float bits
            uint32_t am[NGS][E];
#pragma unroll
            for (int gi = 0; gi < NGS; ++gi) {
                if constexpr (sizeof(T) == 2) {
#pragma unroll
                    for (int wd = 0; wd < 4; ++wd) {
                        uint32_t mx = 0u;                    // bf16 pair max of |x| (sign bits cleared)
#pragma unroll
                        for (int q = gi * QPG; q < (gi + 1) * QPG; ++q)
                            mx = bf16x2_max(mx, reinterpret_cast<const uint32_t*>(&raw[q])[wd] & 0x7FFF7FFFu);
                        am[gi][2 * wd] = mx << 16;
                        am[gi][2 * wd + 1] = mx & 0xFFFF0000u;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        float a = 0.0f;
#pragma unroll
                        for (int q = gi * QPG; q < (gi + 1) * QPG; ++q)
                            a = fmaxf(a, fabsf(to_f32(reinterpret_cast<const T*>(&raw[q])[e])));
                        am[gi][e] = __float_as_uint(a);
                    }
                }
            }
            uint32_t mine = 0u;
#pragma unroll
            for (int gi = 0; gi < NGS; ++gi)
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const uint32_t v = __reduce_max_sync(0xffffffffu, am[gi][e]);
                    if (pl == gi * E + e) mine = v;
                }
            float sc, fmine;
            uint32_t eb;
            group_scale<FMT, RECIP>(__uint_as_float(mine), sc, fmine, eb);
            {
                const int64_t i = i0 + p_e;
                const int64_t g = band * NGS + p_gi;
                if constexpr (FMT != kSfPacked) {
                    float* sp = static_cast<float*>(sf) + i * ssm + g * ssg;
                    if (lane < NP && i < m && g < G && QL_IN(bnd, 2, sp, 4)) *sp = sc;
                } else if constexpr (GRAN == 128) {
                    uint8_t* word = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(sf) + i * ssm + (g / 4) * ssg);
                    if (lane < NP && i < m && g < G && QL_IN(bnd, 2, word, 4)) {
                        word[g % 4] = static_cast<uint8_t>(eb);
                        if (g == G - 1)
                            for (int z = static_cast<int>(g % 4) + 1; z < 4; ++z) word[z] = 0;
                    }
                } else {
                    // the stage's four 1 x 32 groups are the four bytes of word `band`
                    const uint32_t b0 = (g < G) ? eb : 0u;
                    const uint32_t b1 = __shfl_sync(0xffffffffu, b0, (lane + E) & 31);
                    const uint32_t b2 = __shfl_sync(0xffffffffu, b0, (lane + 2 * E) & 31);
                    const uint32_t b3 = __shfl_sync(0xffffffffu, b0, (lane + 3 * E) & 31);
                    int32_t* wp = static_cast<int32_t*>(sf) + i * ssm + band * ssg;
                    if (lane < E && i < m && band * 4 < G && QL_IN(bnd, 2, wp, 4))
                        *wp = static_cast<int32_t>(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24));
                }
            }
            float f[NGS][E];
#pragma unroll
            for (int gi = 0; gi < NGS; ++gi)
#pragma unroll
                for (int e = 0; e < E; ++e) f[gi][e] = __shfl_sync(0xffffffffu, fmine, gi * E + e);
            uint8_t* otile = nullptr;
            if (tile_out) {
                const uint32_t b = it & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&oempty[b], ((it >> 1) & 1u) ^ 1u, ctl))) break;
                otile = obuf + b * kOutBytes;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = lane + 32 * q;
                const int64_t j = band * kRows + r;
                const T* t = reinterpret_cast<const T*>(&raw[q]);
                const float* fq = f[q / QPG];
                uint32_t w[E / 4];
#pragma unroll
                for (int b = 0; b < E / 4; ++b)
                    w[b] = e4m3x2(__fmul_rn(to_f32(t[4 * b]), fq[4 * b]), __fmul_rn(to_f32(t[4 * b + 1]), fq[4 * b + 1])) |
                           (e4m3x2(__fmul_rn(to_f32(t[4 * b + 2]), fq[4 * b + 2]),
                                   __fmul_rn(to_f32(t[4 * b + 3]), fq[4 * b + 3])) << 16);
                if constexpr (E == 8) {
                    if (tile_out) {
                        // bytes cw*8 .. cw*8+8 of tile row r, in the store map's 128-byte swizzle;
                        // the TMA store drops rows past n and columns past m
                        *reinterpret_cast<uint2*>(otile + r * 128 + ((((cw >> 1) ^ (r & 7)) << 4) | ((cw & 1) << 3))) =
                            make_uint2(w[0], w[1]);
                        continue;
                    }
                }
                if (j >= n) break;
                uint8_t* dst = out + j * ldo + i0;
                if (vec_out && i0 + E <= m) {
                    if (QL_IN(bnd, 1, dst, E)) {
                        if constexpr (E == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
                        else *reinterpret_cast<uint32_t*>(dst) = w[0];
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        if (i0 + e < m && QL_IN(bnd, 1, dst + e, 1)) dst[e] = static_cast<uint8_t>(w[e / 4] >> (8 * (e % 4)));
                }
            }
            if (tile_out) {
                fence_proxy_async_smem();                    // the tile's bytes are visible to the TMA store
                __syncwarp();
                if (lane == 0) mbar_arrive(&ofull[it & 1u]);
            }
        }
    }
    __syncthreads();
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Generic per-token cast: any strides. One thread per (row, run of four
// groups), so a packed int32 word is always written whole. Slow path.
// ---------------------------------------------------------------------------
template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(128) cast_generic_kernel(const T* __restrict__ x, int64_t m, int64_t n,
                                                           int64_t sxm, int64_t sxn, uint8_t* __restrict__ out,
                                                           int64_t som, int64_t son, void* __restrict__ sf,
                                                           int64_t ssm, int64_t ssg, const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    const int64_t G = (n + GRAN - 1) / GRAN;
    const int64_t W = (G + 3) / 4;
    const int64_t total = m * W;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = t / W, w = t % W;
        uint32_t word = 0;
        for (int q = 0; q < 4; ++q) {
            const int64_t g = w * 4 + q;
            if (g >= G) break;
            const int64_t j0 = g * GRAN, j1 = (j0 + GRAN < n) ? j0 + GRAN : n;
            float amax = 0.0f;
            for (int64_t j = j0; j < j1; ++j)
                if (QL_IN(bnd, 0, x + i * sxm + j * sxn, sizeof(T))) amax = fmaxf(amax, fabsf(to_f32(x[i * sxm + j * sxn])));
            float s, f;
            uint32_t ebyte;
            group_scale<FMT, RECIP>(amax, s, f, ebyte);
            for (int64_t j = j0; j < j1; ++j)
                if (QL_IN(bnd, 0, x + i * sxm + j * sxn, sizeof(T)) && QL_IN(bnd, 1, out + i * som + j * son, 1))
                    out[i * som + j * son] =
                        static_cast<uint8_t>(e4m3x2(__fmul_rn(to_f32(x[i * sxm + j * sxn]), f), 0.0f) & 0xFFu);
            if constexpr (FMT != kSfPacked) {
                float* sp = static_cast<float*>(sf) + i * ssm + g * ssg;
                if (QL_IN(bnd, 2, sp, 4)) *sp = s;
            }
            word |= ebyte << (8 * q);
        }
        if constexpr (FMT == kSfPacked) {
            int32_t* wp = static_cast<int32_t*>(sf) + i * ssm + w * ssg;
            if (QL_IN(bnd, 2, wp, 4)) *wp = static_cast<int32_t>(word);
        }
    }
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// 128x128 block cast. One CTA (256 threads) per block; each thread holds 64
// elements in registers. Loads follow whichever input axis is contiguous; the
// E4M3 bytes are staged in shared memory and written along whichever output
// axis is contiguous, so W and W^T are produced by the same kernel. With
// `sf_t` the block's scale is also written into the scale grid of the
// transposed cast (block (r, c) at [c][r], packed along r): a block's amax
// does not depend on orientation, so that grid is exactly the one
// cast_per_block(W^T) makes, and W's own E4M3 bytes read MN-major with it
// give the data-gradient operand without a second cast.
// in_mode: 0 rows contiguous (vector), 1 columns contiguous (vector), 2 generic
// out_mode: 0 rows contiguous, 1 columns contiguous, 2 generic
// ---------------------------------------------------------------------------
template <typename T, int FMT, bool RECIP>
__global__ void __launch_bounds__(256, sizeof(T) == 2 ? 4 : 2) cast_block_kernel(const T* __restrict__ x, int64_t m, int64_t n,
                                                         int64_t sxm, int64_t sxn, int in_mode,
                                                         uint8_t* __restrict__ out, int64_t som, int64_t son,
                                                         int out_mode, void* __restrict__ sf, int64_t ssr,
                                                         int64_t ssc, void* __restrict__ sf_t, int64_t sst_c,
                                                         int64_t sst_r, const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    constexpr int B = 128;
    // E4M3 bytes of the block, [row][col] with a row pitch of 144 bytes (16-byte
    // rows: 8-byte stores, 16-byte loads) for row-contiguous input, or 129 bytes
    // for column-contiguous input, whose per-lane byte stores go down a column
    // (an odd pitch puts rows 8 apart in distinct banks).
    __shared__ __align__(16) uint8_t qbuf[B * 144];
    const int pitch = (in_mode == 1) ? 129 : 144;
    __shared__ float red[8];
    const int tid = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * B;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * B;

    // element e (0..63) of this thread: (a, b) in block coordinates along the
    // (contiguous, strided) input axes: b = v*16 + tid/16, a = (tid%16)*8 + e%8.
    // The elements are kept as the raw input words (bf16 pairs, or fp32), so
    // the block costs 32 registers of data per thread for bf16 input.
    constexpr int WPG = (8 * static_cast<int>(sizeof(T))) / 4;      // words per 8 elements
    uint32_t raw[8 * WPG];
    auto elem_bits = [&](const T* q) -> uint32_t {
        if constexpr (sizeof(T) == 2) return __bfloat16_as_ushort(*q);
        else return __float_as_uint(*q);
    };
    auto put = [&](int it, int e, uint32_t bits) {
        if constexpr (sizeof(T) == 2) {
            uint32_t& w = raw[it * WPG + e / 2];
            w = (e & 1) ? ((w & 0xFFFFu) | (bits << 16)) : ((w & 0xFFFF0000u) | bits);
        } else {
            raw[it * WPG + e] = bits;
        }
    };
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int bb = it * 16 + tid / 16;
        const int a0 = (tid % 16) * 8;
        int64_t r, c;  // block-relative row/col of element a0
        if (in_mode == 1) { r = a0; c = bb; } else { r = bb; c = a0; }
        const int64_t gr = r0 + r, gc = c0 + c;
        const T* p;
        bool full;
        int64_t step;                                   // element stride along a
        if (in_mode == 0) { p = x + gr * sxm + gc; full = gr < m && gc + 8 <= n; step = 1; }
        else if (in_mode == 1) { p = x + gr + gc * sxn; full = gc < n && gr + 8 <= m; step = 1; }
        else { p = x + gr * sxm + gc * sxn; full = false; step = sxn; }
        if (full && QL_IN(bnd, 0, p, 8 * sizeof(T))) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
            raw[it * WPG + 0] = u.x; raw[it * WPG + 1] = u.y; raw[it * WPG + 2] = u.z; raw[it * WPG + 3] = u.w;
            if constexpr (sizeof(T) == 4) {
                const uint4 u2 = __ldg(reinterpret_cast<const uint4*>(p) + 1);
                raw[it * WPG + 4] = u2.x; raw[it * WPG + 5] = u2.y; raw[it * WPG + 6] = u2.z; raw[it * WPG + 7] = u2.w;
            }
        } else {
#pragma unroll
            for (int w = 0; w < WPG; ++w) raw[it * WPG + w] = 0u;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const bool in = (in_mode == 1) ? (gc < n && gr + e < m) : (gr < m && gc + e < n);
                if (in && QL_IN(bnd, 0, p + e * step, sizeof(T))) put(it, e, elem_bits(p + e * step));
            }
        }
    }
    float amax;
    if constexpr (sizeof(T) == 2) {
        __nv_bfloat162 m2 = __float2bfloat162_rn(0.0f);
#pragma unroll
        for (int w = 0; w < 8 * WPG; ++w) {
            const uint32_t u = raw[w];
            m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&u)));
        }
        amax = fmaxf(__low2float(m2), __high2float(m2));
    } else {
        amax = 0.0f;
#pragma unroll
        for (int w = 0; w < 8 * WPG; ++w) amax = fmaxf(amax, fabsf(__uint_as_float(raw[w])));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    float s, f;
    uint32_t ebyte;
    group_scale<FMT, RECIP>(amax, s, f, ebyte);
    if (tid == 0) {
        const int64_t br = blockIdx.y, bc = blockIdx.x;
        if constexpr (FMT != kSfPacked) {
            float* sp = static_cast<float*>(sf) + br * ssr + bc * ssc;
            if (QL_IN(bnd, 2, sp, 4)) *sp = s;
        } else {
            // packed along the column-block axis: block bc is byte bc % 4 of
            // word bc / 4; the last column block also zeroes the pad bytes
            uint8_t* word = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(sf) + br * ssr + (bc / 4) * ssc);
            if (QL_IN(bnd, 2, word, 4)) {
                word[bc % 4] = static_cast<uint8_t>(ebyte);
                if (bc == static_cast<int64_t>(gridDim.x) - 1)
                    for (int64_t z = bc % 4 + 1; z < 4; ++z) word[z] = 0;
            }
        }
        if (sf_t != nullptr) {
            if constexpr (FMT != kSfPacked) {
                float* sp = static_cast<float*>(sf_t) + bc * sst_c + br * sst_r;
                if (QL_IN(bnd, 3, sp, 4)) *sp = s;
            } else {
                // packed along the row-block axis: block br is byte br % 4 of word br / 4
                uint8_t* word = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(sf_t) + bc * sst_c + (br / 4) * sst_r);
                if (QL_IN(bnd, 3, word, 4)) {
                    word[br % 4] = static_cast<uint8_t>(ebyte);
                    if (br == static_cast<int64_t>(gridDim.y) - 1)
                        for (int64_t z = br % 4 + 1; z < 4; ++z) word[z] = 0;
                }
            }
        }
    }

    // quantise into shared memory, block-relative [row][col]
    auto val = [&](int it, int e) -> float {
        if constexpr (sizeof(T) == 2) {
            const uint32_t w = raw[it * WPG + e / 2];
            return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
        } else {
            return __uint_as_float(raw[it * WPG + e]);
        }
    };
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int bb = it * 16 + tid / 16;
        const int a0 = (tid % 16) * 8;
        const uint32_t lo = quant4_pk(val(it, 0), val(it, 1), val(it, 2), val(it, 3), f);
        const uint32_t hi = quant4_pk(val(it, 4), val(it, 5), val(it, 6), val(it, 7), f);
        if (in_mode == 1) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qbuf[(a0 + e) * pitch + bb] = static_cast<uint8_t>(lo >> (8 * e));
                qbuf[(a0 + 4 + e) * pitch + bb] = static_cast<uint8_t>(hi >> (8 * e));
            }
        } else {
            *reinterpret_cast<uint2*>(&qbuf[bb * pitch + a0]) = make_uint2(lo, hi);
        }
    }
    __syncthreads();
    // store: 16 bytes per thread per pass, 4 passes cover 128 x 128
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int line = p * 32 + tid / 8;    // contiguous output line within the block
        const int off = (tid % 8) * 16;       // 16-byte segment along it
        if (out_mode == 0) {
            const int64_t gr = r0 + line, gc = c0 + off;
            if (gr >= m) continue;
            uint8_t* o = out + gr * som + gc;
            uint4 u;
            if (pitch == 144) {
                u = *reinterpret_cast<const uint4*>(&qbuf[line * pitch + off]);
            } else {
                uint32_t* uw = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint8_t* b = &qbuf[line * pitch + off + 4 * e];
                    uw[e] = b[0] | (b[1] << 8) | (b[2] << 16) | (static_cast<uint32_t>(b[3]) << 24);
                }
            }
            if (gc + 16 <= n) {
                if (QL_IN(bnd, 1, o, 16)) *reinterpret_cast<uint4*>(o) = u;
            } else {
                const uint8_t* ub = reinterpret_cast<const uint8_t*>(&u);
                for (int e = 0; e < 16; ++e)
                    if (gc + e < n && QL_IN(bnd, 1, o + e, 1)) o[e] = ub[e];
            }
        } else if (out_mode == 1) {
            const int64_t gc = c0 + line, gr = r0 + off;
            if (gc >= n) continue;
            uint8_t* o = out + gr + gc * son;
            uint8_t b16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) b16[e] = qbuf[(off + e) * pitch + line];
            if (gr + 16 <= m) {
                uint4 u;
                uint32_t* uw = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    uw[e] = b16[4 * e] | (b16[4 * e + 1] << 8) | (b16[4 * e + 2] << 16) | (static_cast<uint32_t>(b16[4 * e + 3]) << 24);
                if (QL_IN(bnd, 1, o, 16)) *reinterpret_cast<uint4*>(o) = u;
            } else {
                for (int e = 0; e < 16; ++e)
                    if (gr + e < m && QL_IN(bnd, 1, o + e, 1)) o[e] = b16[e];
            }
        } else {
            const int64_t gr = r0 + line, gc = c0 + off;
            if (gr >= m) continue;
            for (int e = 0; e < 16; ++e)
                if (gc + e < n && QL_IN(bnd, 1, out + gr * som + (gc + e) * son, 1))
                    out[gr * som + (gc + e) * son] = qbuf[line * pitch + off + e];
        }
    }
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Dual per-token cast: from one read of a row-contiguous x [m, n], both the
// per-token cast of x (1 x 128 groups along n: the forward / data-gradient
// operand) and the per-token cast of x^T (1 x 128 groups along m: the
// weight-gradient operand, kept in x's own [m, n] layout for the MN-major
// GEMM). A 128 x 128 tile of x holds exactly 128 groups of each cast: its rows
// and its columns. One CTA of 512 threads per tile: thread t holds rows
// 32i + t/16 (i < 4) at columns 8(t%16) .. +8 as raw input words, so a row's
// amax is a 16-lane reduction and a column's a reduction over the thread's 4
// rows, the lane 16 apart and the 16 warps (through shared memory). Each row's and column's
// scale is made by one thread; the E4M3 bytes of both casts leave with one
// 8-byte store per row per cast (16 threads cover 128 contiguous bytes).
// ---------------------------------------------------------------------------
namespace dual {
constexpr int kRowsPerThread = 4;                         // of the tile's 128 rows
constexpr int kThreads = 16 * (128 / kRowsPerThread);      // 16 threads per row: 512
constexpr int kWarps = kThreads / 32;
}  // namespace dual

// Input value e (< 8) of the thread's it-th row from its raw words.
template <typename T>
__device__ __forceinline__ float dual_val(const uint32_t* raw, int it, int e) {
    constexpr int WPG = (8 * static_cast<int>(sizeof(T))) / 4;      // words per 8 elements
    if constexpr (sizeof(T) == 2) {
        const uint32_t w = raw[it * WPG + e / 2];
        return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
    } else {
        return __uint_as_float(raw[it * WPG + e]);
    }
}

// First half of a tile: the column maxima over this warp's rows into red[warp]
// and the maxima of the thread's rows (one half-warp per row; non-negative
// floats order as their bits).
template <typename T>
__device__ __forceinline__ void dual_maxima(const uint32_t* raw, float (*red)[128], int a0, int lane, int warp,
                                            uint32_t (&rmax)[dual::kRowsPerThread]) {
    constexpr int NIT = dual::kRowsPerThread;
    const uint32_t half = 0xFFFFu << (lane & 16);
    if constexpr (sizeof(T) == 2) {
        // bf16: maxima of |x| on pairs of columns (max.bf16x2 is exact and,
        // like fmaxf, returns the other operand for a NaN; an all-NaN pair
        // reaches red as NaN, which the column reduction's fmaxf from 0 drops)
        uint32_t ab[NIT][4];
#pragma unroll
        for (int it = 0; it < NIT; ++it)
#pragma unroll
            for (int w = 0; w < 4; ++w) ab[it][w] = raw[it * 4 + w] & 0x7FFF7FFFu;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t c = bf16x2_max(bf16x2_max(ab[0][w], ab[1][w]), bf16x2_max(ab[2][w], ab[3][w]));
            c = bf16x2_max(c, __shfl_xor_sync(0xffffffffu, c, 16));
            if (lane < 16) {
                red[warp][a0 + 2 * w] = __uint_as_float(c << 16);
                red[warp][a0 + 2 * w + 1] = __uint_as_float(c & 0xFFFF0000u);
            }
        }
        static_assert(dual::kRowsPerThread == 4, "four rows per thread");
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const uint32_t r = bf16x2_max(bf16x2_max(ab[it][0], ab[it][1]), bf16x2_max(ab[it][2], ab[it][3]));
            const float a = fmaxf(fmaxf(0.0f, __uint_as_float(r << 16)), __uint_as_float(r & 0xFFFF0000u));
            rmax[it] = __reduce_max_sync(half, __float_as_uint(a));
        }
    } else {
        float cmax[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float a = 0.0f;
#pragma unroll
            for (int it = 0; it < NIT; ++it) a = fmaxf(a, fabsf(dual_val<T>(raw, it, e)));
            cmax[e] = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
        }
        if (lane < 16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) red[warp][a0 + e] = cmax[e];
        }
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            float a = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(dual_val<T>(raw, it, e)));
            rmax[it] = __reduce_max_sync(half, __float_as_uint(a));
        }
    }
}

// Output pointers and strides of the dual cast.
struct DualOut {
    uint8_t* qr;
    int64_t ldr;
    void* sfr;
    int64_t srm, srg;
    uint8_t* qc;
    int64_t ldc;
    void* sfc;
    int64_t scn, scg;
    int vec_out;
};

// Second half of a tile (after the barrier that completes red): the row and
// column scales, one thread per row and per column, then the E4M3 bytes of
// both casts, 8 per row per cast (16 threads cover 128 contiguous bytes).
// last_bc / last_br: the tile is in the last column / row block (packed words
// there are completed with zero bytes). Contains one __syncthreads.
template <typename T, int FMT, bool RECIP>
__device__ __forceinline__ void dual_emit(const uint32_t* raw, const uint32_t (&rmax)[dual::kRowsPerThread],
                                          float (*red)[128], float* fcol, int64_t br, int64_t bc, bool last_br,
                                          bool last_bc, int64_t m, int64_t n, const DualOut& o, const Bounds& bnd) {
    constexpr int NIT = dual::kRowsPerThread;
    constexpr int RS = 128 / NIT;       // rows between a thread's rows
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t r0 = br * 128, c0 = bc * 128;
    const int a0 = (tid % 16) * 8;
    const int64_t gc = c0 + a0;
    // lane i (i < NIT) of each half-warp makes the scale of its i-th row
    const int my_it = lane & 15;
    uint32_t mine = rmax[0];
#pragma unroll
    for (int it = 1; it < NIT; ++it)
        if (my_it == it) mine = rmax[it];
    float s_r, f_r;
    uint32_t e_r;
    group_scale<FMT, RECIP>(__uint_as_float(mine), s_r, f_r, e_r);
    if (my_it < NIT) {
        const int64_t gr = r0 + my_it * RS + tid / 16;
        if (gr < m) {
            if constexpr (FMT != kSfPacked) {
                float* sp = static_cast<float*>(o.sfr) + gr * o.srm + bc * o.srg;
                if (QL_IN(bnd, 2, sp, 4)) *sp = s_r;
            } else {
                uint8_t* word = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(o.sfr) + gr * o.srm + (bc / 4) * o.srg);
                if (QL_IN(bnd, 2, word, 4)) {
                    word[bc % 4] = static_cast<uint8_t>(e_r);
                    if (last_bc)
                        for (int64_t z = bc % 4 + 1; z < 4; ++z) word[z] = 0;
                }
            }
        }
    }
    float frow[NIT];
#pragma unroll
    for (int it = 0; it < NIT; ++it) frow[it] = __shfl_sync(0xffffffffu, f_r, (lane & 16) + it);
    if (tid < 128) {
        float a = 0.0f;
#pragma unroll
        for (int w = 0; w < dual::kWarps; ++w) a = fmaxf(a, red[w][tid]);
        float s_c, f_c;
        uint32_t e_c;
        group_scale<FMT, RECIP>(a, s_c, f_c, e_c);
        fcol[tid] = f_c;
        const int64_t col = c0 + tid;
        if (col < n) {
            if constexpr (FMT != kSfPacked) {
                float* sp = static_cast<float*>(o.sfc) + col * o.scn + br * o.scg;
                if (QL_IN(bnd, 4, sp, 4)) *sp = s_c;
            } else {
                uint8_t* word = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(o.sfc) + col * o.scn + (br / 4) * o.scg);
                if (QL_IN(bnd, 4, word, 4)) {
                    word[br % 4] = static_cast<uint8_t>(e_c);
                    if (last_br)
                        for (int64_t z = br % 4 + 1; z < 4; ++z) word[z] = 0;
                }
            }
        }
    }
    __syncthreads();
    float fc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) fc[e] = fcol[a0 + e];
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int64_t gr = r0 + it * RS + tid / 16;
        if (gr >= m) continue;
        auto v = [&](int e) { return dual_val<T>(raw, it, e); };
        const uint32_t r_lo = quant4(v(0), v(1), v(2), v(3), frow[it]);
        const uint32_t r_hi = quant4(v(4), v(5), v(6), v(7), frow[it]);
        const uint32_t c_lo = e4m3x2(__fmul_rn(v(0), fc[0]), __fmul_rn(v(1), fc[1])) |
                              (e4m3x2(__fmul_rn(v(2), fc[2]), __fmul_rn(v(3), fc[3])) << 16);
        const uint32_t c_hi = e4m3x2(__fmul_rn(v(4), fc[4]), __fmul_rn(v(5), fc[5])) |
                              (e4m3x2(__fmul_rn(v(6), fc[6]), __fmul_rn(v(7), fc[7])) << 16);
        uint8_t* dr = o.qr + gr * o.ldr + gc;
        uint8_t* dc = o.qc + gr * o.ldc + gc;
        if (o.vec_out && gc + 8 <= n) {
            if (QL_IN(bnd, 1, dr, 8)) *reinterpret_cast<uint2*>(dr) = make_uint2(r_lo, r_hi);
            if (QL_IN(bnd, 3, dc, 8)) *reinterpret_cast<uint2*>(dc) = make_uint2(c_lo, c_hi);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (gc + e < n) {
                    if (QL_IN(bnd, 1, dr + e, 1)) dr[e] = static_cast<uint8_t>((e < 4 ? r_lo : r_hi) >> (8 * (e & 3)));
                    if (QL_IN(bnd, 3, dc + e, 1)) dc[e] = static_cast<uint8_t>((e < 4 ? c_lo : c_hi) >> (8 * (e & 3)));
                }
            }
        }
    }
}

// One CTA per tile; each thread loads its four rows' 8 elements from x.
template <typename T, int FMT, bool RECIP>
__global__ void __launch_bounds__(dual::kThreads, 2)
    cast_dual_kernel(const T* __restrict__ x, int64_t m, int64_t n, int64_t ldx, const DualOut o, int vec_in,
                     const Bounds bnd) {
    pdl_wait_prior();           // the previous kernel's writes are complete and visible
    constexpr int WPG = (8 * static_cast<int>(sizeof(T))) / 4;      // words per 8 elements
    constexpr int NIT = dual::kRowsPerThread;
    constexpr int RS = 128 / NIT;
    __shared__ float red[dual::kWarps][128];   // per-warp column maxima
    __shared__ float fcol[128];         // column factors
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t br = blockIdx.y, bc = blockIdx.x;
    const int64_t r0 = br * 128, c0 = bc * 128;
    const int a0 = (tid % 16) * 8;
    const int64_t gc = c0 + a0;

    uint32_t raw[NIT * WPG];
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int64_t gr = r0 + it * RS + tid / 16;
        const T* p = x + gr * ldx + gc;
        if (vec_in && gr < m && gc + 8 <= n && QL_IN(bnd, 0, p, 8 * sizeof(T))) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
            raw[it * WPG + 0] = u.x; raw[it * WPG + 1] = u.y; raw[it * WPG + 2] = u.z; raw[it * WPG + 3] = u.w;
            if constexpr (sizeof(T) == 4) {
                const uint4 u2 = __ldg(reinterpret_cast<const uint4*>(p) + 1);
                raw[it * WPG + 4] = u2.x; raw[it * WPG + 5] = u2.y; raw[it * WPG + 6] = u2.z; raw[it * WPG + 7] = u2.w;
            }
        } else {
            union { uint32_t w[WPG]; T t[8]; } tmp;
#pragma unroll
            for (int e = 0; e < 8; ++e) tmp.t[e] = (gr < m && gc + e < n && QL_IN(bnd, 0, p + e, sizeof(T))) ? p[e] : T(0.0f);
#pragma unroll
            for (int w = 0; w < WPG; ++w) raw[it * WPG + w] = tmp.w[w];
        }
    }
    uint32_t rmax[NIT];
    dual_maxima<T>(raw, red, a0, lane, warp, rmax);
    __syncthreads();
    dual_emit<T, FMT, RECIP>(raw, rmax, red, fcol, br, bc, br == static_cast<int64_t>(gridDim.y) - 1,
                             bc == static_cast<int64_t>(gridDim.x) - 1, m, n, o, bnd);
    // this CTA's work is done: the next kernel of the stream may be scheduled
    pdl_launch_dependents();
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream finishes; every cast kernel waits
// for that kernel (griddepcontrol.wait) before it reads or writes memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Byte ranges of the buffers of each cast (checked in bounds-checked builds).
Bounds token_bounds(const CastTokenArgs& a, int64_t es, int gran, int fmt) {
    Bounds b{};
    const int64_t G = (a.n + gran - 1) / gran;
    b.s[0] = span_of(a.x, es, a.m, a.sxm, a.n, a.sxn);
    b.s[1] = span_of(a.out, 1, a.m, a.som, a.n, a.son);
    b.s[2] = span_of(a.sf, 4, a.m, a.ssm, fmt == kSfPacked ? (G + 3) / 4 : G, a.ssg);
    b.status = a.dev_status;
    return b;
}

Bounds block_bounds(const CastBlockArgs& a, int64_t es, int fmt) {
    Bounds b{};
    const int64_t rb = (a.m + 127) / 128, cb = (a.n + 127) / 128;
    const bool packed = fmt == kSfPacked;
    b.s[0] = span_of(a.x, es, a.m, a.sxm, a.n, a.sxn);
    b.s[1] = span_of(a.out, 1, a.m, a.som, a.n, a.son);
    b.s[2] = span_of(a.sf, 4, rb, a.ssr, packed ? (cb + 3) / 4 : cb, a.ssc);
    b.s[3] = span_of(a.sf_t, 4, cb, a.sst_c, packed ? (rb + 3) / 4 : rb, a.sst_r);
    b.status = a.dev_status;
    return b;
}

Bounds dual_bounds(const CastDualArgs& a, int64_t es, int fmt) {
    Bounds b{};
    const int64_t gr = (a.n + 127) / 128, gc = (a.m + 127) / 128;
    const bool packed = fmt == kSfPacked;
    b.s[0] = span_of(a.x, es, a.m, a.sxm, a.n, 1);
    b.s[1] = span_of(a.qr, 1, a.m, a.ldr, a.n, 1);
    b.s[2] = span_of(a.sfr, 4, a.m, a.srm, packed ? (gr + 3) / 4 : gr, a.srg);
    b.s[3] = span_of(a.qc, 1, a.m, a.ldc, a.n, 1);
    b.s[4] = span_of(a.sfc, 4, a.n, a.scn, packed ? (gc + 3) / 4 : gc, a.scg);
    b.status = a.dev_status;
    return b;
}

template <typename T, int GRAN, int FMT, bool RECIP>
cudaError_t launch_token_t(const CastTokenArgs& a, cudaStream_t st, int num_sms) {
    const T* x = static_cast<const T*>(a.x);
    const Bounds bnd = token_bounds(a, sizeof(T), GRAN, FMT);
    if (a.sxn == 1 && a.son == 1) {
        const int vec_in = aligned16(x) && ((a.sxm * static_cast<int64_t>(sizeof(T))) % 16 == 0);
        const int vec_out = aligned16(a.out) && (a.som % 16 == 0);
        const int64_t chunks = (a.n + 32 * (64 / sizeof(T)) - 1) / (32 * (64 / sizeof(T)));
        const int64_t warps = a.m * chunks;
        int64_t blocks = (warps + 7) / 8;
        // one resident wave (4 CTAs of 8 warps per SM) walks all tasks: no CTA
        // launches after the first, and a shorter tail at sub-L2 sizes
        const int64_t cap = static_cast<int64_t>(num_sms) * 4;
        if (blocks > cap) blocks = cap;
        return launch_pdl(cast_rows_kernel<T, GRAN, FMT, RECIP>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                          x, a.m, a.n, a.sxm, a.out, a.som, a.sf, a.ssm, a.ssg, chunks, vec_in, vec_out, bnd);
    }
    if (a.sxm == 1 && a.som == 1 && a.tma_ok) {
        using namespace colmajor_sw;
        constexpr int E = 16 / sizeof(T);
        constexpr int BH = 128 / sizeof(T);
        CUtensorMap tmap;
        if (encode_2d_map(&tmap, x, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          a.n, a.m, a.sxn * static_cast<int64_t>(sizeof(T)), kRows, BH, /*swizzle=*/128)) {
            const int vec_out = ((reinterpret_cast<uintptr_t>(a.out) % E) == 0) && (a.son % E == 0);
            CUtensorMap omap = {};
            // a TMA store may write a row's last 16-byte chunk whole: rows must start and end aligned
            const int tma_out = sizeof(T) == 2 && aligned16(a.out) && a.son > 0 && a.son % 16 == 0 &&
                                a.m % 16 == 0 &&
                                encode_2d_map(&omap, a.out, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.n, a.m, a.son, kRows, 128,
                                              /*swizzle=*/128);
            auto kern = cast_colmajor_sw_kernel<T, GRAN, FMT, RECIP>;
            if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), kSmemBytes); e != cudaSuccess)
                return e;
            const int64_t units = ((a.m + 2 * BH - 1) / (2 * BH)) * ((a.n + kRows - 1) / kRows);
            int64_t grid = num_sms;
            if (grid > units) grid = units;
            return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, st, tmap, omap, a.m,
                              a.n, a.out, a.son, a.sf, a.ssm, a.ssg, vec_out, tma_out, a.dev_status, a.wait_limit_ns, bnd);
        }
    }
    if (a.sxm == 1 && a.som == 1) {
        constexpr int V = colmajor::kLaneBytes / sizeof(T);
        const int vec_in = (reinterpret_cast<uintptr_t>(x) % 8 == 0) && ((a.sxn * static_cast<int64_t>(sizeof(T))) % 8 == 0);
        const int vec_out = ((reinterpret_cast<uintptr_t>(a.out) % V) == 0) && (a.son % V == 0);
        dim3 grid(static_cast<unsigned>((a.m + 32 * V - 1) / (32 * V)), static_cast<unsigned>((a.n + 127) / 128));
        return launch_pdl(cast_colmajor_kernel<T, GRAN, FMT, RECIP>, grid, dim3(32 * colmajor::kWarps), 0, st, x, a.m,
                          a.n, a.sxn, a.out, a.son, a.sf, a.ssm, a.ssg, vec_in, vec_out, bnd);
    }
    if (a.sxm == 1 && a.son == 1 && a.tma_ok) {
        using namespace cols_tma;
        constexpr int BI = 128 / sizeof(T);
        CUtensorMap tmap;
        if (encode_2d_map(&tmap, x, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          a.n, a.m, a.sxn * static_cast<int64_t>(sizeof(T)), kRows, BI)) {
            const int vec_out = aligned16(a.out) && (a.som % 16 == 0);
            const int smem = kStages * kBoxBytes + 2 * kStages * 8 + 16 + 1024;
            auto kern = cast_cols_tma_kernel<T, GRAN, FMT, RECIP>;
            if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem); e != cudaSuccess)
                return e;
            const int64_t units = ((a.m + BI - 1) / BI) * ((a.n + kUnit * kRows - 1) / (kUnit * kRows));
            int64_t grid = static_cast<int64_t>(num_sms) * 3;
            if (grid > units) grid = units;
            return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, st, tmap, a.m, a.n, a.out,
                              a.som, a.sf, a.ssm, a.ssg, vec_out, a.dev_status, a.wait_limit_ns, bnd);
        }
    }
    if (a.sxm == 1 && a.son == 1) {
        constexpr int V = 16 / sizeof(T);
        const int vec_in = aligned16(x) && ((a.sxn * static_cast<int64_t>(sizeof(T))) % 16 == 0);
        const int vec_out = aligned16(a.out) && (a.som % 16 == 0);
        constexpr int kRowsPerCta = (FMT == kSfPacked && GRAN == 128) ? 512 : 128;
        dim3 grid(static_cast<unsigned>((a.m + 32 * V - 1) / (32 * V)),
                  static_cast<unsigned>((a.n + kRowsPerCta - 1) / kRowsPerCta));
        return launch_pdl(cast_cols_kernel<T, GRAN, FMT, RECIP>, grid, dim3(256), 0, st, x, a.m, a.n, a.sxn, a.out,
                          a.som, a.sf, a.ssm, a.ssg, vec_in, vec_out, bnd);
    }
    const int64_t G = (a.n + GRAN - 1) / GRAN;
    const int64_t total = a.m * ((G + 3) / 4);
    int64_t blocks = (total + 127) / 128;
    if (blocks > static_cast<int64_t>(num_sms) * 16) blocks = static_cast<int64_t>(num_sms) * 16;
    if (blocks < 1) blocks = 1;
    return launch_pdl(cast_generic_kernel<T, GRAN, FMT, RECIP>, dim3(static_cast<unsigned>(blocks)), dim3(128), 0, st,
                      x, a.m, a.n, a.sxm, a.sxn, a.out, a.som, a.son, a.sf, a.ssm, a.ssg, bnd);
}

template <typename T, int GRAN>
cudaError_t launch_token_fmt(const CastTokenArgs& a, cudaStream_t st, int num_sms) {
    switch (a.fmt) {
        case kSfFp32: return a.recip ? launch_token_t<T, GRAN, kSfFp32, true>(a, st, num_sms)
                                     : launch_token_t<T, GRAN, kSfFp32, false>(a, st, num_sms);
        case kSfUe8m0: return launch_token_t<T, GRAN, kSfUe8m0, false>(a, st, num_sms);
        default: return launch_token_t<T, GRAN, kSfPacked, false>(a, st, num_sms);
    }
}

template <typename T, int FMT, bool RECIP>
cudaError_t launch_block_t(const CastBlockArgs& a, cudaStream_t st) {
    const T* x = static_cast<const T*>(a.x);
    const int64_t es = sizeof(T);
    int in_mode = 2;
    if (a.sxn == 1 && aligned16(x) && (a.sxm * es) % 16 == 0) in_mode = 0;
    else if (a.sxm == 1 && aligned16(x) && (a.sxn * es) % 16 == 0) in_mode = 1;
    int out_mode = 2;
    if (a.son == 1 && aligned16(a.out) && a.som % 16 == 0) out_mode = 0;
    else if (a.som == 1 && aligned16(a.out) && a.son % 16 == 0) out_mode = 1;
    dim3 grid(static_cast<unsigned>((a.n + 127) / 128), static_cast<unsigned>((a.m + 127) / 128));
    return launch_pdl(cast_block_kernel<T, FMT, RECIP>, grid, dim3(256), 0, st, x, a.m, a.n, a.sxm, a.sxn, in_mode,
                      a.out, a.som, a.son, out_mode, a.sf, a.ssr, a.ssc, a.sf_t, a.sst_c, a.sst_r,
                      block_bounds(a, es, FMT));
}

template <typename T>
cudaError_t launch_block_fmt(const CastBlockArgs& a, cudaStream_t st) {
    if (a.fmt == kSfUe8m0) return launch_block_t<T, kSfUe8m0, false>(a, st);
    if (a.fmt == kSfPacked) return launch_block_t<T, kSfPacked, false>(a, st);
    return a.recip ? launch_block_t<T, kSfFp32, true>(a, st) : launch_block_t<T, kSfFp32, false>(a, st);
}

}  // namespace

cudaError_t launch_cast_per_token(const CastTokenArgs& a, cudaStream_t st, int num_sms) {
    if (a.is_bf16) {
        return a.gran == 32 ? launch_token_fmt<__nv_bfloat16, 32>(a, st, num_sms)
                            : launch_token_fmt<__nv_bfloat16, 128>(a, st, num_sms);
    }
    return a.gran == 32 ? launch_token_fmt<float, 32>(a, st, num_sms) : launch_token_fmt<float, 128>(a, st, num_sms);
}

cudaError_t launch_cast_per_block(const CastBlockArgs& a, cudaStream_t st) {
    return a.is_bf16 ? launch_block_fmt<__nv_bfloat16>(a, st) : launch_block_fmt<float>(a, st);
}

namespace {

template <typename T, int FMT, bool RECIP>
cudaError_t launch_dual_t(const CastDualArgs& a, cudaStream_t st) {
    const T* x = static_cast<const T*>(a.x);
    const int vec_in = aligned16(x) && (a.sxm * static_cast<int64_t>(sizeof(T))) % 16 == 0;
    const int vec_out = (reinterpret_cast<uintptr_t>(a.qr) % 8 == 0) && (reinterpret_cast<uintptr_t>(a.qc) % 8 == 0) &&
                        a.ldr % 8 == 0 && a.ldc % 8 == 0;
    const DualOut o{a.qr, a.ldr, a.sfr, a.srm, a.srg, a.qc, a.ldc, a.sfc, a.scn, a.scg, vec_out};
    dim3 grid(static_cast<unsigned>((a.n + 127) / 128), static_cast<unsigned>((a.m + 127) / 128));
    return launch_pdl(cast_dual_kernel<T, FMT, RECIP>, grid, dim3(dual::kThreads), 0, st, x, a.m, a.n, a.sxm, o, vec_in,
                      dual_bounds(a, sizeof(T), FMT));
}

template <typename T>
cudaError_t launch_dual_fmt(const CastDualArgs& a, cudaStream_t st) {
    if (a.fmt == kSfUe8m0) return launch_dual_t<T, kSfUe8m0, false>(a, st);
    if (a.fmt == kSfPacked) return launch_dual_t<T, kSfPacked, false>(a, st);
    return a.recip ? launch_dual_t<T, kSfFp32, true>(a, st) : launch_dual_t<T, kSfFp32, false>(a, st);
}

}  // namespace

cudaError_t launch_cast_dual(const CastDualArgs& a, cudaStream_t st) {
    return a.is_bf16 ? launch_dual_fmt<__nv_bfloat16>(a, st) : launch_dual_fmt<float>(a, st);
}

}  // namespace ql
