// FP8 casts for sm_103a.
//
// Per-token cast ("DeepGEMM Essentials: High-Performance FP8 Matrix
// Multiplication" Part 3, options of "deep-gemm: fused per-token FP8 cast in
// Triton (fused_per_token_cast_to_fp8), version 3") and 128x128 block cast
// (Part 4). Each kernel reads its input once from HBM and writes E4M3 data and
// scales straight into the caller's (possibly strided) views.
//
// Arithmetic per group (bit-exact):
//   amax = max(|x|) in fp32 (exact), clamped below at the float nearest 1e-4
//   fp32 scales : s = amax / 448 and f = 448 / amax, both correctly rounded
//                 (or f = 1 / s with the recip-of-scale option)
//   UE8M0       : s rounded up to a power of two: E = biased exponent of s,
//                 plus one if s has any mantissa bit; f = 2^(127 - E) exactly
//   data        : E4M3 round-to-nearest-even of fl32(x * f), sign kept
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cast.cuh"

namespace ql {
namespace {

constexpr int kSfFp32 = 0, kSfUe8m0 = 1, kSfPacked = 2;

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Scale, factor and UE8M0 exponent byte of one group from its amax.
template <int FMT, bool RECIP>
__device__ __forceinline__ void group_scale(float amax, float& s_store, float& f, uint32_t& ebyte) {
    const float a = fmaxf(amax, 1e-4f);          // 1e-4f is the float nearest 1e-4
    const float s = __fdiv_rn(a, 448.0f);
    if constexpr (FMT == kSfFp32) {
        s_store = s;
        f = RECIP ? __fdiv_rn(1.0f, s) : __fdiv_rn(448.0f, a);
        ebyte = 0;
    } else {
        const uint32_t b = __float_as_uint(s);   // s is a positive normal float
        const uint32_t E = ((b >> 23) & 0xFFu) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
        s_store = __uint_as_float(E << 23);
        f = __uint_as_float((254u - E) << 23);   // 2^(127 - E)
        ebyte = E;
    }
}

// Two fp32 values to two E4M3 bytes (lo -> low byte), round to nearest even.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float f) {
    return e4m3x2(__fmul_rn(a, f), __fmul_rn(b, f)) | (e4m3x2(__fmul_rn(c, f), __fmul_rn(d, f)) << 16);
}

// ---------------------------------------------------------------------------
// Row-contiguous per-token cast (x_stride_n == 1, out_stride_n == 1).
// One warp task = (row, chunk of 32*E elements); each lane owns E consecutive
// elements, E = 64 bytes of input (32 bf16 or 16 fp32: four 16-byte loads, all
// issued before use), so a group of G elements is G/E consecutive lanes and its
// amax is a shuffle reduction over them (none for bf16 with G = 32).
// ---------------------------------------------------------------------------
template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(256) cast_rows_kernel(const T* __restrict__ x, int64_t m, int64_t n, int64_t ldx,
                                                        uint8_t* __restrict__ out, int64_t ldo,
                                                        void* __restrict__ sf, int64_t ssm, int64_t ssg,
                                                        int64_t chunks_per_row, int vec_in, int vec_out) {
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
                raw[l] = __ldg(reinterpret_cast<const uint4*>(xr + e));
            } else {
                T tmp[kVec];
#pragma unroll
                for (int i = 0; i < kVec; ++i) tmp[i] = (e + i < n) ? xr[e + i] : T(0.0f);
                raw[l] = *reinterpret_cast<const uint4*>(tmp);
            }
        }
        float v[kElemsPerLane];
#pragma unroll
        for (int l = 0; l < kLoads; ++l) {
            const T* t = reinterpret_cast<const T*>(&raw[l]);
#pragma unroll
            for (int i = 0; i < kVec; ++i) v[l * kVec + i] = to_f32(t[i]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kElemsPerLane; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int off = 1; off < kLanesPerGroup; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

        float s, f;
        uint32_t ebyte;
        group_scale<FMT, RECIP>(amax, s, f, ebyte);

        if (e0 < n) {
            uint8_t* orow = out + row * ldo;
            uint32_t w[kElemsPerLane / 4];
#pragma unroll
            for (int q = 0; q < kElemsPerLane / 4; ++q) w[q] = quant4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], f);
            if (vec_out && e0 + kElemsPerLane <= n) {
#pragma unroll
                for (int q = 0; q < kElemsPerLane / 16; ++q)
                    *reinterpret_cast<uint4*>(orow + e0 + 16 * q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < kElemsPerLane; ++i)
                    if (e0 + i < n) orow[e0 + i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
            }
        }

        const int64_t g = e0 / GRAN;
        if constexpr (FMT != kSfPacked) {
            if ((lane % kLanesPerGroup) == 0 && g < G) static_cast<float*>(sf)[row * ssm + g * ssg] = s;
        } else {
            // four consecutive groups per int32 word; groups past the last are 0
            constexpr int kWordLanes = 4 * kLanesPerGroup;  // 4 .. 32
            const uint32_t mine = (g < G) ? ebyte : 0u;
            const int base = (lane / kWordLanes) * kWordLanes;
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word |= __shfl_sync(0xffffffffu, mine, base + j * kLanesPerGroup) << (8 * j);
            if ((lane % kWordLanes) == 0 && g < G)
                static_cast<int32_t*>(sf)[row * ssm + (g / 4) * ssg] = static_cast<int32_t>(word);
        }
    }
}

// ---------------------------------------------------------------------------
// Transposed per-token cast (x_stride_m == 1): logical row i is a column of the
// physical array P[j][i] = x[i + j*ldx]. A CTA stages a TJ x 32 tile of P in
// shared memory (coalesced 32-wide loads along i), reduces each logical row's
// groups down the tile's columns, then writes each logical row's TJ bytes
// contiguously (16 B per thread).
// TJ = 128, or 4*GRAN for packed UE8M0 (so a CTA owns whole int32 words).
// ---------------------------------------------------------------------------
template <typename T, int GRAN, int FMT, bool RECIP, int TJ>
__global__ void __launch_bounds__(256) cast_cols_kernel(const T* __restrict__ x, int64_t m, int64_t n, int64_t ldx,
                                                        uint8_t* __restrict__ out, int64_t ldo,
                                                        void* __restrict__ sf, int64_t ssm, int64_t ssg,
                                                        int vec_out) {
    constexpr int TI = 32;
    constexpr int kGroups = TJ / GRAN;
    constexpr int kParts = TJ / 16;          // 16-row partial reductions per column
    extern __shared__ float smem_cast[];
    float* tile = smem_cast;                 // [TJ][TI + 1]
    float* part = tile + TJ * (TI + 1);      // [kParts][TI]
    float* fac = part + kParts * TI;         // [kGroups][TI]
    uint32_t* ebuf = reinterpret_cast<uint32_t*>(fac + kGroups * TI);  // [kGroups][TI]

    const int tid = threadIdx.x;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * TI;
    const int64_t j0 = static_cast<int64_t>(blockIdx.y) * TJ;

    // load: warp w reads physical rows w, w+8, ...; lane = column i
    {
        const int li = tid & 31;
        const int64_t i = i0 + li;
        for (int lj = tid >> 5; lj < TJ; lj += 8) {
            const int64_t j = j0 + lj;
            float val = 0.0f;
            if (i < m && j < n) val = to_f32(x[j * ldx + i]);
            tile[lj * (TI + 1) + li] = val;
        }
    }
    __syncthreads();
    // partial amax over 16 rows: thread (p, i)
    for (int t = tid; t < kParts * TI; t += 256) {
        const int p = t / TI, li = t % TI;
        float a = 0.0f;
#pragma unroll
        for (int r = 0; r < 16; ++r) a = fmaxf(a, fabsf(tile[(p * 16 + r) * (TI + 1) + li]));
        part[p * TI + li] = a;
    }
    __syncthreads();
    // per (group, i): scale, factor; scale store
    const int64_t Gtot = (n + GRAN - 1) / GRAN;
    for (int t = tid; t < kGroups * TI; t += 256) {
        const int gl = t / TI, li = t % TI;
        float a = 0.0f;
#pragma unroll
        for (int p = 0; p < GRAN / 16; ++p) a = fmaxf(a, part[(gl * (GRAN / 16) + p) * TI + li]);
        float s, f;
        uint32_t ebyte;
        group_scale<FMT, RECIP>(a, s, f, ebyte);
        fac[gl * TI + li] = f;
        const int64_t i = i0 + li;
        const int64_t g = j0 / GRAN + gl;
        if constexpr (FMT != kSfPacked) {
            if (i < m && g < Gtot) static_cast<float*>(sf)[i * ssm + g * ssg] = s;
        } else {
            ebuf[gl * TI + li] = (g < Gtot) ? ebyte : 0u;
        }
    }
    __syncthreads();
    if constexpr (FMT == kSfPacked) {
        // kGroups is a multiple of 4: one word per 4 groups per column
        for (int t = tid; t < (kGroups / 4) * TI; t += 256) {
            const int wl = t / TI, li = t % TI;
            const int64_t i = i0 + li;
            const int64_t g = j0 / GRAN + wl * 4;
            uint32_t word = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) word |= ebuf[(wl * 4 + q) * TI + li] << (8 * q);
            if (i < m && g < Gtot) static_cast<int32_t*>(sf)[i * ssm + (g / 4) * ssg] = static_cast<int32_t>(word);
        }
    }
    // quantise + store: thread -> (i, 16-element segment of j)
    constexpr int kSegs = TJ / 16;
    for (int t = tid; t < TI * kSegs; t += 256) {
        const int li = t / kSegs, seg = t % kSegs;
        const int64_t i = i0 + li;
        const int64_t jb = j0 + seg * 16;
        if (i >= m || jb >= n) continue;
        const float f = fac[(seg * 16 / GRAN) * TI + li];
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float* c = tile + (seg * 16 + 4 * q) * (TI + 1) + li;
            w[q] = quant4(c[0], c[TI + 1], c[2 * (TI + 1)], c[3 * (TI + 1)], f);
        }
        uint8_t* orow = out + i * ldo;
        if (vec_out && jb + 16 <= n) {
            *reinterpret_cast<uint4*>(orow + jb) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            for (int e = 0; e < 16; ++e)
                if (jb + e < n) orow[jb + e] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
        }
    }
}

// ---------------------------------------------------------------------------
// Generic per-token cast: any strides. One thread per (row, run of four
// groups), so a packed int32 word is always written whole. Slow path.
// ---------------------------------------------------------------------------
template <typename T, int GRAN, int FMT, bool RECIP>
__global__ void __launch_bounds__(128) cast_generic_kernel(const T* __restrict__ x, int64_t m, int64_t n,
                                                           int64_t sxm, int64_t sxn, uint8_t* __restrict__ out,
                                                           int64_t som, int64_t son, void* __restrict__ sf,
                                                           int64_t ssm, int64_t ssg) {
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
            for (int64_t j = j0; j < j1; ++j) amax = fmaxf(amax, fabsf(to_f32(x[i * sxm + j * sxn])));
            float s, f;
            uint32_t ebyte;
            group_scale<FMT, RECIP>(amax, s, f, ebyte);
            for (int64_t j = j0; j < j1; ++j)
                out[i * som + j * son] =
                    static_cast<uint8_t>(e4m3x2(__fmul_rn(to_f32(x[i * sxm + j * sxn]), f), 0.0f) & 0xFFu);
            if constexpr (FMT != kSfPacked) static_cast<float*>(sf)[i * ssm + g * ssg] = s;
            word |= ebyte << (8 * q);
        }
        if constexpr (FMT == kSfPacked) static_cast<int32_t*>(sf)[i * ssm + w * ssg] = static_cast<int32_t>(word);
    }
}

// ---------------------------------------------------------------------------
// 128x128 block cast. One CTA (256 threads) per block; each thread holds 64
// elements in registers. Loads follow whichever input axis is contiguous; the
// E4M3 bytes are staged in shared memory and written along whichever output
// axis is contiguous, so W and W^T are produced by the same kernel.
// in_mode: 0 rows contiguous (vector), 1 columns contiguous (vector), 2 generic
// out_mode: 0 rows contiguous, 1 columns contiguous, 2 generic
// ---------------------------------------------------------------------------
template <typename T, int FMT, bool RECIP>
__global__ void __launch_bounds__(256) cast_block_kernel(const T* __restrict__ x, int64_t m, int64_t n,
                                                         int64_t sxm, int64_t sxn, int in_mode,
                                                         uint8_t* __restrict__ out, int64_t som, int64_t son,
                                                         int out_mode, void* __restrict__ sf, int64_t ssr,
                                                         int64_t ssc) {
    constexpr int B = 128, kPad = 16;
    __shared__ __align__(16) uint8_t q[B][B + kPad];
    __shared__ float red[8];
    const int tid = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * B;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * B;

    // element e (0..63) of this thread: (a, b) in block coordinates along the
    // (contiguous, strided) input axes: b = v*16 + tid/16, a = (tid%16)*8 + e%8
    float v[64];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int bb = it * 16 + tid / 16;
        const int a0 = (tid % 16) * 8;
        int64_t r, c;  // block-relative row/col of element a0
        if (in_mode == 1) { r = a0; c = bb; } else { r = bb; c = a0; }
        const int64_t gr = r0 + r, gc = c0 + c;
        if (in_mode == 0) {
            const T* p = x + gr * sxm + gc;
            if (gr < m && gc + 8 <= n) {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
                const T* t = reinterpret_cast<const T*>(&u);
                if constexpr (sizeof(T) == 2) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[it * 8 + e] = to_f32(t[e]);
                } else {
                    const uint4 u2 = __ldg(reinterpret_cast<const uint4*>(p) + 1);
                    const T* t2 = reinterpret_cast<const T*>(&u2);
#pragma unroll
                    for (int e = 0; e < 4; ++e) { v[it * 8 + e] = to_f32(t[e]); v[it * 8 + 4 + e] = to_f32(t2[e]); }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[it * 8 + e] = (gr < m && gc + e < n) ? to_f32(p[e]) : 0.0f;
            }
        } else if (in_mode == 1) {
            const T* p = x + gr + gc * sxn;
            if (gc < n && gr + 8 <= m) {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
                const T* t = reinterpret_cast<const T*>(&u);
                if constexpr (sizeof(T) == 2) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[it * 8 + e] = to_f32(t[e]);
                } else {
                    const uint4 u2 = __ldg(reinterpret_cast<const uint4*>(p) + 1);
                    const T* t2 = reinterpret_cast<const T*>(&u2);
#pragma unroll
                    for (int e = 0; e < 4; ++e) { v[it * 8 + e] = to_f32(t[e]); v[it * 8 + 4 + e] = to_f32(t2[e]); }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[it * 8 + e] = (gc < n && gr + e < m) ? to_f32(p[e]) : 0.0f;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[it * 8 + e] = (gr < m && gc + e < n) ? to_f32(x[gr * sxm + (gc + e) * sxn]) : 0.0f;
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 64; ++e) amax = fmaxf(amax, fabsf(v[e]));
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
            static_cast<float*>(sf)[br * ssr + bc * ssc] = s;
        } else {
            // packed along the column-block axis: block bc is byte bc % 4 of
            // word bc / 4; the last column block also zeroes the pad bytes
            uint8_t* word = reinterpret_cast<uint8_t*>(static_cast<int32_t*>(sf) + br * ssr + (bc / 4) * ssc);
            word[bc % 4] = static_cast<uint8_t>(ebyte);
            if (bc == static_cast<int64_t>(gridDim.x) - 1)
                for (int64_t z = bc % 4 + 1; z < 4; ++z) word[z] = 0;
        }
    }

    // quantise into shared memory, block-relative [row][col]
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int bb = it * 16 + tid / 16;
        const int a0 = (tid % 16) * 8;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint32_t w2 = e4m3x2(__fmul_rn(v[it * 8 + e], f), __fmul_rn(v[it * 8 + e + 1], f));
            if (in_mode == 1) {
                q[a0 + e][bb] = static_cast<uint8_t>(w2);
                q[a0 + e + 1][bb] = static_cast<uint8_t>(w2 >> 8);
            } else {
                q[bb][a0 + e] = static_cast<uint8_t>(w2);
                q[bb][a0 + e + 1] = static_cast<uint8_t>(w2 >> 8);
            }
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
            if (gc + 16 <= n) {
                *reinterpret_cast<uint4*>(o) = *reinterpret_cast<const uint4*>(&q[line][off]);
            } else {
                for (int e = 0; e < 16; ++e)
                    if (gc + e < n) o[e] = q[line][off + e];
            }
        } else if (out_mode == 1) {
            const int64_t gc = c0 + line, gr = r0 + off;
            if (gc >= n) continue;
            uint8_t* o = out + gr + gc * son;
            uint8_t b16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) b16[e] = q[off + e][line];
            if (gr + 16 <= m) {
                uint4 u;
                uint32_t* uw = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    uw[e] = b16[4 * e] | (b16[4 * e + 1] << 8) | (b16[4 * e + 2] << 16) | (static_cast<uint32_t>(b16[4 * e + 3]) << 24);
                *reinterpret_cast<uint4*>(o) = u;
            } else {
                for (int e = 0; e < 16; ++e)
                    if (gr + e < m) o[e] = b16[e];
            }
        } else {
            const int64_t gr = r0 + line, gc = c0 + off;
            if (gr >= m) continue;
            for (int e = 0; e < 16; ++e)
                if (gc + e < n) out[gr * som + (gc + e) * son] = q[line][off + e];
        }
    }
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T, int GRAN, int FMT, bool RECIP>
cudaError_t launch_token_t(const CastTokenArgs& a, cudaStream_t st, int num_sms) {
    const T* x = static_cast<const T*>(a.x);
    if (a.sxn == 1 && a.son == 1) {
        const int vec_in = aligned16(x) && ((a.sxm * static_cast<int64_t>(sizeof(T))) % 16 == 0);
        const int vec_out = aligned16(a.out) && (a.som % 16 == 0);
        const int64_t chunks = (a.n + 32 * (64 / sizeof(T)) - 1) / (32 * (64 / sizeof(T)));
        const int64_t warps = a.m * chunks;
        int64_t blocks = (warps + 7) / 8;
        const int64_t cap = static_cast<int64_t>(num_sms) * 8 * 4;   // enough warps for full-rate HBM
        if (blocks > cap) blocks = cap;
        cast_rows_kernel<T, GRAN, FMT, RECIP><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
            x, a.m, a.n, a.sxm, a.out, a.som, a.sf, a.ssm, a.ssg, chunks, vec_in, vec_out);
        return cudaGetLastError();
    }
    if (a.sxm == 1 && a.son == 1) {
        constexpr int TJ = (FMT == kSfPacked) ? ((4 * GRAN > 128) ? 4 * GRAN : 128) : 128;
        const size_t smem = (static_cast<size_t>(TJ) * 33 + (TJ / 16) * 32 + 2 * (TJ / GRAN) * 32) * sizeof(float);
        auto kern = cast_cols_kernel<T, GRAN, FMT, RECIP, TJ>;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        const int vec_out = aligned16(a.out) && (a.som % 16 == 0);
        dim3 grid(static_cast<unsigned>((a.m + 31) / 32), static_cast<unsigned>((a.n + TJ - 1) / TJ));
        kern<<<grid, 256, smem, st>>>(x, a.m, a.n, a.sxn, a.out, a.som, a.sf, a.ssm, a.ssg, vec_out);
        return cudaGetLastError();
    }
    const int64_t G = (a.n + GRAN - 1) / GRAN;
    const int64_t total = a.m * ((G + 3) / 4);
    int64_t blocks = (total + 127) / 128;
    if (blocks > static_cast<int64_t>(num_sms) * 16) blocks = static_cast<int64_t>(num_sms) * 16;
    if (blocks < 1) blocks = 1;
    cast_generic_kernel<T, GRAN, FMT, RECIP><<<static_cast<unsigned>(blocks), 128, 0, st>>>(
        x, a.m, a.n, a.sxm, a.sxn, a.out, a.som, a.son, a.sf, a.ssm, a.ssg);
    return cudaGetLastError();
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
    cast_block_kernel<T, FMT, RECIP><<<grid, 256, 0, st>>>(x, a.m, a.n, a.sxm, a.sxn, in_mode, a.out, a.som, a.son,
                                                          out_mode, a.sf, a.ssr, a.ssc);
    return cudaGetLastError();
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

}  // namespace ql
