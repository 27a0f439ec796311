// Launch arguments of the block-scaled GEMM (validated by the C ABI layer).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"

namespace ql {

// Kernel parameters (passed by value).
struct GemmParams {
    int64_t m, n;
    int num_kb;               // ceil(k / 128)
    int tiles_m, tiles_n, group_m;
    const void* sfa;
    int64_t sam, sak;
    const void* sfb;
    int64_t sbn, sbk;
    int fmt;                  // 0/1: fp32 values, 2: packed UE8M0 words
    void* d;
    int64_t ldd;
    int accumulate;           // fp32 output only
    int vec_store;            // 16-byte output stores allowed
    uint32_t* dev_status;
    uint64_t wait_limit_ns;
    int stall_producer;       // test hook: the producer issues no copies (waits time out)
    // M-grouped contiguous layout: expert index per row of A (nullptr: one B)
    const int* m_indices;
    int num_groups;
    int64_t b_group_rows;     // rows of B per expert (n) in B's tensor map
    int64_t sbg;              // sfb elements (or packed words) between experts
    // E4M3 output with per-token scales (the GEMM kernels' OUT_FP8 form)
    void* dsf;
    int64_t dsm, dsg;
    int dgran;                // 32 or 128
    int dfmt;                 // 0 fp32, 1 UE8M0 (fp32 powers of two), 2 packed UE8M0
    int drecip;               // fp32 scales: factor 1 / s
    // operands stored K-outer ([K][M] / [K][N]) and read MN-major
    int a_mn, b_mn;
    // fp32 output written (or added) through the kernel's D tensor map
    int tma_d;
    // byte ranges of sfa, sfb, D, D's scales and m_indices, checked in
    // bounds-checked builds (status: dev_status)
    Bounds bnd;
};

// Host-side description of one GEMM call.
struct GemmLaunch {
    const uint8_t* a;
    int64_t lda;
    const uint8_t* b;
    int64_t ldb;
    int64_t m, n, k;
    const void* sfa;
    int64_t sam, sak;
    const void* sfb;
    int64_t sbn, sbk;
    int fmt;
    bool per_row_b;           // wgrad: one B scale per row
    bool out_f32;             // wgrad: fp32 output
    void* d;
    int64_t ldd;
    int accumulate;
    int block_n;              // 0 = heuristic, else 32/64/128/256
    int path;                 // 0 = auto, 1 = CUDA-core promotion, 2 = block-scaled MMA on one SM,
                              // 3 = block-scaled MMA on CTA pairs, 4 = split-K over a cluster
                              // (3 and 4: UE8M0 formats only), 5 = CUDA-core promotion on
                              // CTA pairs, 6 = CUDA-core promotion on one SM, 7 = CUDA-core
                              // promotion split-K over a cluster
    uint32_t* dev_status;
    uint64_t wait_limit_ns;
    int stall_producer;
    const int* m_indices;     // M-grouped contiguous layout (nullptr: plain GEMM)
    int num_groups;
    int64_t sbg;
    bool out_fp8;             // E4M3 output + per-token scales (fwd form only)
    void* dsf;
    int64_t dsm, dsg;
    int dgran, dfmt, drecip;
    bool a_mn, b_mn;          // A stored [k][m] / B stored [k][n] (row strides lda / ldb)
};

// Rows of A per M tile; in the M-grouped contiguous layout every expert's
// segment starts on a multiple of it.
constexpr int kGroupAlignM = 128;

#ifdef __CUDACC__
// Expert of M tile `mb` in the M-grouped contiguous layout (0 for a plain
// GEMM), read from the tile's first row. Returns -1 when the tile is padding
// (index -1) and when the index lies outside [-1, num_groups): such a tile is
// skipped by every role of the CTA; the caller passing report = true records a
// bad index in the device status word.
__device__ __forceinline__ int tile_expert(const GemmParams& p, int mb, bool report) {
    if (p.m_indices == nullptr) return 0;
    const int* ip = p.m_indices + static_cast<int64_t>(mb) * kGroupAlignM;
    const int e = QL_IN(p.bnd, 4, ip, 4) ? __ldg(ip) : -1;
    if (e < -1 || e >= p.num_groups) {
        if (report) atomicOr(p.dev_status, kDevErrBadIndex);
        return -1;
    }
    return e;
}

// Whether the epilogue thread owning `row` of a tile of expert `e` stores it:
// padding rows (-1) are left untouched; a row of another expert (a segment
// not starting on the alignment) is not stored and is recorded as a bad index.
__device__ __forceinline__ bool row_in_expert(const GemmParams& p, int64_t row, int e) {
    if (p.m_indices == nullptr) return true;
    const int r = QL_IN(p.bnd, 4, p.m_indices + row, 4) ? __ldg(p.m_indices + row) : -1;
    if (r == e) return true;
    if (r != -1) atomicOr(p.dev_status, kDevErrBadIndex);
    return false;
}

// The same decision without recording (for the other threads of the row).
__device__ __forceinline__ bool row_in_expert_quiet(const GemmParams& p, int64_t row, int e) {
    return p.m_indices == nullptr || (QL_IN(p.bnd, 4, p.m_indices + row, 4) && __ldg(p.m_indices + row) == e);
}
#endif

// Launch of a GEMM kernel (384 threads; its tensor maps and the parameters)
// with programmatic stream serialization, so its prologue and the L2
// prefetch of its first weight tiles overlap the previous kernel's tail; the
// kernel waits for the previous kernel before it reads any input. `cluster`
// > 1 adds a cluster dimension.
template <typename Kern, typename... Args>
inline cudaError_t launch_gemm_kernel(Kern kern, unsigned grid, unsigned cluster, size_t smem, cudaStream_t st,
                                      const Args&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(384, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

int choose_block_n(int64_t m, int64_t n, int num_sms);
cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t st, int num_sms);
cudaError_t launch_gemm_mx(const GemmLaunch& L, const GemmParams& p, int bn, cudaStream_t st, int num_sms);
cudaError_t launch_gemm_mx2(const GemmLaunch& L, const GemmParams& p, cudaStream_t st, int num_sms);
// CUDA-core promotion (any fp32 scales) on CTA pairs, 256 x 256 tiles; plain
// GEMMs with bf16 output or fp32 (wgrad) output, K- or MN-major operands.
cudaError_t launch_gemm_pair(const GemmLaunch& L, const GemmParams& p, cudaStream_t st, int num_sms);
// Split-K over a thread-block cluster (bf16 output, UE8M0 formats): cluster
// size for the shape (1 = no split applies) and the launch.
int choose_split_k(int64_t m, int64_t n, int64_t k, int num_sms);
cudaError_t launch_gemm_mx_sk(const GemmLaunch& L, GemmParams p, int split, cudaStream_t st);
// Split-K over a cluster with CUDA-core promotion (any fp32 scales): K-major
// operands, bf16 output, plain GEMM; split 2 or 4.
cudaError_t launch_gemm_prom_sk(const GemmLaunch& L, GemmParams p, int split, cudaStream_t st);

// Raises `kern`'s dynamic shared-memory limit to `bytes` on the current device,
// once per (kernel, device): the attribute is per device. Thread-safe.
cudaError_t ensure_smem_attr(const void* kern, int bytes);
// The number of clusters of `cfg`'s shape that can be resident at once for
// `kern` on the current device (at least 1), computed once per (kernel,
// device). Thread-safe.
int max_active_clusters(const void* kern, const cudaLaunchConfig_t& cfg);

// 2-D uint8 tensor map [rows, cols] (cols contiguous, row stride ld bytes),
// box [box_rows x 128 bytes], 128-byte swizzle, zero fill out of bounds.
bool encode_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows);

// 2-D tensor map of `rows` rows of `cols` elements (row stride in bytes), box
// [box_rows x box_cols] elements, zero fill out of bounds; `swizzle` 0 (none),
// 64 or 128 selects the 64- or 128-byte swizzle (box_cols x element size must
// then equal it).
bool encode_2d_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int64_t rows, int64_t cols,
                   int64_t row_stride_bytes, int box_rows, int box_cols, int swizzle = 0);

}  // namespace ql
