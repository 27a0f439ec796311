// Launch arguments of the block-scaled GEMM (validated by the C ABI layer).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

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
                              // 3 = block-scaled MMA on CTA pairs (UE8M0 formats only)
    uint32_t* dev_status;
    uint64_t wait_limit_ns;
    int stall_producer;
};

int choose_block_n(int64_t m, int64_t n, int num_sms);
cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t st, int num_sms);
cudaError_t launch_gemm_mx(const GemmLaunch& L, const GemmParams& p, int bn, cudaStream_t st, int num_sms);
cudaError_t launch_gemm_mx2(const GemmLaunch& L, const GemmParams& p, cudaStream_t st, int num_sms);

// 2-D uint8 tensor map [rows, cols] (cols contiguous, row stride ld bytes),
// box [box_rows x 128 bytes], 128-byte swizzle, zero fill out of bounds.
bool encode_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows);

// 2-D tensor map of `rows` rows of `cols` elements (row stride in bytes), box
// [box_rows x box_cols] elements, no swizzle, zero fill out of bounds.
bool encode_2d_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int64_t rows, int64_t cols,
                   int64_t row_stride_bytes, int box_rows, int box_cols);

}  // namespace ql
