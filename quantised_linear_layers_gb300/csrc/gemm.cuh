// Launch arguments of the block-scaled GEMM (validated by the C ABI layer).
#pragma once
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
    uint32_t* dev_status;
    uint64_t wait_limit_ns;
};

int choose_block_n(int64_t m, int64_t n, int num_sms);
cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t st, int num_sms);

}  // namespace ql
