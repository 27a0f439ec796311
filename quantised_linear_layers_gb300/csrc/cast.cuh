// Launch arguments of the cast kernels (validated by the C ABI layer).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace ql {

struct CastTokenArgs {
    const void* x;
    bool is_bf16;
    int64_t m, n, sxm, sxn;
    int gran;      // 32 | 128
    int fmt;       // 0 fp32, 1 UE8M0 (fp32 storage), 2 packed UE8M0
    bool recip;    // factor = 1 / scale (fp32 format only)
    uint8_t* out;
    int64_t som, son;
    void* sf;
    int64_t ssm, ssg;
    bool tma_ok;            // the transposed view may be read with TMA
    uint32_t* dev_status;   // time-out flags of the TMA-staged kernel; bounds violations
    uint64_t wait_limit_ns;
};

struct CastBlockArgs {
    const void* x;
    bool is_bf16;
    int64_t m, n, sxm, sxn;
    int fmt;       // 0 fp32, 1 UE8M0 (fp32 storage), 2 packed UE8M0 (along column blocks)
    bool recip;
    uint8_t* out;
    int64_t som, son;
    void* sf;
    int64_t ssr, ssc;
    // optional second scale grid, of the transposed block layout (nullptr: none):
    // block (r, c) at [c*sst_c + r*sst_r], packed along r for packed UE8M0
    void* sf_t;
    int64_t sst_c, sst_r;
    uint32_t* dev_status;   // bounds-checked builds record violations here
};

// Per-token cast of x and of x^T from one read (1 x 128 groups both ways).
struct CastDualArgs {
    const void* x;
    bool is_bf16;
    int64_t m, n, sxm;          // x [m, n], rows contiguous
    int fmt;
    bool recip;
    uint8_t* qr;                // cast of x: [m, n], row stride ldr
    int64_t ldr;
    void* sfr;                  // its scales [m, ceil(n/128)] at (srm, srg)
    int64_t srm, srg;
    uint8_t* qc;                // cast of x^T, in x's layout: [m, n], row stride ldc
    int64_t ldc;
    void* sfc;                  // its scales [n, ceil(m/128)] at (scn, scg)
    int64_t scn, scg;
    uint32_t* dev_status;       // bounds-checked builds record violations here
};

cudaError_t launch_cast_per_token(const CastTokenArgs& a, cudaStream_t st, int num_sms);
cudaError_t launch_cast_dual(const CastDualArgs& a, cudaStream_t st);
cudaError_t launch_cast_per_block(const CastBlockArgs& a, cudaStream_t st);

}  // namespace ql
