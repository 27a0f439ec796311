// The host-buffer forward call for callers that cannot allocate device memory.
//
// ql_cast_gemm_host stages its row chunks in a device workspace the caller
// allocates. Some callers cannot make that allocation at the point of the
// call: a plug-in inside a host application whose device memory is all owned
// by the application's own pool, or a serving process that allows no new
// device allocation once it is warmed up so that its footprint stays fixed.
// ql_cast_gemm_host_noalloc stages the chunks in a fixed array compiled into
// this library instead, and otherwise runs the very same pipeline.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/qlinear.h"

namespace {

constexpr int kMaxDevices = 64;

// The staging area. Every GPU that loads the library holds these bytes until
// the process exits. In host code this name only stands in for the symbol:
// its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QL_NOALLOC_SCRATCH_BYTES];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the staging area on the current device, looked up once
// per device with that device current.
ql_status scratch_address(void*& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return QL_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    out = g_scratch_addr[dev];
    return QL_OK;
}

}  // namespace

extern "C" ql_status ql_cast_gemm_host_noalloc(const void* x_host, int64_t ldx, const uint8_t* b, int64_t ldb,
                                               const void* sfb, int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt,
                                               uint16_t* d_host, int64_t ldd, int64_t m, int64_t n, int64_t k,
                                               int64_t chunk_rows, ql_stream_t stream) {
    // the checks of ql_cast_gemm_host that come before any size, in its order
    if (m < 0 || n < 0 || k <= 0 || chunk_rows <= 0) return QL_ERR_INVALID_ARG;
    if (fmt < QL_SF_FP32 || fmt > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return QL_OK;
    const size_t need = ql_cast_gemm_host_workspace_size(n, k, chunk_rows, fmt);
    if (need == 0 || need > QL_NOALLOC_SCRATCH_BYTES) return QL_ERR_UNSUPPORTED;   // does not fit: fewer rows per chunk
    void* ws = nullptr;
    const ql_status st = scratch_address(ws);
    if (st != QL_OK) return st;
    return ql_cast_gemm_host(x_host, ldx, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, d_host, ldd, m, n, k,
                             chunk_rows, ws, QL_NOALLOC_SCRATCH_BYTES, stream);
}
