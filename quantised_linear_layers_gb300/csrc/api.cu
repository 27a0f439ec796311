// C ABI of libqlinear.so (declared in include/qlinear.h): host-side argument
// validation, kernel selection and launch on the caller's stream. No call
// synchronises the host except ql_device_status().
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/qlinear.h"
#include "cast.cuh"
#include "gemm.cuh"

namespace {

constexpr int kMaxDevices = 64;

// Device status word (time-out flags raised by kernels). One copy per device
// that loads the library; its address is looked up once per device.
__device__ uint32_t g_dev_status = 0;

std::atomic<int> g_num_sms_override{0};
std::atomic<int> g_block_n_override{0};
std::atomic<int> g_gemm_path{0};
std::atomic<int> g_stall_producer{0};
std::atomic<int> g_wait_limit_ms{2000};

struct DeviceInfo {
    int num_sms = 0;
    uint32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

ql_status device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.num_sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return QL_ERR_CUDA;
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_dev_status) != cudaSuccess || addr == nullptr) return QL_ERR_CUDA;
        d.status = static_cast<uint32_t*>(addr);
        d.num_sms = sms;
    }
    out = d;
    return QL_OK;
}

int effective_sms(const DeviceInfo& d) {
    const int o = g_num_sms_override.load();
    return (o > 0 && o < d.num_sms) ? o : d.num_sms;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ql_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return QL_OK;
    if (e == cudaErrorInvalidValue) return QL_ERR_INVALID_ARG;
    return QL_ERR_CUDA;
}

ql_status gemm_common(const uint8_t* a, int64_t lda, const void* sfa, int64_t sam, int64_t sak, const uint8_t* b,
                      int64_t ldb, const void* sfb, int64_t sbn, int64_t sbk, int fmt, void* d, int64_t ldd,
                      int64_t m, int64_t n, int64_t k, bool wgrad, int accumulate, cudaStream_t st,
                      const int32_t* m_indices = nullptr, int num_groups = 1, int64_t sbg = 0,
                      const ql::GemmLaunch* fp8out = nullptr, bool a_mn = false, bool b_mn = false) {
    if (m < 0 || n < 0 || k < 0) return QL_ERR_INVALID_ARG;
    if (fmt < QL_SF_FP32 || fmt > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (m >= (int64_t(1) << 31) || n >= (int64_t(1) << 31) || k >= (int64_t(1) << 31)) return QL_ERR_UNSUPPORTED;
    if (m == 0 || n == 0) return QL_OK;
    if (d == nullptr || ldd < n) return QL_ERR_INVALID_ARG;
    const size_t es = wgrad ? 4 : 2;
    if (k == 0 && fp8out != nullptr) return QL_ERR_UNSUPPORTED;
    if (k == 0) {
        if (wgrad && accumulate) return QL_OK;
        return from_cuda(cudaMemset2DAsync(d, static_cast<size_t>(ldd) * es, 0, static_cast<size_t>(n) * es,
                                           static_cast<size_t>(m), st));
    }
    if (a == nullptr || b == nullptr || sfa == nullptr || sfb == nullptr) return QL_ERR_INVALID_ARG;
    // a K-major operand has rows of k bytes; an MN-major one rows of m (or n) bytes
    if (lda < (a_mn ? m : k) || ldb < (b_mn ? n : k)) return QL_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || lda % 16 != 0 || ldb % 16 != 0) return QL_ERR_ALIGNMENT;
    DeviceInfo di;
    ql_status s = device_info(di);
    if (s != QL_OK) return s;
    ql::GemmLaunch L{};
    L.a = a;
    L.lda = lda;
    L.b = b;
    L.ldb = ldb;
    L.m = m;
    L.n = n;
    L.k = k;
    L.sfa = sfa;
    L.sam = sam;
    L.sak = sak;
    L.sfb = sfb;
    L.sbn = sbn;
    L.sbk = sbk;
    L.fmt = fmt;
    L.per_row_b = wgrad;
    L.out_f32 = wgrad;
    L.d = d;
    L.ldd = ldd;
    L.accumulate = accumulate ? 1 : 0;
    L.block_n = g_block_n_override.load();
    L.path = g_gemm_path.load();
    L.stall_producer = g_stall_producer.load();
    L.dev_status = di.status;
    L.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ms.load()) * 1000000ull;
    L.m_indices = m_indices;
    L.num_groups = num_groups;
    L.sbg = sbg;
    L.a_mn = a_mn;
    L.b_mn = b_mn;
    if (fp8out != nullptr) {
        L.out_fp8 = true;
        L.dsf = fp8out->dsf;
        L.dsm = fp8out->dsm;
        L.dsg = fp8out->dsg;
        L.dgran = fp8out->dgran;
        L.dfmt = fp8out->dfmt;
        L.drecip = fp8out->drecip;
    }
    return from_cuda(ql::launch_gemm(L, st, effective_sms(di)));
}

}  // namespace

extern "C" {

const char* ql_status_string(ql_status s) {
    switch (s) {
        case QL_OK: return "QL_OK";
        case QL_ERR_INVALID_ARG: return "QL_ERR_INVALID_ARG: invalid argument";
        case QL_ERR_UNSUPPORTED: return "QL_ERR_UNSUPPORTED: unsupported request";
        case QL_ERR_ALIGNMENT: return "QL_ERR_ALIGNMENT: pointer or stride alignment not met";
        case QL_ERR_CUDA: return "QL_ERR_CUDA: CUDA runtime error";
        case QL_ERR_DEVICE_TIMEOUT: return "QL_ERR_DEVICE_TIMEOUT: a kernel wait ran out of time";
    }
    return "unknown ql_status";
}

ql_status fp8_cast_per_token(const void* x, ql_dtype x_dtype, int64_t m, int64_t n, int64_t x_stride_m,
                             int64_t x_stride_n, int gran_k, int fmt, uint8_t* out, int64_t out_stride_m,
                             int64_t out_stride_n, void* out_sf, int64_t sf_stride_m, int64_t sf_stride_g,
                             ql_stream_t stream) {
    if (m < 0 || n < 0) return QL_ERR_INVALID_ARG;
    if (x_dtype != QL_BF16 && x_dtype != QL_F32) return QL_ERR_INVALID_ARG;
    if (gran_k != 32 && gran_k != 128) return QL_ERR_INVALID_ARG;
    const bool recip = (fmt & QL_CAST_RECIP_OF_SCALE) != 0;
    const int base = fmt & ~QL_CAST_RECIP_OF_SCALE;
    if (base < QL_SF_FP32 || base > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (recip && base != QL_SF_FP32) return QL_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return QL_OK;
    if (x == nullptr || out == nullptr || out_sf == nullptr) return QL_ERR_INVALID_ARG;
    DeviceInfo di;
    ql_status s = device_info(di);
    if (s != QL_OK) return s;
    ql::CastTokenArgs a{};
    a.x = x;
    a.is_bf16 = x_dtype == QL_BF16;
    a.m = m;
    a.n = n;
    a.sxm = x_stride_m;
    a.sxn = x_stride_n;
    a.gran = gran_k;
    a.fmt = base;
    a.recip = recip;
    a.out = out;
    a.som = out_stride_m;
    a.son = out_stride_n;
    a.sf = out_sf;
    a.ssm = sf_stride_m;
    a.ssg = sf_stride_g;
    const int64_t es = x_dtype == QL_BF16 ? 2 : 4;
    a.tma_ok = aligned16(x) && x_stride_n > 0 && (x_stride_n * es) % 16 == 0 && x_stride_n * es < (int64_t(1) << 40) &&
               m < (int64_t(1) << 31) && n < (int64_t(1) << 31);
    a.dev_status = di.status;
    a.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ms.load()) * 1000000ull;
    return from_cuda(ql::launch_cast_per_token(a, reinterpret_cast<cudaStream_t>(stream), di.num_sms));
}

ql_status fp8_cast_per_block(const void* x, ql_dtype x_dtype, int64_t m, int64_t n, int64_t x_stride_m,
                             int64_t x_stride_n, int fmt, uint8_t* out, int64_t out_stride_m, int64_t out_stride_n,
                             void* out_sf, int64_t sf_stride_r, int64_t sf_stride_c, ql_stream_t stream) {
    if (m < 0 || n < 0) return QL_ERR_INVALID_ARG;
    if (x_dtype != QL_BF16 && x_dtype != QL_F32) return QL_ERR_INVALID_ARG;
    const bool recip = (fmt & QL_CAST_RECIP_OF_SCALE) != 0;
    const int base = fmt & ~QL_CAST_RECIP_OF_SCALE;
    if (base < QL_SF_FP32 || base > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (recip && base != QL_SF_FP32) return QL_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return QL_OK;
    if (x == nullptr || out == nullptr || out_sf == nullptr) return QL_ERR_INVALID_ARG;
    if ((m + 127) / 128 > 65535) return QL_ERR_UNSUPPORTED;
    ql::CastBlockArgs a{};
    a.x = x;
    a.is_bf16 = x_dtype == QL_BF16;
    a.m = m;
    a.n = n;
    a.sxm = x_stride_m;
    a.sxn = x_stride_n;
    a.fmt = base;
    a.recip = recip;
    a.out = out;
    a.som = out_stride_m;
    a.son = out_stride_n;
    a.sf = out_sf;
    a.ssr = sf_stride_r;
    a.ssc = sf_stride_c;
    return from_cuda(ql::launch_cast_per_block(a, reinterpret_cast<cudaStream_t>(stream)));
}

ql_status gemm_fp8_nt_bf16(const uint8_t* a, int64_t lda, const void* sfa, int64_t sfa_stride_m,
                           int64_t sfa_stride_k, const uint8_t* b, int64_t ldb, const void* sfb,
                           int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt, uint16_t* d, int64_t ldd,
                           int64_t m, int64_t n, int64_t k, void* workspace, size_t ws_bytes, ql_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    return gemm_common(a, lda, sfa, sfa_stride_m, sfa_stride_k, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, d, ldd,
                       m, n, k, false, 0, reinterpret_cast<cudaStream_t>(stream));
}

ql_status gemm_fp8_wgrad_fp32(const uint8_t* a, int64_t lda, const void* sfa, int64_t sfa_stride_m,
                              int64_t sfa_stride_k, const uint8_t* b, int64_t ldb, const void* sfb,
                              int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt, float* d, int64_t ldd,
                              int64_t m, int64_t n, int64_t k, int accumulate, void* workspace, size_t ws_bytes,
                              ql_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    return gemm_common(a, lda, sfa, sfa_stride_m, sfa_stride_k, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, d, ldd,
                       m, n, k, true, accumulate, reinterpret_cast<cudaStream_t>(stream));
}

ql_status m_grouped_gemm_fp8_nt_bf16_contiguous(const uint8_t* a, int64_t lda, const void* sfa,
                                                int64_t sfa_stride_m, int64_t sfa_stride_k, const uint8_t* b,
                                                int64_t ldb, const void* sfb, int64_t sfb_stride_g,
                                                int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt, uint16_t* d,
                                                int64_t ldd, const int32_t* m_indices, int num_groups, int64_t m,
                                                int64_t n, int64_t k, ql_stream_t stream) {
    if (m < 0 || n < 0 || k < 0 || num_groups < 1) return QL_ERR_INVALID_ARG;
    if (m % ql::kGroupAlignM != 0) return QL_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_groups) * n >= (int64_t(1) << 31)) return QL_ERR_UNSUPPORTED;
    if (m == 0 || n == 0) return QL_OK;
    if (m_indices == nullptr) return QL_ERR_INVALID_ARG;
    // k == 0 would make every expert row zero while leaving padding rows
    // untouched; that needs the indices on the host, so it is refused.
    if (k == 0) return QL_ERR_UNSUPPORTED;
    return gemm_common(a, lda, sfa, sfa_stride_m, sfa_stride_k, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, d, ldd,
                       m, n, k, false, 0, reinterpret_cast<cudaStream_t>(stream), m_indices, num_groups,
                       sfb_stride_g);
}

int ql_get_m_alignment_for_contiguous_layout(void) { return ql::kGroupAlignM; }

ql_status gemm_fp8_wgrad_fp32_mn(const uint8_t* a, int64_t lda, const void* sfa, int64_t sfa_stride_m,
                                 int64_t sfa_stride_k, const uint8_t* b, int64_t ldb, const void* sfb,
                                 int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt, float* d, int64_t ldd,
                                 int64_t m, int64_t n, int64_t k, int accumulate, ql_stream_t stream) {
    return gemm_common(a, lda, sfa, sfa_stride_m, sfa_stride_k, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, d, ldd,
                       m, n, k, true, accumulate, reinterpret_cast<cudaStream_t>(stream), nullptr, 1, 0, nullptr,
                       true, true);
}

ql_status gemm_fp8_nn_bf16(const uint8_t* a, int64_t lda, const void* sfa, int64_t sfa_stride_m,
                           int64_t sfa_stride_k, const uint8_t* b, int64_t ldb, const void* sfb,
                           int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt, uint16_t* d, int64_t ldd, int64_t m,
                           int64_t n, int64_t k, ql_stream_t stream) {
    return gemm_common(a, lda, sfa, sfa_stride_m, sfa_stride_k, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, d, ldd,
                       m, n, k, false, 0, reinterpret_cast<cudaStream_t>(stream), nullptr, 1, 0, nullptr, false,
                       true);
}

ql_status gemm_fp8_nt_fp8out(const uint8_t* a, int64_t lda, const void* sfa, int64_t sfa_stride_m,
                             int64_t sfa_stride_k, const uint8_t* b, int64_t ldb, const void* sfb,
                             int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt, uint8_t* d, int64_t ldd,
                             void* d_sf, int64_t d_sf_stride_m, int64_t d_sf_stride_g, int d_gran_k, int d_fmt,
                             int64_t m, int64_t n, int64_t k, ql_stream_t stream) {
    if (d_gran_k != 32 && d_gran_k != 128) return QL_ERR_INVALID_ARG;
    const bool recip = (d_fmt & QL_CAST_RECIP_OF_SCALE) != 0;
    const int base = d_fmt & ~QL_CAST_RECIP_OF_SCALE;
    if (base < QL_SF_FP32 || base > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (recip && base != QL_SF_FP32) return QL_ERR_INVALID_ARG;
    if (m > 0 && n > 0 && d_sf == nullptr) return QL_ERR_INVALID_ARG;
    ql::GemmLaunch o{};
    o.dsf = d_sf;
    o.dsm = d_sf_stride_m;
    o.dsg = d_sf_stride_g;
    o.dgran = d_gran_k;
    o.dfmt = base;
    o.drecip = recip ? 1 : 0;
    return gemm_common(a, lda, sfa, sfa_stride_m, sfa_stride_k, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, d, ldd,
                       m, n, k, false, 0, reinterpret_cast<cudaStream_t>(stream), nullptr, 1, 0, &o);
}

size_t ql_gemm_workspace_size(int64_t m, int64_t n, int64_t k) {
    (void)m;
    (void)n;
    (void)k;
    return 0;
}

ql_status ql_set_num_sms(int num_sms) {
    g_num_sms_override.store(num_sms > 0 ? num_sms : 0);
    return QL_OK;
}

int ql_get_num_sms(void) {
    DeviceInfo di;
    if (device_info(di) != QL_OK) return 0;
    return effective_sms(di);
}

ql_status ql_set_wait_limit_ms(int ms) {
    if (ms <= 0) return QL_ERR_INVALID_ARG;
    g_wait_limit_ms.store(ms);
    return QL_OK;
}

ql_status ql_set_gemm_block_n(int block_n) {
    if (block_n != 0 && block_n != 32 && block_n != 64 && block_n != 128 && block_n != 256)
        return QL_ERR_INVALID_ARG;
    g_block_n_override.store(block_n);
    return QL_OK;
}

ql_status ql_set_gemm_path(int path) {
    if (path < 0 || path > 4) return QL_ERR_INVALID_ARG;
    g_gemm_path.store(path);
    return QL_OK;
}

ql_status ql_test_stall_gemm_producer(int enable) {
    g_stall_producer.store(enable ? 1 : 0);
    return QL_OK;
}

ql_status ql_device_status(ql_stream_t stream) {
    DeviceInfo di;
    ql_status s = device_info(di);
    if (s != QL_OK) return s;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QL_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, di.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QL_ERR_CUDA;
    if (v != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(di.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return QL_ERR_CUDA;
        return (v & ql::kDevErrTimeout) ? QL_ERR_DEVICE_TIMEOUT : QL_ERR_INVALID_ARG;
    }
    return QL_OK;
}

}  // extern "C"
