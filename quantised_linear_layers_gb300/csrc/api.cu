// C ABI of libqlinear.so (declared in include/qlinear.h): host-side argument
// validation, kernel selection and launch on the caller's stream. No call
// synchronises the host except ql_device_status().
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/qlinear.h"
#include "bounds.cuh"
#include "cast.cuh"
#include "gemm.cuh"

namespace {

constexpr int kMaxDevices = 64;

// Device status words: [0] flags raised by kernels (time-out, invalid grouped
// index, out-of-bounds access in bounds-checked builds), [2..3] the first
// out-of-bounds address as a 64-bit word. One copy per device that loads the
// library; its address is looked up once per device.
__device__ __align__(16) uint32_t g_dev_status[4] = {0u, 0u, 0u, 0u};

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

// ---------------------------------------------------------------------------
// Host-buffer forward pipeline (ql_cast_gemm_host): rows of X are copied to
// the device, cast and multiplied chunk by chunk, and D comes back, with the
// copy in, the kernels and the copy out of successive chunks overlapped on
// three streams. The streams and events are created once per device and kept.
// ---------------------------------------------------------------------------
constexpr int kPipeSlots = 2;

struct Pipe {
    std::atomic<bool> ready{false};   // published only after every stream and event exists
    std::mutex init_mu;               // serialises the one-time set-up
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kPipeSlots] = {}, comp_done[kPipeSlots] = {}, out_done[kPipeSlots] = {};
    std::mutex mu;                    // one call at a time runs the pipeline
};
Pipe g_pipe[kMaxDevices];

// Destroys whatever a failed set-up created, so that the next call retries.
void pipe_destroy(Pipe& p) {
    cudaEvent_t* evs[] = {&p.start, &p.end};
    for (cudaEvent_t* e : evs)
        if (*e) { cudaEventDestroy(*e); *e = nullptr; }
    for (int i = 0; i < kPipeSlots; ++i) {
        cudaEvent_t* slot[] = {&p.in_done[i], &p.comp_done[i], &p.out_done[i]};
        for (cudaEvent_t* e : slot)
            if (*e) { cudaEventDestroy(*e); *e = nullptr; }
    }
    cudaStream_t* sts[] = {&p.in, &p.comp, &p.out};
    for (cudaStream_t* s : sts)
        if (*s) { cudaStreamDestroy(*s); *s = nullptr; }
}

// The current device's pipeline; its streams and events are created by the
// first call on the device, under a lock, and published once all exist.
ql_status pipe_for_device(Pipe*& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QL_ERR_CUDA;
    Pipe& p = g_pipe[dev];
    if (!p.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(p.init_mu);
        if (!p.ready.load(std::memory_order_relaxed)) {
            const unsigned fl = cudaEventDisableTiming;
            bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
                      cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) == cudaSuccess &&
                      cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
                      cudaEventCreateWithFlags(&p.start, fl) == cudaSuccess &&
                      cudaEventCreateWithFlags(&p.end, fl) == cudaSuccess;
            for (int i = 0; ok && i < kPipeSlots; ++i)
                ok = cudaEventCreateWithFlags(&p.in_done[i], fl) == cudaSuccess &&
                     cudaEventCreateWithFlags(&p.comp_done[i], fl) == cudaSuccess &&
                     cudaEventCreateWithFlags(&p.out_done[i], fl) == cudaSuccess;
            if (!ok) {
                pipe_destroy(p);
                return QL_ERR_CUDA;
            }
            p.ready.store(true, std::memory_order_release);
        }
    }
    out = &p;
    return QL_OK;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Byte sizes of one slot's buffers: X rows (bf16), their E4M3 cast (rows of
// ldq bytes), the M-major scales, and D rows (bf16).
struct SlotLayout {
    size_t x, q, s, d, total;
    int64_t ldq, sld, scols;
};

SlotLayout slot_layout(int64_t n, int64_t k, int64_t rows, int fmt) {
    SlotLayout L{};
    L.ldq = (k + 15) / 16 * 16;
    const int64_t g = (k + 127) / 128;
    L.scols = (fmt == QL_SF_PACKED_UE8M0) ? (g + 3) / 4 : g;
    L.sld = (rows + 3) / 4 * 4;
    L.x = align256(static_cast<size_t>(rows) * k * 2);
    L.q = align256(static_cast<size_t>(rows) * L.ldq);
    L.s = align256(static_cast<size_t>(L.scols) * L.sld * 4);
    L.d = align256(static_cast<size_t>(rows) * n * 2);
    L.total = L.x + L.q + L.s + L.d;
    return L;
}

// Never launched: its attributes tell which binary the runtime loaded for
// this library's kernels.
__global__ void ql_probe_kernel() {}

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
        case QL_ERR_OUT_OF_BOUNDS: return "QL_ERR_OUT_OF_BOUNDS: a bounds-checked build skipped an out-of-range access";
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

static ql_status cast_per_block_common(const void* x, ql_dtype x_dtype, int64_t m, int64_t n,
                                       int64_t x_stride_m, int64_t x_stride_n, int fmt, uint8_t* out,
                                       int64_t out_stride_m, int64_t out_stride_n, void* out_sf,
                                       int64_t sf_stride_r, int64_t sf_stride_c, void* out_sf_t,
                                       int64_t sf_t_stride_c, int64_t sf_t_stride_r, bool dual,
                                       ql_stream_t stream) {
    if (m < 0 || n < 0) return QL_ERR_INVALID_ARG;
    if (x_dtype != QL_BF16 && x_dtype != QL_F32) return QL_ERR_INVALID_ARG;
    const bool recip = (fmt & QL_CAST_RECIP_OF_SCALE) != 0;
    const int base = fmt & ~QL_CAST_RECIP_OF_SCALE;
    if (base < QL_SF_FP32 || base > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (recip && base != QL_SF_FP32) return QL_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return QL_OK;
    if (x == nullptr || out == nullptr || out_sf == nullptr) return QL_ERR_INVALID_ARG;
    if (dual && out_sf_t == nullptr) return QL_ERR_INVALID_ARG;
    if ((m + 127) / 128 > 65535) return QL_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (ql_status s = device_info(di); s != QL_OK) return s;
    ql::CastBlockArgs a{};
    a.dev_status = di.status;
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
    a.sf_t = dual ? out_sf_t : nullptr;
    a.sst_c = sf_t_stride_c;
    a.sst_r = sf_t_stride_r;
    return from_cuda(ql::launch_cast_per_block(a, reinterpret_cast<cudaStream_t>(stream)));
}

ql_status fp8_cast_per_token_dual(const void* x, ql_dtype x_dtype, int64_t m, int64_t n, int64_t x_stride_m,
                                  int fmt, uint8_t* out_rows, int64_t out_rows_stride_m, void* sf_rows,
                                  int64_t sf_rows_stride_m, int64_t sf_rows_stride_g, uint8_t* out_cols,
                                  int64_t out_cols_stride_m, void* sf_cols, int64_t sf_cols_stride_n,
                                  int64_t sf_cols_stride_g, ql_stream_t stream) {
    if (m < 0 || n < 0) return QL_ERR_INVALID_ARG;
    if (x_dtype != QL_BF16 && x_dtype != QL_F32) return QL_ERR_INVALID_ARG;
    const bool recip = (fmt & QL_CAST_RECIP_OF_SCALE) != 0;
    const int base = fmt & ~QL_CAST_RECIP_OF_SCALE;
    if (base < QL_SF_FP32 || base > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (recip && base != QL_SF_FP32) return QL_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return QL_OK;
    if (x == nullptr || out_rows == nullptr || sf_rows == nullptr || out_cols == nullptr || sf_cols == nullptr)
        return QL_ERR_INVALID_ARG;
    if (x_stride_m < n || out_rows_stride_m < n || out_cols_stride_m < n) return QL_ERR_INVALID_ARG;
    if ((m + 127) / 128 > 65535) return QL_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (ql_status s = device_info(di); s != QL_OK) return s;
    ql::CastDualArgs a{};
    a.dev_status = di.status;
    a.x = x;
    a.is_bf16 = x_dtype == QL_BF16;
    a.m = m;
    a.n = n;
    a.sxm = x_stride_m;
    a.fmt = base;
    a.recip = recip;
    a.qr = out_rows;
    a.ldr = out_rows_stride_m;
    a.sfr = sf_rows;
    a.srm = sf_rows_stride_m;
    a.srg = sf_rows_stride_g;
    a.qc = out_cols;
    a.ldc = out_cols_stride_m;
    a.sfc = sf_cols;
    a.scn = sf_cols_stride_n;
    a.scg = sf_cols_stride_g;
    return from_cuda(ql::launch_cast_dual(a, reinterpret_cast<cudaStream_t>(stream)));
}

ql_status fp8_cast_per_block(const void* x, ql_dtype x_dtype, int64_t m, int64_t n, int64_t x_stride_m,
                             int64_t x_stride_n, int fmt, uint8_t* out, int64_t out_stride_m, int64_t out_stride_n,
                             void* out_sf, int64_t sf_stride_r, int64_t sf_stride_c, ql_stream_t stream) {
    return cast_per_block_common(x, x_dtype, m, n, x_stride_m, x_stride_n, fmt, out, out_stride_m, out_stride_n,
                                 out_sf, sf_stride_r, sf_stride_c, nullptr, 0, 0, false, stream);
}

ql_status fp8_cast_per_block_dual(const void* x, ql_dtype x_dtype, int64_t m, int64_t n, int64_t x_stride_m,
                                  int64_t x_stride_n, int fmt, uint8_t* out, int64_t out_stride_m,
                                  int64_t out_stride_n, void* out_sf, int64_t sf_stride_r, int64_t sf_stride_c,
                                  void* out_sf_t, int64_t sf_t_stride_c, int64_t sf_t_stride_r, ql_stream_t stream) {
    return cast_per_block_common(x, x_dtype, m, n, x_stride_m, x_stride_n, fmt, out, out_stride_m, out_stride_n,
                                 out_sf, sf_stride_r, sf_stride_c, out_sf_t, sf_t_stride_c, sf_t_stride_r, true,
                                 stream);
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

size_t ql_cast_gemm_host_workspace_size(int64_t n, int64_t k, int64_t chunk_rows, int fmt) {
    if (n <= 0 || k <= 0 || chunk_rows <= 0) return 0;
    return kPipeSlots * slot_layout(n, k, chunk_rows, fmt).total;
}

ql_status ql_cast_gemm_host(const void* x_host, int64_t ldx, const uint8_t* b, int64_t ldb, const void* sfb,
                            int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt, uint16_t* d_host, int64_t ldd,
                            int64_t m, int64_t n, int64_t k, int64_t chunk_rows, void* workspace, size_t ws_bytes,
                            ql_stream_t stream) {
    if (m < 0 || n < 0 || k <= 0 || chunk_rows <= 0) return QL_ERR_INVALID_ARG;
    if (fmt < QL_SF_FP32 || fmt > QL_SF_PACKED_UE8M0) return QL_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return QL_OK;
    if (x_host == nullptr || d_host == nullptr || b == nullptr || sfb == nullptr || workspace == nullptr)
        return QL_ERR_INVALID_ARG;
    if (ldx < k || ldd < n) return QL_ERR_INVALID_ARG;
    // the GEMM's own checks of B, made here so that an error returns before
    // anything is queued
    if (n >= (int64_t(1) << 31) || k >= (int64_t(1) << 31)) return QL_ERR_UNSUPPORTED;
    if (ldb < k) return QL_ERR_INVALID_ARG;
    if (!aligned16(b) || ldb % 16 != 0) return QL_ERR_ALIGNMENT;
    const SlotLayout sl = slot_layout(n, k, chunk_rows, fmt);
    if (ws_bytes < kPipeSlots * sl.total) return QL_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QL_ERR_ALIGNMENT;
    Pipe* pp = nullptr;
    ql_status st = pipe_for_device(pp);
    if (st != QL_OK) return st;
    Pipe& P = *pp;
    std::lock_guard<std::mutex> lk(P.mu);
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    // the pipeline starts after the caller's earlier work and the caller's
    // stream resumes after its last copy
    if (!ck(cudaEventRecord(P.start, cs)) || !ck(cudaStreamWaitEvent(P.in, P.start, 0)) ||
        !ck(cudaStreamWaitEvent(P.comp, P.start, 0)) || !ck(cudaStreamWaitEvent(P.out, P.start, 0)))
        return QL_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t chunks = (m + chunk_rows - 1) / chunk_rows;
    for (int64_t c = 0; c < chunks && st == QL_OK; ++c) {
        const int slot = static_cast<int>(c % kPipeSlots);
        const int64_t r0 = c * chunk_rows;
        const int64_t rc = (m - r0) < chunk_rows ? (m - r0) : chunk_rows;
        uint8_t* base = ws + slot * sl.total;
        uint16_t* xb = reinterpret_cast<uint16_t*>(base);
        uint8_t* qb = base + sl.x;
        void* sb = base + sl.x + sl.q;
        uint16_t* db = reinterpret_cast<uint16_t*>(base + sl.x + sl.q + sl.s);
        // copy in: the slot's X buffer is free once chunk c - slots was cast
        if (c >= kPipeSlots && !ck(cudaStreamWaitEvent(P.in, P.comp_done[slot], 0))) { st = QL_ERR_CUDA; break; }
        if (!ck(cudaMemcpy2DAsync(xb, static_cast<size_t>(k) * 2,
                                  static_cast<const uint8_t*>(x_host) + static_cast<size_t>(r0) * ldx * 2,
                                  static_cast<size_t>(ldx) * 2, static_cast<size_t>(k) * 2, static_cast<size_t>(rc),
                                  cudaMemcpyHostToDevice, P.in)) ||
            !ck(cudaEventRecord(P.in_done[slot], P.in))) {
            st = QL_ERR_CUDA;
            break;
        }
        // cast + GEMM: after the copy in, and after the slot's D went out
        if (!ck(cudaStreamWaitEvent(P.comp, P.in_done[slot], 0)) ||
            (c >= kPipeSlots && !ck(cudaStreamWaitEvent(P.comp, P.out_done[slot], 0)))) {
            st = QL_ERR_CUDA;
            break;
        }
        st = fp8_cast_per_token(xb, QL_BF16, rc, k, k, 1, 128, fmt, qb, sl.ldq, 1, sb, 1, sl.sld,
                                reinterpret_cast<ql_stream_t>(P.comp));
        if (st == QL_OK)
            st = gemm_fp8_nt_bf16(qb, sl.ldq, sb, 1, sl.sld, b, ldb, sfb, sfb_stride_n, sfb_stride_k, fmt, db, n, rc,
                                  n, k, nullptr, 0, reinterpret_cast<ql_stream_t>(P.comp));
        if (st != QL_OK) break;
        if (!ck(cudaEventRecord(P.comp_done[slot], P.comp))) { st = QL_ERR_CUDA; break; }
        // copy out
        if (!ck(cudaStreamWaitEvent(P.out, P.comp_done[slot], 0)) ||
            !ck(cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(d_host) + static_cast<size_t>(r0) * ldd * 2,
                                  static_cast<size_t>(ldd) * 2, db, static_cast<size_t>(n) * 2,
                                  static_cast<size_t>(n) * 2, static_cast<size_t>(rc), cudaMemcpyDeviceToHost, P.out)) ||
            !ck(cudaEventRecord(P.out_done[slot], P.out))) {
            st = QL_ERR_CUDA;
            break;
        }
    }
    // Whatever happened, the caller's stream resumes only after everything the
    // call queued on the three streams (copies touching the caller's host
    // buffers included), so an error return leaves nothing unordered.
    if (!ck(cudaEventRecord(P.in_done[0], P.in)) || !ck(cudaStreamWaitEvent(P.out, P.in_done[0], 0)) ||
        !ck(cudaEventRecord(P.comp_done[0], P.comp)) || !ck(cudaStreamWaitEvent(P.out, P.comp_done[0], 0)) ||
        !ck(cudaEventRecord(P.end, P.out)) || !ck(cudaStreamWaitEvent(cs, P.end, 0)))
        return QL_ERR_CUDA;
    return st;
}

int ql_binary_version(void) {
    cudaFuncAttributes attr{};
    if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(&ql_probe_kernel)) != cudaSuccess) return 0;
    return attr.binaryVersion;
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
    if (path < 0 || path > 7) return QL_ERR_INVALID_ARG;
    g_gemm_path.store(path);
    return QL_OK;
}

ql_status ql_test_stall_gemm_producer(int enable) {
    g_stall_producer.store(enable ? 1 : 0);
    return QL_OK;
}

ql_status ql_device_status_detail(ql_stream_t stream, uint32_t* flags, uint64_t* first_bad_address) {
    DeviceInfo di;
    ql_status s = device_info(di);
    if (s != QL_OK) return s;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QL_ERR_CUDA;
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (cudaMemcpy(v, di.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QL_ERR_CUDA;
    if (flags != nullptr) *flags = v[0];
    if (first_bad_address != nullptr) *first_bad_address = static_cast<uint64_t>(v[2]) | (static_cast<uint64_t>(v[3]) << 32);
    if (v[0] != 0 || v[2] != 0 || v[3] != 0) {
        const uint32_t zero[4] = {0u, 0u, 0u, 0u};
        if (cudaMemcpy(di.status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return QL_ERR_CUDA;
    }
    if (v[0] & ql::kDevErrTimeout) return QL_ERR_DEVICE_TIMEOUT;
    if (v[0] & ql::kDevErrBounds) return QL_ERR_OUT_OF_BOUNDS;
    if (v[0] != 0) return QL_ERR_INVALID_ARG;
    return QL_OK;
}

ql_status ql_device_status(ql_stream_t stream) { return ql_device_status_detail(stream, nullptr, nullptr); }

int ql_bounds_checked(void) {
#ifdef QL_BOUNDS_CHECK
    return 1;
#else
    return 0;
#endif
}

}  // extern "C"
