// Bounds-checked builds.
//
// Compiled with -DQL_BOUNDS_CHECK, every plain global load and store of the
// kernels is checked against the byte range of the caller's buffer it belongs
// to (TMA copies need no check: the hardware clips them to their tensor maps).
// An access outside its range is skipped, not made; the kernel raises a bit in
// the device status word and keeps the first offending address beside it, and
// ql_device_status() reports QL_ERR_OUT_OF_BOUNDS. No trap, no assert: the
// context stays usable. In normal builds the checks compile to nothing and the
// ranges are passed but unused.
#pragma once

#include <stdint.h>

namespace ql {

constexpr uint32_t kDevErrBounds = 4u;   // a bounds-checked access was out of range

// Byte range [lo, hi) of one buffer.
struct Span {
    uint64_t lo, hi;
};

constexpr int kMaxSpans = 6;

// The ranges of the buffers one kernel touches with plain loads and stores,
// and the device status word (bits at status[0], first offending address as
// a 64-bit word at status + 2).
struct Bounds {
    Span s[kMaxSpans];
    uint32_t* status;
};

// Byte range of a [d0 x d1 x d2] view of es-byte elements with element
// strides s0, s1, s2 (any sign) at base; empty when base is null or any
// extent is zero.
inline Span span_of(const void* base, int64_t es, int64_t d0, int64_t s0, int64_t d1 = 1, int64_t s1 = 0,
                    int64_t d2 = 1, int64_t s2 = 0) {
    if (base == nullptr || d0 <= 0 || d1 <= 0 || d2 <= 0) return Span{0, 0};
    int64_t lo = 0, hi = 0;
    const int64_t ext[3] = {(d0 - 1) * s0, (d1 - 1) * s1, (d2 - 1) * s2};
    for (int i = 0; i < 3; ++i) {
        if (ext[i] < 0) lo += ext[i];
        else hi += ext[i];
    }
    const uint64_t b = reinterpret_cast<uint64_t>(base);
    return Span{b + static_cast<uint64_t>(lo * es), b + static_cast<uint64_t>((hi + 1) * es)};
}

#ifdef __CUDACC__
#ifdef QL_BOUNDS_CHECK
__device__ __forceinline__ bool in_span(const Bounds& b, int i, const void* p, uint32_t bytes) {
    const uint64_t a = reinterpret_cast<uint64_t>(p);
    if (a >= b.s[i].lo && a + bytes <= b.s[i].hi) return true;
    if (b.status != nullptr) {
        atomicOr(b.status, kDevErrBounds);
        atomicCAS(reinterpret_cast<unsigned long long*>(b.status + 2), 0ull, static_cast<unsigned long long>(a));
    }
    return false;
}
#define QL_IN(b, i, p, bytes) ::ql::in_span((b), (i), (p), static_cast<uint32_t>(bytes))
#else
#define QL_IN(b, i, p, bytes) true
#endif
#endif

}  // namespace ql
