/*
 * CPU oracle for the fine-grained-scaled FP8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do. It shares no code, header, table or constant with
 * the CUDA library: everything below is written from the format and method
 * definitions, plainly and slowly, in double precision where the method does
 * not fix the precision.
 *
 * Sources (page titles; section in brackets):
 *  - "DeepGEMM Essentials: High-Performance FP8 Matrix Multiplication"
 *    [Part 3] per-token cast in 1x128 groups, amax clamped at 1e-4,
 *    data = x * (448 / amax) cast to E4M3, scale = amax / 448;
 *    [Part 4] the same over zero-padded 128x128 blocks;
 *    [Part 5] RHS scales [ceil(n/128), ceil(k/128)] contiguous;
 *    [Part 6] D = LHS * RHS^T; [Part 12-13] wgrad with fp32 accumulation.
 *  - "[Help] Starter script for nn.Linear for fwd,bwd" (DeepGEMM issue #102)
 *    [maintainer's reply on RHS scales] the RHS scale grid is read row-wise,
 *    one row (1, ceil(k/128)) per 128-row block of RHS, for every K block.
 *  - "deep-gemm: fused per-token FP8 cast in Triton
 *    (fused_per_token_cast_to_fp8), version 3" [description] gran_k 32|128,
 *    UE8M0 scales, packed UE8M0, correctly rounded reciprocal.
 *  - The OCP 8-bit floating point specification (E4M3 "FN": bias 7, three
 *    mantissa bits, subnormals, no infinities, max 448, NaN S.1111.111).
 *
 * Readings taken where the pages are silent (listed with reasons in the
 * design notes of the repository):
 *  - factor: f = fl32(448 / amax) by default (Part 3's printed formula);
 *    the alternative f = fl32(1 / fl32(amax / 448)) is selected by `recip`.
 *  - UE8M0: the scale is rounded UP to the next power of two, so that
 *    |x * f| <= 448 still holds; stored as an fp32 holding that power of two,
 *    or as the biased exponent byte when packed.
 *  - packed UE8M0: group j's byte is byte (j % 4) (little-endian) of int32
 *    word j / 4; bytes of groups past the last real group are 0.
 *    (parity unpinned: the pages do not print the packing.)
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ----- element types and scale formats (values mirror the public ABI's
 * enumerations only by value; this file includes no header of it) ------- */
enum { OR_BF16 = 0, OR_F32 = 1 };
enum { OR_SF_FP32 = 0, OR_SF_UE8M0 = 1, OR_SF_PACKED_UE8M0 = 2 };

/* Number of E4M3 encodings that needed saturation (|y| above 464). The
 * method never produces such a value; the tests assert this stays 0. */
static long long g_overflow_count = 0;

long long oracle_overflow_count(void) { return g_overflow_count; }
void oracle_reset_overflow_count(void) { g_overflow_count = 0; }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

/* ------------------------------------------------------------------------
 * E4M3FN, from the OCP definition.
 *   value(b) = (-1)^s * 2^(e-7) * (1 + m/8)   for e in 1..15 (except e=15,m=7)
 *            = (-1)^s * 2^(-6) * (m/8)        for e = 0 (subnormal)
 *   e=15, m=7 is NaN; there is no infinity; max magnitude 448 (e=15, m=6).
 * ---------------------------------------------------------------------- */
double oracle_e4m3_decode(uint8_t b) {
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);           /* m/8 * 2^-6 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even encoding of a finite real v (given as a double that
 * holds an fp32 value). The representable magnitudes are the multiples of
 * the quantum 2^(E-3) in the binade [2^E, 2^(E+1)), E >= -6, and multiples of
 * 2^-9 below 2^-6. Magnitudes that round above 448 saturate (counted). */
uint8_t oracle_e4m3_encode(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    if (a == 0.0) return sign;
    /* a >= 464 rounds past 448 (464 itself is a tie and goes to 448's even
     * mantissa); the method never gets here. */
    if (a > 464.0) { g_overflow_count++; return (uint8_t)(sign | 0x7E); }
    int ex;
    frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;                /* a in [2^E, 2^(E+1)) */
    if (E < -6) E = -6;            /* subnormals share the quantum 2^-9 */
    double quantum = ldexp(1.0, E - 3);
    double q = a / quantum;        /* exact: scaling by a power of two */
    double r = nearbyint(q);       /* default rounding mode: to nearest even */
    double val = r * quantum;      /* exact */
    if (val == 0.0) return sign;
    if (val > 448.0) { g_overflow_count++; return (uint8_t)(sign | 0x7E); }
    int ex2;
    frexp(val, &ex2);
    int E2 = ex2 - 1;
    if (E2 < -6) {                 /* subnormal: val = m * 2^-9 */
        int m = (int)ldexp(val, 9);
        return (uint8_t)(sign | m);
    }
    int m = (int)ldexp(val, 3 - E2) - 8;            /* (val/2^E2 - 1) * 8 */
    return (uint8_t)(sign | ((E2 + 7) << 3) | m);
}

/* Batch helpers used by the pins. */
void oracle_e4m3_encode_f32_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode((double)v[i]);
}
void oracle_e4m3_decode_array(const uint8_t* b, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(b[i]);
}

/* ------------------------------------------------------------------------
 * Output rounding of the GEMM. The fwd/dgrad GEMM writes bf16 (8 significant
 * bits, bias 127): round to nearest, ties to even, directly from the exact
 * (double) value. The wgrad GEMM writes fp32: (float) conversion is RNE.
 * ---------------------------------------------------------------------- */
double oracle_round_bf16(double v) {
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    double a = fabs(v);
    int ex;
    frexp(a, &ex);
    int E = ex - 1;                /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;        /* bf16 subnormals: quantum 2^-133 */
    double quantum = ldexp(1.0, E - 7);
    double r = nearbyint(a / quantum) * quantum;
    return v < 0 ? -r : r;
}

void oracle_round_array(double* v, int64_t n, int mode) {
    for (int64_t i = 0; i < n; ++i) {
        if (mode == 1) v[i] = oracle_round_bf16(v[i]);
        else if (mode == 2) v[i] = (double)(float)v[i];
    }
}

/* ------------------------------------------------------------------------
 * Scalars of the cast.
 * ---------------------------------------------------------------------- */
static float bf16_bits_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;      /* bf16 is the top half of fp32 */
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static float load_elem(const void* x, int dtype, int64_t off) {
    if (dtype == OR_BF16) return bf16_bits_to_float(((const uint16_t*)x)[off]);
    return ((const float*)x)[off];
}

/* fl32(1e-4): the clamp floor of Part 3 applied to an fp32 tensor. */
static float clamp_floor(void) { return (float)1e-4; }

/* Smallest power of two >= s (s > 0, finite, normal). */
static double pow2_ceil(double s) {
    int ex;
    double f = frexp(s, &ex);                       /* s = f * 2^ex */
    if (f == 0.5) return s;                         /* already 2^(ex-1) */
    return ldexp(1.0, ex);
}

/* Biased exponent byte of a power of two p = 2^(B-127). */
static uint8_t ue8m0_byte(double p) {
    int ex;
    frexp(p, &ex);                                  /* p = 0.5 * 2^ex */
    return (uint8_t)((ex - 1) + 127);
}

/* Scale and factor of one group (or block) from its amax.
 *   fp32 format : s = fl32(amax/448),  f = fl32(448/amax)  (or 1/s, recip)
 *   UE8M0       : s = 2^ceil(log2 fl32(amax/448)),  f = 1/s  (exact)
 * Division in double then rounding to fp32 is correctly rounded for fp32
 * operands (double rounding is harmless for division at 53 >= 2*24+2). */
static void group_scale(float amax, int fmt, int recip, double* s_out, float* f_out) {
    float a = amax > clamp_floor() ? amax : clamp_floor();
    float s = (float)((double)a / 448.0);
    if (fmt == OR_SF_FP32) {
        *s_out = s;
        if (recip) *f_out = (float)(1.0 / (double)s);
        else *f_out = (float)(448.0 / (double)a);
    } else {
        double p = pow2_ceil((double)s);
        *s_out = p;
        *f_out = (float)(1.0 / p);                  /* exact power of two */
    }
}

/* Quantise one element: y = fl32(x * f), then E4M3 round-to-nearest-even. */
static uint8_t quantise(float x, float f) {
    float y = (float)((double)x * (double)f);      /* product exact in double */
    return oracle_e4m3_encode((double)y);
}

/* ------------------------------------------------------------------------
 * Per-token cast (Part 3; gran_k and UE8M0 options of the fused-cast PR).
 * x[i*sxm + j*sxn], out[i*som + j*son]; scales at sf[i*ssm + g*ssg]
 * (fp32 elements) or, packed, int32 words at sf[i*ssm + w*ssg].
 * Returns 0, or -1 on bad arguments.
 * ---------------------------------------------------------------------- */
int oracle_cast_per_token(const void* x, int dtype, int64_t m, int64_t n,
                          int64_t sxm, int64_t sxn, int gran, int fmt, int recip,
                          uint8_t* out, int64_t som, int64_t son,
                          void* sf, int64_t ssm, int64_t ssg) {
    if (gran <= 0 || m < 0 || n < 0) return -1;
    int64_t G = (n + gran - 1) / gran;
    int64_t W = (G + 3) / 4;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i) {
        if (fmt == OR_SF_PACKED_UE8M0) {
            for (int64_t w = 0; w < W; ++w) ((int32_t*)sf)[i * ssm + w * ssg] = 0;
        }
        for (int64_t g = 0; g < G; ++g) {
            int64_t j0 = g * gran, j1 = j0 + gran < n ? j0 + gran : n;
            float amax = 0.0f;
            for (int64_t j = j0; j < j1; ++j) {
                float v = fabsf(load_elem(x, dtype, i * sxm + j * sxn));
                if (v > amax) amax = v;
            }
            double s; float f;
            group_scale(amax, fmt, recip, &s, &f);
            for (int64_t j = j0; j < j1; ++j)
                out[i * som + j * son] = quantise(load_elem(x, dtype, i * sxm + j * sxn), f);
            if (fmt == OR_SF_FP32 || fmt == OR_SF_UE8M0) {
                ((float*)sf)[i * ssm + g * ssg] = (float)s;
            } else {
                uint32_t* word = (uint32_t*)sf + (i * ssm + (g / 4) * ssg);
                *word |= ((uint32_t)ue8m0_byte(s)) << (8 * (g % 4));
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Per-block (128x128) cast (Part 4). Scales fp32 [ceil(m/128), ceil(n/128)]
 * at sf[r*ssr + c*ssc] (fp32 or UE8M0-as-fp32), or packed UE8M0 int32 words
 * along the column-block axis: block c is byte c % 4 of word c / 4.
 * ---------------------------------------------------------------------- */
int oracle_cast_per_block(const void* x, int dtype, int64_t m, int64_t n,
                          int64_t sxm, int64_t sxn, int fmt, int recip,
                          uint8_t* out, int64_t som, int64_t son,
                          void* sf, int64_t ssr, int64_t ssc) {
    const int64_t B = 128;
    if (m < 0 || n < 0) return -1;
    int64_t R = (m + B - 1) / B, C = (n + B - 1) / B;
    if (fmt == OR_SF_PACKED_UE8M0)          /* words along the column-block axis start at 0 */
        for (int64_t r = 0; r < R; ++r)
            for (int64_t w = 0; w < (C + 3) / 4; ++w) ((int32_t*)sf)[r * ssr + w * ssc] = 0;
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t c = 0; c < C; ++c) {
            int64_t i1 = (r + 1) * B < m ? (r + 1) * B : m;
            int64_t j1 = (c + 1) * B < n ? (c + 1) * B : n;
            float amax = 0.0f;
            for (int64_t i = r * B; i < i1; ++i)
                for (int64_t j = c * B; j < j1; ++j) {
                    float v = fabsf(load_elem(x, dtype, i * sxm + j * sxn));
                    if (v > amax) amax = v;
                }
            double s; float f;
            group_scale(amax, fmt, recip, &s, &f);
            for (int64_t i = r * B; i < i1; ++i)
                for (int64_t j = c * B; j < j1; ++j)
                    out[i * som + j * son] = quantise(load_elem(x, dtype, i * sxm + j * sxn), f);
            if (fmt == OR_SF_PACKED_UE8M0) {
                uint32_t* word = (uint32_t*)sf + (r * ssr + (c / 4) * ssc);
                #pragma omp atomic
                *word |= ((uint32_t)ue8m0_byte(s)) << (8 * (c % 4));
            } else {
                ((float*)sf)[r * ssr + c * ssc] = (float)s;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Block-scaled GEMM, D = A * B^T (Part 6; scale orientation from the issue
 * reply; wgrad form of Parts 12-13 with per-row B scales).
 *
 *   D[i,j] = sum_kb  sa(i,kb) * sb(j,kb) * sum_{k in kb} dec(A[i,k]) dec(B[j,k])
 *
 * sb(j,kb) = sfb[(j/128)*sbn + kb*sbk] when b_per_row == 0 (128x128 blocks),
 *          = sfb[j*sbn + kb*sbk]       when b_per_row == 1 (1x128 per row).
 * Scales are fp32 values (fmt 0 or 1), or packed UE8M0 (fmt 2): the
 * exponent byte (kb % 4) of int32 word kb / 4, value 2^(byte-127).
 * kgran is the scale granularity along K (128).
 * Output in double: d[i*ldd + j]; if d_in is given it is added (accumulate).
 * rows: optional list of nrows row indices to compute (sampled checks);
 *       when rows is NULL all m rows are computed and nrows is ignored.
 * ---------------------------------------------------------------------- */
static double load_scale(const void* sf, int fmt, int64_t row_off, int64_t kb, int64_t sk) {
    if (fmt != OR_SF_PACKED_UE8M0) return (double)((const float*)sf)[row_off + kb * sk];
    uint32_t w = ((const uint32_t*)sf)[row_off + (kb / 4) * sk];
    int byte = (int)((w >> (8 * (kb % 4))) & 0xFF);
    return ldexp(1.0, byte - 127);
}

int oracle_gemm(const uint8_t* a, int64_t lda, const void* sfa, int64_t sam, int64_t sak,
                const uint8_t* b, int64_t ldb, const void* sfb, int64_t sbn, int64_t sbk,
                int fmt, int b_per_row, int kgran,
                int64_t m, int64_t n, int64_t k,
                const int64_t* rows, int64_t nrows,
                double* d, int64_t ldd, const double* d_in, int64_t ldd_in) {
    if (kgran <= 0 || m < 0 || n < 0 || k < 0) return -1;
    /* decode table of all 256 codes, from the definition above */
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = oracle_e4m3_decode((uint8_t)c);
    int64_t KB = (k + kgran - 1) / kgran;
    int64_t R = rows ? nrows : m;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                int64_t k0 = kb * kgran, k1 = k0 + kgran < k ? k0 + kgran : k;
                double part = 0.0;                    /* exact for E4M3 inputs */
                for (int64_t kk = k0; kk < k1; ++kk)
                    part += dec[a[i * lda + kk]] * dec[b[j * ldb + kk]];
                double sa = load_scale(sfa, fmt, i * sam, kb, sak);
                int64_t brow = b_per_row ? j : j / 128;
                double sb = load_scale(sfb, fmt, brow * sbn, kb, sbk);
                acc += (sa * sb) * part;
            }
            if (d_in) acc += d_in[i * ldd_in + j];
            d[r * ldd + j] = acc;
        }
    }
    return 0;
}
