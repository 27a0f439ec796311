/*
 * qlinear.h — C ABI of libqlinear.so: the fine-grained-scaled FP8 linear layer
 * on GB300 (sm_103a).
 *
 * Two operations, each a CUDA kernel launched on the caller's stream:
 *   - the FP8 cast (per token in 1x128 / 1x32 groups, or per 128x128 block),
 *   - the block-scaled FP8 GEMM D = A * B^T (bf16 output for fwd/dgrad,
 *     fp32 output, optionally accumulated, for wgrad).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     allocates no device memory and never frees caller memory.
 *   - Strides are in ELEMENTS of the tensor's own type (bf16/fp32: 2/4 bytes,
 *     e4m3: 1 byte, scales: 4 bytes), signed 64-bit. A "view" (any strides) of
 *     a larger buffer may be passed; only the view's elements are written
 *     (bytes outside it are never touched).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous: no call synchronises the host. Arguments are validated on
 *     the host before any launch; an invalid call launches nothing.
 *   - Errors are returned as ql_status; no exception crosses the ABI.
 *     Device-side wait time-outs are recorded in a device status word that
 *     ql_device_status() reads (that call synchronises the given stream).
 *   - E4M3 means the OCP E4M3FN byte format (max 448, no infinities).
 */
#ifndef QLINEAR_H
#define QLINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* ql_stream_t;   /* same type as cudaStream_t */

typedef enum {
    QL_OK = 0,
    QL_ERR_INVALID_ARG = 1,     /* null pointer, negative size, bad enum value */
    QL_ERR_UNSUPPORTED = 2,     /* valid request this build does not implement */
    QL_ERR_ALIGNMENT = 3,       /* pointer / stride alignment the kernel needs is not met */
    QL_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed */
    QL_ERR_DEVICE_TIMEOUT = 5,  /* a kernel's bounded wait ran out (see ql_device_status) */
    QL_ERR_OUT_OF_BOUNDS = 6    /* bounds-checked builds only: an access outside its buffer was skipped */
} ql_status;

typedef enum { QL_BF16 = 0, QL_F32 = 1 } ql_dtype;

/* Scale-factor storage (the use_ue8m0 / use_packed_ue8m0 options of
 * "deep-gemm: fused per-token FP8 cast in Triton (fused_per_token_cast_to_fp8),
 * version 3" [description]):
 *   QL_SF_FP32          fp32 scale = fl32(amax / 448)
 *   QL_SF_UE8M0         fp32 tensor holding 2^ceil(log2(amax / 448)) (a power of two)
 *   QL_SF_PACKED_UE8M0  int32 words, 4 biased-exponent bytes per word along the
 *                       group axis: group g is byte (g % 4), little-endian, of
 *                       word g / 4; bytes of groups past the last are 0.
 * QL_CAST_RECIP_OF_SCALE may be OR-ed into the format of a cast with
 * QL_SF_FP32: the quantisation factor is then fl32(1 / scale) instead of the
 * default fl32(448 / amax) (both correctly rounded). */
typedef enum { QL_SF_FP32 = 0, QL_SF_UE8M0 = 1, QL_SF_PACKED_UE8M0 = 2 } ql_sf_format;
#define QL_CAST_RECIP_OF_SCALE 0x100

/* Human-readable name of a status code (static storage). */
const char* ql_status_string(ql_status s);

/* ---------------------------------------------------------------------------
 * fp8_cast_per_token
 * Per-token cast of "DeepGEMM Essentials: High-Performance FP8 Matrix
 * Multiplication" Part 3, with the options of "deep-gemm: fused per-token FP8
 * cast in Triton (fused_per_token_cast_to_fp8), version 3" [description]
 * (gran_k, UE8M0, packed UE8M0, in-place out / out_sf).
 *
 * For each row i and group g (columns [g*gran_k, min(n, (g+1)*gran_k))):
 *   amax   = max(max_j |x[i,j]|, fl32(1e-4))      (exact, fp32)
 *   scale  = fl32(amax / 448), rounded up to a power of two for UE8M0 formats
 *   factor = fl32(448 / amax) for QL_SF_FP32 (fl32(1/scale) with
 *            QL_CAST_RECIP_OF_SCALE); 1/scale (exact) for UE8M0 formats
 *   out[i,j] = E4M3_rn(fl32(x[i,j] * factor))  (sign kept; |.| <= 448)
 * The result is bit-exact (data and scale bytes).
 *
 *   x            [m, n] bf16 or fp32, element (i,j) at x[i*x_stride_m + j*x_stride_n].
 *                A transposed view (x_stride_m == 1) casts along the other axis:
 *                this is how the wgrad operands (dY^T, X^T) are produced.
 *   gran_k       32 or 128.
 *   fmt          ql_sf_format, optionally | QL_CAST_RECIP_OF_SCALE.
 *   out          [m, n] E4M3 bytes at out[i*out_stride_m + j*out_stride_n].
 *   out_sf       [m, ceil(n/gran_k)] fp32 at out_sf[i*sf_stride_m + g*sf_stride_g],
 *                or for QL_SF_PACKED_UE8M0 [m, ceil(ceil(n/gran_k)/4)] int32 words
 *                at out_sf[i*sf_stride_m + w*sf_stride_g]. sf_stride_m == 1 with
 *                sf_stride_g a multiple of 4 gives the M-major, TMA-aligned
 *                layout the GEMM's LHS scales use (Part 5).
 * Fast paths: x_stride_n == 1 (rows contiguous) or x_stride_m == 1 (transposed),
 * with out_stride_n == 1; any other strides use a slower generic kernel.
 * m == 0 or n == 0 is a no-op. Returns QL_ERR_INVALID_ARG for null pointers with
 * m*n > 0, negative sizes, gran_k not in {32,128}, or an unknown format.
 * ------------------------------------------------------------------------- */
ql_status fp8_cast_per_token(const void* x, ql_dtype x_dtype, int64_t m, int64_t n,
                             int64_t x_stride_m, int64_t x_stride_n,
                             int gran_k, int fmt,
                             uint8_t* out, int64_t out_stride_m, int64_t out_stride_n,
                             void* out_sf, int64_t sf_stride_m, int64_t sf_stride_g,
                             ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * fp8_cast_per_token_dual
 * Both per-token casts the Linear layer takes of one activation, from a single
 * read of it: fp8_cast_per_token(x, 128, fmt) and fp8_cast_per_token(x^T,
 * 128, fmt). In "[Help] Starter script for nn.Linear for fwd,bwd" X is cast
 * along its features for the forward GEMM and along the tokens for the weight
 * gradient, and dY likewise for the data and weight gradients. The results are
 * bit-identical to the two separate calls.
 *   x          [m, n] bf16 or fp32, rows contiguous, row stride x_stride_m >= n.
 *   out_rows   [m, n] E4M3, the cast of x (1x128 groups along n), row stride
 *              out_rows_stride_m >= n; sf_rows [m, ceil(n/128)] at
 *              sf_rows[i*sf_rows_stride_m + g*sf_rows_stride_g] (packed UE8M0:
 *              int32 words along g, as fp8_cast_per_token).
 *   out_cols   [m, n] E4M3, the cast of x^T (1x128 groups along m) kept in x's
 *              own layout: element (i, j) of x at out_cols[i*out_cols_stride_m + j]
 *              (the K-outer operand of gemm_fp8_wgrad_fp32_mn); sf_cols
 *              [n, ceil(m/128)] at sf_cols[j*sf_cols_stride_n + g*sf_cols_stride_g].
 *   fmt        ql_sf_format, optionally | QL_CAST_RECIP_OF_SCALE with QL_SF_FP32.
 * m == 0 or n == 0 is a no-op. QL_ERR_INVALID_ARG for null pointers with
 * m*n > 0, negative sizes, a row stride below n, or an unknown format.
 * ------------------------------------------------------------------------- */
ql_status fp8_cast_per_token_dual(const void* x, ql_dtype x_dtype, int64_t m, int64_t n,
                                  int64_t x_stride_m, int fmt,
                                  uint8_t* out_rows, int64_t out_rows_stride_m, void* sf_rows,
                                  int64_t sf_rows_stride_m, int64_t sf_rows_stride_g,
                                  uint8_t* out_cols, int64_t out_cols_stride_m, void* sf_cols,
                                  int64_t sf_cols_stride_n, int64_t sf_cols_stride_g,
                                  ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * fp8_cast_per_block
 * 128x128 block cast of "DeepGEMM Essentials" Part 4 (the RHS / weight cast).
 * Same arithmetic as fp8_cast_per_token with the group being a 128x128 block
 * (edge blocks partial). Scales fp32 [ceil(m/128), ceil(n/128)] at
 * out_sf[r*sf_stride_r + c*sf_stride_c] for QL_SF_FP32 / QL_SF_UE8M0
 * (optionally | QL_CAST_RECIP_OF_SCALE with QL_SF_FP32); for
 * QL_SF_PACKED_UE8M0 int32 words [ceil(m/128), ceil(ceil(n/128)/4)] packed
 * along the column-block axis (block c is byte c % 4 of word c / 4, pad bytes
 * 0) at out_sf[r*sf_stride_r + w*sf_stride_c]: the GEMM's B-scale layout.
 * Either view may be transposed: x_stride_m == 1 reads x column-wise, and
 * out_stride_m == 1 writes the data transposed. Since a block's amax does not
 * depend on orientation, cast_per_block(W^T) (the dgrad operand of "[Help]
 * Starter script for nn.Linear for fwd,bwd") is obtained either by passing
 * x = W^T as a transposed view of W, or (fp32 / UE8M0 scales) by writing W's
 * cast through transposed out / out_sf views; for packed scales use the first
 * form, so that the words pack along W^T's column blocks.
 * ------------------------------------------------------------------------- */
ql_status fp8_cast_per_block(const void* x, ql_dtype x_dtype, int64_t m, int64_t n,
                             int64_t x_stride_m, int64_t x_stride_n, int fmt,
                             uint8_t* out, int64_t out_stride_m, int64_t out_stride_n,
                             void* out_sf, int64_t sf_stride_r, int64_t sf_stride_c,
                             ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * fp8_cast_per_block_dual
 * fp8_cast_per_block that also writes, in the same pass, the scale grid of
 * the transposed cast: block (r, c) of x into out_sf_t at
 * [c*sf_t_stride_c + r*sf_t_stride_r] (fp32 / UE8M0), or for
 * QL_SF_PACKED_UE8M0 as byte r % 4 of int32 word [c*sf_t_stride_c +
 * (r/4)*sf_t_stride_r] (words packed along the row-block axis, pad bytes 0);
 * out_sf_t is [ceil(n/128), ceil(m/128)] (fp32) or [ceil(n/128),
 * ceil(ceil(m/128)/4)] (words). A block's amax does not depend on orientation
 * ("DeepGEMM Essentials" Part 4; the W^T requantisation of "[Help] Starter
 * script for nn.Linear for fwd,bwd"), so out_sf_t equals the scales of
 * fp8_cast_per_block(x^T) byte for byte, and out read MN-major with out_sf_t
 * is the data-gradient operand of gemm_fp8_nn_bf16 in every scale format: no
 * cast of W^T is needed. Other arguments, requirements and errors as
 * fp8_cast_per_block; out_sf_t == NULL with m*n > 0 is QL_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
ql_status fp8_cast_per_block_dual(const void* x, ql_dtype x_dtype, int64_t m, int64_t n,
                                  int64_t x_stride_m, int64_t x_stride_n, int fmt,
                                  uint8_t* out, int64_t out_stride_m, int64_t out_stride_n,
                                  void* out_sf, int64_t sf_stride_r, int64_t sf_stride_c,
                                  void* out_sf_t, int64_t sf_t_stride_c, int64_t sf_t_stride_r,
                                  ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_fp8_nt_bf16
 * D = A * B^T of "DeepGEMM Essentials" Parts 1 and 6 (gemm_fp8_fp8_bf16_nt),
 * with the scale semantics of "[Help] Starter script for nn.Linear for fwd,bwd"
 * (maintainer's reply: the RHS scale grid is read row-wise, one row
 * (1, ceil(k/128)) per 128-row block of B, for every K block):
 *
 *   D[i,j] = bf16_rn( sum_kb sa[i,kb] * sb[j/128,kb] * sum_{k in kb} A[i,k] B[j,k] )
 *
 * accumulated in fp32, one promotion per 128-wide K block.
 *   a    [m, k] E4M3, row stride lda bytes (K contiguous).
 *   sfa  [m, ceil(k/128)] scales at sfa[i*sfa_stride_m + kb*sfa_stride_k]
 *        (fp32 values for QL_SF_FP32 / QL_SF_UE8M0; for QL_SF_PACKED_UE8M0
 *        int32 words with kb -> byte kb%4 of word kb/4, i.e. stride_k counts words).
 *   b    [n, k] E4M3, row stride ldb bytes.
 *   sfb  [ceil(n/128), ceil(k/128)] at sfb[r*sfb_stride_n + kb*sfb_stride_k], same format.
 *   d    [m, n] bf16 at d[i*ldd + j].
 *   workspace / ws_bytes: reserved, may be NULL / 0 (ql_gemm_workspace_size returns 0).
 * Requirements (QL_ERR_ALIGNMENT otherwise): a, b 16-byte aligned; lda, ldb
 * multiples of 16 (the tensor-memory-access unit moves 16-byte rows). Any k:
 * the operand tiles are zero-filled past column k. m == 0 or n == 0 is a
 * no-op; k == 0 writes D = 0.
 * ------------------------------------------------------------------------- */
ql_status gemm_fp8_nt_bf16(const uint8_t* a, int64_t lda, const void* sfa,
                           int64_t sfa_stride_m, int64_t sfa_stride_k,
                           const uint8_t* b, int64_t ldb, const void* sfb,
                           int64_t sfb_stride_n, int64_t sfb_stride_k,
                           int fmt, uint16_t* d, int64_t ldd,
                           int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t ws_bytes, ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_fp8_wgrad_fp32
 * The weight-gradient GEMM (wgrad_gemm_fp8_fp8_fp32_nt) of "[Help] Starter
 * script for nn.Linear for fwd,bwd" and "DeepGEMM Essentials" Parts 12-13:
 * both operands carry 1x128 per-row scales along K (K = tokens), output fp32:
 *
 *   D[i,j] (+)= sum_kb sa[i,kb] * sb[j,kb] * sum_{k in kb} A[i,k] B[j,k]
 *
 *   sfb  [n, ceil(k/128)] at sfb[j*sfb_stride_n + kb*sfb_stride_k].
 *   d    [m, n] fp32 at d[i*ldd + j]; accumulate != 0 adds to the existing D.
 * Other arguments and requirements as gemm_fp8_nt_bf16.
 * ------------------------------------------------------------------------- */
ql_status gemm_fp8_wgrad_fp32(const uint8_t* a, int64_t lda, const void* sfa,
                              int64_t sfa_stride_m, int64_t sfa_stride_k,
                              const uint8_t* b, int64_t ldb, const void* sfb,
                              int64_t sfb_stride_n, int64_t sfb_stride_k,
                              int fmt, float* d, int64_t ldd,
                              int64_t m, int64_t n, int64_t k, int accumulate,
                              void* workspace, size_t ws_bytes, ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * m_grouped_gemm_fp8_nt_bf16_contiguous
 * The M-grouped GEMM over the contiguous layout of "DeepGEMM Essentials"
 * Parts 8-11 (m_grouped_gemm_fp8_fp8_bf16_nt_contiguous), as used for the
 * experts of a mixture-of-experts layer: the tokens of all experts are stacked
 * in one matrix A, each expert's rows padded up to a multiple of
 * ql_get_m_alignment_for_contiguous_layout() (128), and m_indices gives the
 * expert of every row (-1 for padding rows). For every row i with
 * e = m_indices[i] >= 0:
 *
 *   D[i,j] = bf16_rn( sum_kb sa[i,kb] * sfb_e[j/128,kb] * sum_{k in kb} A[i,k] B_e[j,k] )
 *
 *   a, sfa     as gemm_fp8_nt_bf16 ([m, k] with 1x128 scales).
 *   b          [num_groups, n, k] E4M3: expert e's row j at b + (e*n + j)*ldb.
 *   sfb        expert e's 128x128 block grid [ceil(n/128), ceil(k/128)] at
 *              sfb[e*sfb_stride_g + r*sfb_stride_n + kb*sfb_stride_k] (Part 10
 *              casts each expert separately), same format rules as sfa.
 *   m_indices  device int32 [m]: expert per row, -1 for padding.
 *   d          [m, n] bf16 at d[i*ldd + j]. Rows with index -1 are not written.
 * Requirements: m a multiple of 128 (QL_ERR_INVALID_ARG otherwise), every
 * expert's segment starting on a multiple of 128, num_groups*n < 2^31,
 * k > 0 (QL_ERR_UNSUPPORTED for k == 0), alignment rules of gemm_fp8_nt_bf16.
 * The indices are read on the device: a 128-row tile whose first index is -1
 * is skipped; an index outside [-1, num_groups), or a row whose expert differs
 * from its tile's first row, is not computed and makes the next
 * ql_device_status() return QL_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
ql_status m_grouped_gemm_fp8_nt_bf16_contiguous(const uint8_t* a, int64_t lda, const void* sfa,
                                                int64_t sfa_stride_m, int64_t sfa_stride_k,
                                                const uint8_t* b, int64_t ldb, const void* sfb,
                                                int64_t sfb_stride_g, int64_t sfb_stride_n,
                                                int64_t sfb_stride_k, int fmt, uint16_t* d,
                                                int64_t ldd, const int32_t* m_indices, int num_groups,
                                                int64_t m, int64_t n, int64_t k, ql_stream_t stream);

/* Row alignment of every expert segment in the contiguous grouped layout
 * ("DeepGEMM Essentials" Part 8: get_m_alignment_for_contiguous_layout): 128. */
int ql_get_m_alignment_for_contiguous_layout(void);

/* ---------------------------------------------------------------------------
 * gemm_fp8_nt_fp8out
 * gemm_fp8_nt_bf16 with the per-token cast of its output fused into the
 * epilogue, so the next layer's E4M3 operand is written directly (the
 * maintainer's advice in "[Help] Starter script for nn.Linear for fwd,bwd":
 * fuse cast and scaling into the previous kernel's output). The result is
 * exactly fp8_cast_per_token(Y, d_gran_k, d_fmt) of Y = the bf16 D that
 * gemm_fp8_nt_bf16 computes with the same tiles:
 *   d      [m, n] E4M3 at d[i*ldd + j] (ldd bytes).
 *   d_sf   [m, ceil(n/d_gran_k)] scales, as fp8_cast_per_token's out_sf
 *          (fp32 at d_sf[i*d_sf_stride_m + g*d_sf_stride_g]; packed UE8M0:
 *          byte g%4 of int32 word d_sf[i*d_sf_stride_m + (g/4)*d_sf_stride_g]).
 *   d_gran_k 32 or 128; d_fmt a ql_sf_format, optionally | QL_CAST_RECIP_OF_SCALE
 *          with QL_SF_FP32.
 * The other arguments and requirements are gemm_fp8_nt_bf16's; k == 0 returns
 * QL_ERR_UNSUPPORTED. The kernels use 256-column tiles for this form.
 * ------------------------------------------------------------------------- */
ql_status gemm_fp8_nt_fp8out(const uint8_t* a, int64_t lda, const void* sfa,
                             int64_t sfa_stride_m, int64_t sfa_stride_k,
                             const uint8_t* b, int64_t ldb, const void* sfb,
                             int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt,
                             uint8_t* d, int64_t ldd, void* d_sf, int64_t d_sf_stride_m,
                             int64_t d_sf_stride_g, int d_gran_k, int d_fmt,
                             int64_t m, int64_t n, int64_t k, ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_fp8_wgrad_fp32_mn
 * gemm_fp8_wgrad_fp32 with both operands MN-major: A stored [k][m] and B
 * stored [k][n] (K = tokens outermost, row strides lda / ldb bytes), i.e. the
 * E4M3 casts of dY [T, out] and X [T, in] kept in their own layout, so the
 * weight gradient of "[Help] Starter script for nn.Linear for fwd,bwd" needs
 * no transposed copies. Scales are those of gemm_fp8_wgrad_fp32 (1x128 along
 * K for every row of A and of B): fp8_cast_per_token of dY^T written into a
 * transposed output view produces both data and scales in this form.
 * Requirements: a, b 16-byte aligned; lda, ldb multiples of 16, lda >= m,
 * ldb >= n (QL_ERR_ALIGNMENT / QL_ERR_INVALID_ARG otherwise).
 * ------------------------------------------------------------------------- */
ql_status gemm_fp8_wgrad_fp32_mn(const uint8_t* a, int64_t lda, const void* sfa,
                                 int64_t sfa_stride_m, int64_t sfa_stride_k,
                                 const uint8_t* b, int64_t ldb, const void* sfb,
                                 int64_t sfb_stride_n, int64_t sfb_stride_k,
                                 int fmt, float* d, int64_t ldd,
                                 int64_t m, int64_t n, int64_t k, int accumulate, ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_fp8_nn_bf16
 * gemm_fp8_nt_bf16 with B MN-major: B stored [k][n] (row stride ldb bytes),
 * D = A * B. For the data gradient dX = dY * W of "[Help] Starter script for
 * nn.Linear for fwd,bwd", B is W's own E4M3 cast [out, in] and its 128x128
 * block grid read transposed (sfb row r = block column r of W's grid), so no
 * cast of W^T is needed. sfb: [ceil(n/128), ceil(k/128)] at
 * sfb[r*sfb_stride_n + kb*sfb_stride_k] (packed UE8M0: words along K).
 * Requirements: as gemm_fp8_nt_bf16, with ldb >= n.
 * ------------------------------------------------------------------------- */
ql_status gemm_fp8_nn_bf16(const uint8_t* a, int64_t lda, const void* sfa,
                           int64_t sfa_stride_m, int64_t sfa_stride_k,
                           const uint8_t* b, int64_t ldb, const void* sfb,
                           int64_t sfb_stride_n, int64_t sfb_stride_k,
                           int fmt, uint16_t* d, int64_t ldd,
                           int64_t m, int64_t n, int64_t k, ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * ql_cast_gemm_host
 * The forward step of the linear layer ("[Help] Starter script for nn.Linear
 * for fwd,bwd": cast X per token, GEMM against W's block cast) with X and D
 * in HOST memory: D = bf16( fp8_cast_per_token(X, 128, fmt) * B^T ).
 *   x_host  bf16 [m, k] on the host, row stride ldx elements (pinned memory
 *           lets the copies overlap the kernels; pageable memory works).
 *   b, sfb  the device-resident E4M3 weight [n, k] and its 128x128 scales, as
 *           gemm_fp8_nt_bf16.
 *   d_host  bf16 [m, n] on the host, row stride ldd elements.
 *   chunk_rows  rows per pipeline step; workspace: caller-owned device memory
 *           of at least ql_cast_gemm_host_workspace_size(n, k, chunk_rows, fmt)
 *           bytes, 256-byte aligned (QL_ERR_INVALID_ARG / QL_ERR_ALIGNMENT).
 * Rows are copied in, cast, multiplied and copied out chunk by chunk, the
 * copies of one chunk overlapping the kernels of the next on three library
 * streams (created once per device) that start after the work already on
 * `stream` and that `stream` waits for at the end. The result equals the
 * device-buffer calls on the same data, bit for bit. Concurrent calls on one
 * device are serialised by a lock.
 * ------------------------------------------------------------------------- */
size_t ql_cast_gemm_host_workspace_size(int64_t n, int64_t k, int64_t chunk_rows, int fmt);
ql_status ql_cast_gemm_host(const void* x_host, int64_t ldx, const uint8_t* b, int64_t ldb,
                            const void* sfb, int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt,
                            uint16_t* d_host, int64_t ldd, int64_t m, int64_t n, int64_t k,
                            int64_t chunk_rows, void* workspace, size_t ws_bytes, ql_stream_t stream);

/* ---------------------------------------------------------------------------
 * ql_cast_gemm_host_noalloc
 * The pages have no counterpart to this call. It is ql_cast_gemm_host for
 * callers that cannot allocate device memory when they call it: a plug-in
 * inside an application whose device memory is all owned by the
 * application's own pool, or a serving process that makes no new device
 * allocation after warm-up so that its footprint stays fixed. Instead of a
 * caller-supplied workspace, the row chunks are staged in one array of
 * QL_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU that loads
 * the library holds that array until the process exits. The call allocates
 * nothing.
 *   Arguments as ql_cast_gemm_host without the workspace. chunk_rows must be
 *   small enough that ql_cast_gemm_host_workspace_size(n, k, chunk_rows, fmt)
 *   <= QL_NOALLOC_SCRATCH_BYTES, else QL_ERR_UNSUPPORTED (the call needs more
 *   staging than the array holds: pass fewer rows per chunk).
 *   The first call on a device looks up the array's device address and, if
 *   ql_cast_gemm_host has not run on that device yet, creates the pipeline's
 *   three streams and its events (driver objects, no device memory); make that
 *   first call before any stream capture.
 *   All calls share the array, and each call writes every staged byte before
 *   reading it, so nothing needs to start at zero. Calls ordered on one
 *   stream are safe; calls that overlap on the GPU (for example issued on two
 *   streams without ordering) race on the array and may corrupt each other's
 *   results.
 * ------------------------------------------------------------------------- */
#define QL_NOALLOC_SCRATCH_BYTES (64u << 20)
ql_status ql_cast_gemm_host_noalloc(const void* x_host, int64_t ldx, const uint8_t* b, int64_t ldb,
                                    const void* sfb, int64_t sfb_stride_n, int64_t sfb_stride_k, int fmt,
                                    uint16_t* d_host, int64_t ldd, int64_t m, int64_t n, int64_t k,
                                    int64_t chunk_rows, ql_stream_t stream);

/* The binary version (major * 10 + minor, 103 for sm_103a) of the kernel
 * image the CUDA runtime loaded for this library on the current device, from
 * cudaFuncGetAttributes; 0 if the runtime reports an error (no device, or no
 * image for it). A diagnostic: it launches nothing. */
int ql_binary_version(void);

/* Workspace bytes a GEMM of this shape needs (0 in this build). */
size_t ql_gemm_workspace_size(int64_t m, int64_t n, int64_t k);

/* ---------------------------------------------------------------------------
 * Knobs ("DeepGEMM Essentials" Part 15: get_num_sms / set_num_sms).
 * The GEMM's persistent grid uses at most this many SMs (default: all SMs of
 * the current device). ql_set_num_sms(n <= 0) restores the default.
 * The budget also decides whether a GEMM with few output tiles splits its K
 * blocks over a cluster, and over how many CTAs: that changes the grouping in
 * which fp32 partial sums are added, so results may differ in the last bit
 * of the output (within the GEMM tolerance). The setting is process-wide.
 * ------------------------------------------------------------------------- */
ql_status ql_set_num_sms(int num_sms);
int ql_get_num_sms(void);

/* Tile width (columns of D per tile) of the GEMM: 32, 64, 128 or 256; 0
 * (default) lets the library choose from the shape. Process-wide; meant for
 * tuning and for tests that exercise every tile width. */
ql_status ql_set_gemm_block_n(int block_n);

/* GEMM promotion path. With UE8M0 scale formats (QL_SF_UE8M0,
 * QL_SF_PACKED_UE8M0) the default (0) promotes inside the tensor core
 * (block-scaled MMA, one power-of-two scale per row and 32-wide K slice), on
 * CTA pairs (256 x 224 or 256 x 256 tiles over two SMs) when the problem has
 * at least one such tile per pair of SMs; with fewer tiles, split over K
 * across a thread-block cluster when that fills the SMs, else on CTA pairs
 * while there is a tile for every other pair, else on single SMs. With
 * QL_SF_FP32 scales the partial product of every 128-wide K block is
 * promoted on the CUDA cores: on one SM per tile or, for a plain GEMM with
 * bf16 output, at least 16 K blocks and too few 128 x 128 tiles to occupy
 * the SMs (small M), on a cluster of 2 or 4 CTAs that split the tile's K
 * blocks and sum their fp32 partials through distributed shared memory.
 * 1 and 6 force the CUDA-core promotion on one SM per tile (for any scale
 * format), 5 runs it on CTA pairs (256 x 256 tiles; plain GEMMs only,
 * measured no faster than one SM per tile) and 7 on the cluster split-K form
 * wherever a split applies (any number of K blocks); 2 forces
 * the single-SM block-scaled kernel, 3 the block-scaled CTA-pair kernel and 4
 * the block-scaled cluster split-K kernel where it applies (2-4 ignored for
 * QL_SF_FP32). All give results within the GEMM tolerance of each other.
 * Process-wide; for tuning and tests. */
ql_status ql_set_gemm_path(int path);

/* Time limit of every bounded wait inside the GEMM kernel, in milliseconds
 * (default 2000). After it runs out the kernel records QL_ERR_DEVICE_TIMEOUT,
 * drains its own copies, frees its tensor memory and returns. Process-wide. */
ql_status ql_set_wait_limit_ms(int ms);

/* Test hook for the failure path (process-wide, default off): while enabled,
 * the GEMM kernels' operand producer issues no copies, so the tensor-core
 * issuer's bounded wait runs out; the kernel then records
 * QL_ERR_DEVICE_TIMEOUT, frees its tensor memory and returns, leaving the
 * context usable. The output is not written. */
ql_status ql_test_stall_gemm_producer(int enable);

/* Synchronises `stream`, then returns and clears the device status word:
 * QL_OK; QL_ERR_DEVICE_TIMEOUT if any kernel's bounded wait ran out since the
 * last call; else QL_ERR_OUT_OF_BOUNDS if a bounds-checked build skipped an
 * access outside its buffer; else QL_ERR_INVALID_ARG if a grouped GEMM met an
 * invalid expert index; QL_ERR_CUDA if the synchronisation itself failed. */
ql_status ql_device_status(ql_stream_t stream);

/* ql_device_status, also returning the raw flag bits (1 time-out, 2 invalid
 * expert index, 4 out-of-bounds access) and the first out-of-bounds address a
 * bounds-checked build recorded (0 if none); either pointer may be null. */
ql_status ql_device_status_detail(ql_stream_t stream, uint32_t* flags, uint64_t* first_bad_address);

/* 1 if this library was built with QL_BOUNDS_CHECK: every plain global load
 * and store of the kernels (TMA copies are clipped by the hardware) is checked
 * against the byte range of the caller's buffer it belongs to, derived from
 * the call's pointers, shapes and strides; an access outside it is skipped
 * and recorded (QL_ERR_OUT_OF_BOUNDS from ql_device_status), never trapped.
 * A debugging build: slower, same results for in-range programs. 0 otherwise. */
int ql_bounds_checked(void);

#ifdef __cplusplus
}
#endif
#endif /* QLINEAR_H */
