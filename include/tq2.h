/*
 * tq2.h -- C ABI of the GB300-native ternary (TQ2_0-style) packed-weight
 * matvec library (libtq2_gb300.so, built for sm_103a).
 *
 * The operation (BitCPM ternary page, "TQ2_0 (llama.cpp)" paragraph and the
 * linear-factoring paragraph): along the reduction axis K, weights are split
 * into 256-element blocks; each weight is a 2-bit code q in {0,1,2} standing
 * for the value q-1 in {-1,0,+1}, and each block carries one fp16 scale d_b.
 * For every activation row m and output row n
 *
 *     y[m][n] = sum_b d[n][b] * sum_{k in b} x'[m][k] * (q[n][k] - 1)
 *
 * where x' = x, or the static int8 fake-quant of x ("gemma4 wNa8o8 requires
 * int8 activations" page): x' = s * clamp(rint(x * (1/s)), -128, 127).
 *
 * Data layout (all row-major, contiguous, caller-owned DEVICE memory):
 *   codes  int8   [N, K]        one code per element (pack input / unpack output)
 *   qs     uint8  [N, K/4]      code k of a row at bits 2*(k%4) of byte k/4
 *   d      fp16   [N, K/256]    block scales, IEEE binary16 bit patterns
 *   W      fp32 or fp16 [N, K]  a dequantised weight, W = d_b * (q - 1)
 *   x      fp16   [M, K]        activations, M in 0..16
 *   y      fp32 or fp16 [M, N]
 * K must be a multiple of 256 (one block); N >= 0.
 *
 * Conventions
 *   - Every call validates its arguments on the host and returns a status
 *     synchronously, before anything is enqueued.  Work is enqueued on the
 *     caller's stream and the call returns without synchronising; launch
 *     failures come back as TQ2_ERR_CUDA.
 *   - The library never allocates, frees or keeps device memory, and holds no
 *     state between calls: calls are safe from several host threads and on
 *     several streams.
 *   - Data-dependent conditions (a code outside {0,1,2}, non-finite or
 *     non-ternary W, a device wait that ran out) are reported by ORing flag
 *     bits into an optional caller-owned device word `d_status` (may be NULL);
 *     they never trap the GPU.  Nothing is truncated or clamped silently.
 *   - Pointers must not alias each other (except as stated).
 *   - Empty shapes (N == 0, M == 0, or K == 0 for pack/unpack/from_dense)
 *     are valid no-ops; with K == 0 the matvec writes y = 0 (empty sums).
 */
#ifndef TQ2_H
#define TQ2_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TQ2_API __attribute__((visibility("default")))
#else
#define TQ2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *tq2_stream_t;

typedef enum {
    TQ2_OK = 0,
    TQ2_ERR_NULL = 1,    /* a required pointer is NULL (with a non-empty shape) */
    TQ2_ERR_SHAPE = 2,   /* K % 256 != 0, a negative size, M > 16, or size overflow */
    TQ2_ERR_ALIGN = 3,   /* a pointer is not aligned as documented */
    TQ2_ERR_DTYPE = 4,   /* unknown tq2_dtype value */
    TQ2_ERR_ARG = 5,     /* act_scale negative / not finite, unknown impl, ... */
    TQ2_ERR_CUDA = 6,    /* a CUDA runtime call or kernel launch failed */
    TQ2_ERR_TIMEOUT = 7  /* reserved: reported through TQ2_FLAG_TIMEOUT */
} tq2_status;

typedef enum { TQ2_F32 = 0, TQ2_F16 = 1 } tq2_dtype;

/* Flag bits ORed (asynchronously, by the kernels) into *d_status. */
#define TQ2_FLAG_BAD_CODE 1u  /* pack: a code not in {0,1,2}; stored as code & 3 */
#define TQ2_FLAG_NONFINITE 2u /* from_dense: NaN/Inf in W, or max|W| overflows fp16 */
#define TQ2_FLAG_INEXACT 4u   /* from_dense: some W != d*(code-1) (lossy recovery) */
#define TQ2_FLAG_TIMEOUT 8u   /* matvec: a bounded device wait ran out; y is invalid */
#define TQ2_FLAG_BOUNDS 16u   /* debug builds (TQ2_BOUNDS_CHECK) only: a kernel computed an index
                                 outside its buffer and skipped that access; the result is invalid */

/*
 * tq2_pack -- codes int8 [N,K] -> qs uint8 [N,K/4].
 * BitCPM ternary page, "TQ2_0 (llama.cpp)" paragraph: 2-bit codes {0,1,2}.
 * Byte j of row n holds codes 4j..4j+3 at bits 0-1, 2-3, 4-5, 6-7.
 * A code outside {0,1,2} is stored as (code & 3) and sets TQ2_FLAG_BAD_CODE.
 * Alignment: none required.  The scale array is not touched: it is passed
 * unchanged to tq2_matvec in its [N, K/256] layout.
 */
TQ2_API tq2_status tq2_pack(const int8_t *codes, int64_t N, int64_t K, uint8_t *qs,
                    uint32_t *d_status, tq2_stream_t stream);

/*
 * tq2_unpack -- qs uint8 [N,K/4] -> codes int8 [N,K], every 2-bit field
 * returned as stored (3 included).  Inverse of tq2_pack on valid codes.
 */
TQ2_API tq2_status tq2_unpack(const uint8_t *qs, int64_t N, int64_t K, int8_t *codes,
                      tq2_stream_t stream);

/*
 * tq2_from_dense -- recover (qs, d) from a dequantised W [N,K]
 * (BitCPM ternary page, recovery paragraph: d_block = max|W| in the block,
 * exact because the nonzero magnitude is d; code = round(W/d) + 1).
 * w_dtype: TQ2_F32 (float) or TQ2_F16 (binary16 bits).
 * d is the fp16 round-to-nearest-even of the block's max|W|; codes are
 * rint(W/d) (one fp32 division by the stored d, ties to even) clamped to
 * [-1,1], plus 1.  An all-zero block gives d = 0 and codes 1; an element whose
 * W/d is NaN gets code 1.  Flags: TQ2_FLAG_NONFINITE, TQ2_FLAG_INEXACT.
 * For a true TQ2_0 W (W = d*(q-1), fp16 d, a nonzero code in the block) the
 * recovery is bit-exact and sets no flag.
 * Alignment: W 4-byte (fp32) or 2-byte (fp16) aligned.
 */
TQ2_API tq2_status tq2_from_dense(const void *W, tq2_dtype w_dtype, int64_t N, int64_t K,
                          uint8_t *qs, uint16_t *d, uint32_t *d_status,
                          tq2_stream_t stream);

/*
 * tq2_matvec -- y[M,N] = x'[M,K] (ternary W)^T, M in 0..16.
 * BitCPM ternary page, linear-factoring paragraph:
 *   sum_k x_k d_b (q_k - 1) = sum_b d_b sum_{k in b} x_k (q_k - 1).
 * act_scale: 0 disables the prologue ("scale 0 = unquantized"); s > 0 applies
 * the static int8 fake-quant of the gemma4 wNa8o8 page to x first, with the
 * integer decision taken as rint(fp32(x) * fp32(1/s)) (ties to even, NaN -> 0)
 * and the product kept as code * s (no fp16 re-rounding).
 * y_dtype: TQ2_F32, or TQ2_F16 (round to nearest even from the fp32 sum).
 * Accuracy: |y - exact| <= 1e-3 * sum_k |d_b x'_k| + 1e-6 per element; the
 * result is bit-identical from run to run.
 * Alignment: x and qs 16-byte aligned; d 2-byte; y 4-byte (fp32) / 2-byte.
 * workspace / workspace_bytes: optional device scratch (workspace_bytes 0:
 * none; else workspace non-NULL (TQ2_ERR_NULL) and 16-byte aligned
 * (TQ2_ERR_ALIGN)).  With act_scale > 0 and a workspace, the call may run
 * the prologue as a pass of its own: x is converted once into the workspace
 * (2 M K bytes: the codes as fp16) and the kernel reads the codes, instead
 * of every CTA converting the x it reads.  It does so where that was
 * measured faster: with the tcgen05 GEMM for N > 512 or M > 64, and with
 * the pre-scaled kernel (impl 4) for M >= 9 and K >= 8192; with a
 * workspace the automatic choice also takes the GEMM for M = 8 when
 * K >= 8192 and N > 512.  A workspace smaller than the pass needs is then
 * TQ2_ERR_ARG (nothing enqueued).  A kernel gives the same bits either
 * way (the codes are those it would compute itself).  The workspace must not overlap x, qs, d or y;
 * it is written and read by the call's kernels in stream order, so a
 * workspace may be reused by the next call on the same stream, but not by
 * calls that may run concurrently (other streams) until this one is done.
 * d_status: optional; TQ2_FLAG_TIMEOUT is set if a bounded device wait ran
 * out (y is then invalid).
 * Weights and scales are prefetched before the kernel waits on the previous
 * kernel in the stream (programmatic dependent launch): qs and d must not be
 * written by the kernel that immediately precedes this call on the stream
 * when that kernel is itself one of this library's products (tq2_matvec,
 * tq2_matvec_impl, tq2_matvec_requant, tq2_matvec_grouped, tq2_gemm,
 * tq2_affine4_matvec), which let the next kernel start early.
 */
TQ2_API tq2_status tq2_matvec(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                      int64_t N, int64_t K, void *y, tq2_dtype y_dtype, float act_scale,
                      void *workspace, size_t workspace_bytes, uint32_t *d_status,
                      tq2_stream_t stream);

/* Largest number of weight matrices in one tq2_matvec_grouped call. */
#define TQ2_MAX_GROUP 4

/*
 * tq2_matvec_grouped -- several matvecs that share x and K (in a decoder
 * layer: q, k and v of the attention input; gate and up of the MLP input),
 * BitCPM ternary page, linear-factoring paragraph, applied to each matrix:
 *   y_j[m][n] = sum_b d_j[n][b] * sum_{k in b} x'[m][k] * (q_j[n][k] - 1).
 *
 *   x          device, fp16 [M, K] row-major, 16-byte aligned, read only.
 *   M, K       as tq2_matvec (M in 0..16, K % 256 == 0).
 *   n_mats     1 .. TQ2_MAX_GROUP.
 *   qs, d, N, y  HOST arrays of n_mats entries (read during the call, not
 *              kept): device pointers to qs_j [N_j, K/4] (16-byte aligned),
 *              d_j [N_j, K/256] fp16, y_j [M, N_j] (y_dtype; 4- or 2-byte
 *              aligned), and the row counts N_j >= 0 (N_j = 0: y_j untouched).
 *   y_dtype, act_scale, d_status, stream  as tq2_matvec (one act_scale for
 *              the shared x).
 *   workspace, workspace_bytes  optional, as for tq2_matvec; the size from
 *              tq2_matvec_grouped_workspace_size.
 *
 * Results equal n_mats tq2_matvec calls with the same x.  They run as ONE
 * kernel launch (the CTAs split between the matrices in proportion to their
 * rows; x staged and the wait on the previous kernel paid once) when M <= 2
 * (the class-column kernel, any K); when 3 <= M <= 8 and each matrix alone
 * would run the pre-scaled kernel (not the GEMM; any K); and when
 * 9 <= M <= 16, K < 8192 and either M <= 11 or some matrix has N_j <= 512
 * (the pre-scaled kernel: q/k/v at M = 9..16 in 8.8-12.1 us against
 * 21.6-22.8 us as separate calls on GB300).  Otherwise they run as
 * consecutive calls on the stream.  In that case, with act_scale > 0 and a
 * workspace, x is fake-quantised ONCE into the workspace for all the
 * matrices (the recipe's one input quantisation shared by q/k/v, and by
 * gate/up), and each call reads the codes; each kernel gives the same bits
 * as converting x itself, but with a workspace a matrix's single call may
 * take the GEMM where it otherwise would not (as for tq2_matvec).  Errors:
 * as tq2_matvec for every matrix (checked before anything is enqueued);
 * TQ2_ERR_ARG for n_mats out of range or a workspace smaller than the pass
 * needs; TQ2_ERR_NULL for a NULL array.
 */
TQ2_API tq2_status tq2_matvec_grouped(const uint16_t *x, int64_t M, int64_t K, int n_mats,
                                      const uint8_t *const *qs, const uint16_t *const *d,
                                      const int64_t *N, void *const *y, tq2_dtype y_dtype,
                                      float act_scale, void *workspace, size_t workspace_bytes,
                                      uint32_t *d_status, tq2_stream_t stream);

/* Bytes of workspace with which tq2_matvec_grouped (and _requant) converts x
 * once for the group (2 M K: when the matrices run as consecutive calls,
 * M >= 3), or 0 (also for invalid arguments).  N: HOST array of n_mats row
 * counts. */
TQ2_API size_t tq2_matvec_grouped_workspace_size(int64_t M, int64_t K, int n_mats, const int64_t *N);

/*
 * tq2_matvec_grouped_requant -- tq2_matvec_grouped with the static int8
 * requantisation of each matrix's result at store, with that matrix's own
 * output scale ("gemma4 wNa8o8 requires int8 activations" page, the recipe:
 * one input quantisation shared by q/k/v and by gate/up, each linear's
 * output requantised with its own output_activation_scale).
 *   out_scale  HOST array of n_mats scales (read during the call, not kept);
 *              each >= 0 and finite, else TQ2_ERR_ARG; 0 stores that
 *              matrix's y unchanged.  NULL: TQ2_ERR_NULL.
 * y_j is what tq2_matvec_requant(..., out_scale[j], ...) stores; everything
 * else as tq2_matvec_grouped.
 */
TQ2_API tq2_status tq2_matvec_grouped_requant(const uint16_t *x, int64_t M, int64_t K, int n_mats,
                                              const uint8_t *const *qs, const uint16_t *const *d,
                                              const int64_t *N, void *const *y, tq2_dtype y_dtype,
                                              float act_scale, const float *out_scale, void *workspace,
                                              size_t workspace_bytes, uint32_t *d_status, tq2_stream_t stream);

/* Bytes of workspace with which tq2_matvec runs the prologue as a pass of
 * its own for this shape (2 M K), or 0 where it would not use one (and for
 * invalid shapes).  tq2_matvec_impl with impl 4 or 6 may use one where
 * tq2_matvec does not: 2 M K bytes (tq2_gemm_workspace_size) suffice for
 * every impl. */
TQ2_API size_t tq2_matvec_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * tq2_matvec_impl -- tq2_matvec with an explicit kernel choice, for
 * measurement: impl 0 = automatic (what tq2_matvec runs), 1 = warp-level
 * tensor cores with one accumulator per code class (mma.sync on masked code
 * words, TMA-staged weights), 2 = CUDA cores (fp32 FMA per code),
 * 4 = warp-level
 * tensor cores with x pre-scaled per code class (one accumulator whose 8
 * columns are 8 activation rows), 6 = the tcgen05 GEMM of tq2_gemm
 * (5th-generation tensor cores, an MMA of 128 weight rows x 16 activation
 * rows), 7 = CUDA cores for a few output rows per CTA (k/v-sized N: codes and
 * scales in registers before the wait on the previous kernel, one
 * reduction).  Impls 1 and 7 take M <= 2 (impl 7 also K <= 16384 and at most
 * 4 rows per CTA, one CTA per SM), impl 4 takes M <= 16;
 * outside their range they return TQ2_ERR_ARG.  Numbers 3 (a tcgen05
 * matvec) and 5 (a dp4a matvec) are retired: both were slower than impl 1 on
 * every shape, and they now return TQ2_ERR_ARG (the numbers are not reused).
 * Same contract as tq2_matvec otherwise.
 */
TQ2_API tq2_status tq2_matvec_impl(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                           int64_t N, int64_t K, void *y, tq2_dtype y_dtype, float act_scale,
                           void *workspace, size_t workspace_bytes, uint32_t *d_status,
                           tq2_stream_t stream, int impl);

/*
 * tq2_matvec_requant -- tq2_matvec_impl followed by the static int8
 * requantisation of the result at store ("gemma4 wNa8o8 requires int8
 * activations" page, "Implemented": fake-quant at every linear boundary,
 * input post-norm and output at store; the recipe's "requantize the result
 * to int8 with output_activation_scale -> dequantize").  With act_scale > 0
 * the block sums are exact integer sums of int8 codes times ternary weights
 * (int8 x ternary -> exact accumulate), and the stored result is
 *   y'[m][n] = out_scale * clamp(rint(y[m][n] * (1/out_scale)), -128, 127)
 * where y[m][n] is the fp32 result tq2_matvec_impl would store before its
 * dtype conversion, the integer decision is taken in fp32 with
 * fp32(1/out_scale) (ties to even; NaN -> 0, +-Inf saturate), and the
 * product code * out_scale is rounded once to fp32, then to y_dtype (RNE).
 *   out_scale  >= 0 and finite, else TQ2_ERR_ARG; 0 stores y unchanged
 *              (the call is then tq2_matvec_impl).
 * Everything else (arguments, impl, errors, accuracy of y before the
 * requantisation) as tq2_matvec_impl.  A code may differ by one from the
 * one of the exact y only where y lies within the accuracy bound of a
 * rounding boundary.
 */
TQ2_API tq2_status tq2_matvec_requant(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                                      int64_t N, int64_t K, void *y, tq2_dtype y_dtype, float act_scale,
                                      float out_scale, void *workspace, size_t workspace_bytes,
                                      uint32_t *d_status, tq2_stream_t stream, int impl);

/*
 * tq2_gemm -- the same product for any number of activation rows (prefill:
 * a prompt's tokens at once), BitCPM ternary page, linear-factoring paragraph:
 *   y[m][n] = sum_b d[n][b] * sum_{k in b} x'[m][k] * (q[n][k] - 1),
 * m < M, with the optional prologue (act_scale) and output requantisation
 * (out_scale) of tq2_matvec_requant.
 *   x          device, fp16 [M, K] row-major, 16-byte aligned, read only.
 *   M          >= 0 (up to 2^30); qs, d, N, K, y, y_dtype, act_scale,
 *              out_scale, workspace, workspace_bytes, d_status, stream as
 *              tq2_matvec_requant (y [M, N]; the workspace size from
 *              tq2_gemm_workspace_size).
 *   impl       0 = automatic, 1 = the tcgen05 GEMM (5th-generation tensor
 *              cores: weights expanded once per 128-row tile into exact fp16
 *              (q - 1) * d_b in tensor memory, x tiles by TMA, fp32
 *              accumulation over all of K; without a workspace the
 *              prologue fake-quantises each x tile in shared memory, in
 *              every weight tile), 2 = the matvec kernels on 16-row
 *              slices of x.  Automatic takes the GEMM for M > 16, the slices
 *              otherwise.
 * Errors and accuracy as tq2_matvec (TQ2_ERR_SHAPE for M out of range;
 * TQ2_ERR_ARG for impl out of range or a shape impl 1 cannot plan).
 */
TQ2_API tq2_status tq2_gemm(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N,
                            int64_t K, void *y, tq2_dtype y_dtype, float act_scale, float out_scale,
                            void *workspace, size_t workspace_bytes, uint32_t *d_status, tq2_stream_t stream,
                            int impl);

/* Bytes of workspace with which tq2_gemm runs the prologue as a pass of its
 * own (2 M K: enough for every impl), or 0 for an invalid shape. */
TQ2_API size_t tq2_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * tq2_gemm_static_ws -- tq2_gemm for callers that must not allocate: the
 * workspace of the prologue's pass is a static device array inside this
 * library (16 MiB per device: the codes of M x K <= 2^23 activations).
 * None of the pages has a counterpart: this is an interface convenience
 * around the same kernels, with the same results bit for bit as tq2_gemm
 * given a workspace of tq2_gemm_workspace_size bytes.
 *   Arguments, results and errors as tq2_gemm without the workspace
 *   arguments; in addition, with act_scale > 0 and M x K > 2^23:
 *   TQ2_ERR_SHAPE (nothing enqueued; tq2_gemm with a workspace of the
 *   caller's has no such limit).
 * Set-up: the first call with act_scale > 0 on a device takes the array's
 * address there (cudaGetSymbolAddress, which may load the library's module;
 * its failure returns TQ2_ERR_CUDA) and keeps it; make that first call before
 * capturing a stream into a CUDA graph.  A later cudaDeviceReset invalidates
 * the kept address: do not use this call after one.
 * Nothing here allocates, and nothing in the array needs to start at zero:
 * each call writes every code it reads before reading it.
 * Concurrency: calls on one stream are ordered (each call's pass waits for
 * the previous kernel on the stream before it writes); calls that may
 * overlap -- on different streams, or from several host threads without
 * stream order between them -- race on the one array and must not be made.
 */
TQ2_API tq2_status tq2_gemm_static_ws(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N,
                                      int64_t K, void *y, tq2_dtype y_dtype, float act_scale, float out_scale,
                                      uint32_t *d_status, tq2_stream_t stream, int impl);

/*
 * tq2_affine4_matvec -- the affine-int4 sibling on the same skeleton
 * ("Custom Metal kernels" page, the note on asymmetric (zero-point) int4: a
 * fused affine-int4 matvec factors the zero point out, acc += s * (dot -
 * z * sum x)):
 *   y[m][n] = sum_g s[n][g] * (sum_{k in g} x[m][k] q[n][k]
 *                              - z[n][g] * sum_{k in g} x[m][k]),
 * i.e. y = W x with W[n][k] = s[n][k/G] * (q[n][k] - z[n][k/G]).
 *   x          device, fp16 [M, K] row-major, 16-byte aligned, read only.
 *   M          0 .. 16 activation rows (two per kernel launch).
 *   qs         device, uint8 [N, K/2]: 4-bit codes q in 0..15, code k of a
 *              row in byte k/2 at bits 4*(k%2) (low nibble first); 16-byte
 *              aligned, read only.
 *   s, z       device, fp16 [N, K/G]: the scale and the zero point (in code
 *              units, any fp16 value) of each group of G codes; 16-byte
 *              aligned, read only.
 *   N, K       N >= 0, K >= 0 with K % 256 == 0 (K % G == 0 follows).
 *   G          64, 128 or 256, else TQ2_ERR_ARG.
 *   y, y_dtype device [M, N] fp32 (TQ2_F32) or fp16 (TQ2_F16, round to
 *              nearest even), 4- or 2-byte aligned, written.
 *   d_status   optional device word; TQ2_FLAG_TIMEOUT if a bounded wait ran
 *              out (y is then invalid).
 *   stream     caller's CUDA stream; the call enqueues and returns.
 * Accuracy: |y - exact| <= 1e-3 * sum_g |s_g| sum_{k in g} |x_k| (q_k +
 * |z_g|) + 1e-6 per element (the magnitude of the two factored sums, which
 * the fp32 accumulation error scales with).  Deterministic run to run.
 * As tq2_matvec, qs, s and z are read before the wait on the previous kernel
 * in the stream: the immediately preceding kernel, if one of this library's,
 * must not write them.
 * Errors: as tq2_matvec (TQ2_ERR_SHAPE, _NULL, _ALIGN, _DTYPE, _CUDA);
 * TQ2_ERR_ARG for G, or a K too long for the x staging to fit in shared
 * memory (x of two activation rows is staged whole: K up to ~90,000 for one
 * row, ~45,000 for two).  M = 0 or N = 0: nothing is done; K = 0: y = 0.
 */
TQ2_API tq2_status tq2_affine4_matvec(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *s,
                                      const uint16_t *z, int64_t N, int64_t K, int64_t G, void *y,
                                      tq2_dtype y_dtype, uint32_t *d_status, tq2_stream_t stream);

/*
 * tq2_test_matvec_stall -- a test hook, not part of the product (the pages
 * have no counterpart): tq2_matvec_impl with impl 1 and fp32 y, except that
 * in every CTA the weight producer skips the copy of pipeline stage
 * stall_stage, and every bounded device wait gives up after wait_limit_us
 * microseconds instead of the normal 200 ms.  The consumers' wait for the
 * skipped stage therefore runs out: the kernel sets TQ2_FLAG_TIMEOUT in
 * *d_status, waits (bounded) for the copies it did issue, and returns
 * without storing y.  A test uses it to check that the timeout path reports
 * the failure and leaves the context usable (the next call is correct).
 *   stall_stage  >= 0, else TQ2_ERR_ARG; a stage index past a CTA's last
 *                stage skips nothing in that CTA.
 *   wait_limit_us  1 .. 200000, else TQ2_ERR_ARG.
 *   d_status   required (TQ2_ERR_NULL if NULL), 4-byte aligned.
 *   Other arguments and errors as tq2_matvec_impl with impl 1 (M <= 2,
 *   TQ2_ERR_ARG for a shape impl 1 cannot plan).  The call takes about two
 *   wait limits on the device.
 */
TQ2_API tq2_status tq2_test_matvec_stall(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                                         int64_t N, int64_t K, float *y, uint32_t *d_status,
                                         tq2_stream_t stream, int stall_stage, int wait_limit_us);

/*
 * tq2_test_gemm_stall -- a test hook, not part of the product (the pages
 * have no counterpart): tq2_gemm with impl 1 (the tcgen05 GEMM) and fp32 y,
 * except that in every CTA the x producer skips the copy of its stage
 * stall_stage (stages of 8 k-steps, counted within the CTA's share of K),
 * and every wait of the stage rings gives up after wait_limit_us
 * microseconds instead of 200 ms (the waits for the MMAs' completion, which
 * guard the release of tensor memory, and the split-K hand-off waits keep
 * 200 ms).  The MMA issuer's wait for that stage runs out: the kernel sets
 * TQ2_FLAG_TIMEOUT in *d_status, drains its copies and MMAs, frees its tensor
 * memory and returns without storing y.
 *   stall_stage, wait_limit_us, d_status  as tq2_test_matvec_stall.
 *   act_scale  as tq2_gemm (> 0 also runs the in-place x conversion, whose
 *              wait runs out too).
 *   Other arguments and errors as tq2_gemm with impl 1 (TQ2_ERR_ARG for a
 *   shape the GEMM cannot plan).  The call takes a few wait limits.
 */
TQ2_API tq2_status tq2_test_gemm_stall(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                                       int64_t N, int64_t K, float *y, float act_scale, uint32_t *d_status,
                                       tq2_stream_t stream, int stall_stage, int wait_limit_us);

/*
 * tq2_trace_size, tq2_trace_read -- diagnostics of the trace build (the
 * library compiled with TQ2_TRACE; the pages have no counterpart).  That
 * build's class-column kernel (impl 1, single calls) stamps the GPU's
 * globaltimer (ns) per CTA at 8 phase points into a static device array of
 * two slots, which consecutive launches use in turn (launch parity; in a
 * CUDA graph, the parity of the capture order): [slot 2][CTA 1024][phase 8]
 * uint64, phases 0 entry, 1 the wait on the previous kernel returned, 2 x
 * staged, 3 the first stage's codes read, 4 the stage loop done, 5 y stored,
 * 6 the producer's last copy issued, 7 unused.  Only CTAs below 1024 stamp.
 *   tq2_trace_size  the array's size in bytes; 0 in other builds.
 *   tq2_trace_read  copies it to host_dst (host memory, at least
 *                   tq2_trace_size() bytes), synchronously after the device's
 *                   work; TQ2_ERR_ARG in other builds or for a smaller
 *                   buffer, TQ2_ERR_NULL for a NULL pointer.
 * The stamps cost about 0.3 us per call; time nothing with the trace build.
 */
TQ2_API size_t tq2_trace_size(void);
TQ2_API tq2_status tq2_trace_read(void *host_dst, size_t bytes);

/* The CUDA error behind the most recent TQ2_ERR_CUDA returned to the calling
 * host thread ("no error" if none): name and description, static storage. */
TQ2_API const char *tq2_last_cuda_error(void);

/* Static, human-readable name of a status. */
TQ2_API const char *tq2_status_string(tq2_status status);

/* Library version, 10000*major + 100*minor + patch. */
TQ2_API int tq2_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ2_H */
