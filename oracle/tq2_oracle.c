/*
 * tq2_oracle.c -- plain, slow CPU oracle for the TQ2_0-style ternary matvec
 * (and its affine-int4 sibling).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product (the CUDA
 * library under quantized_gemv_tq2_gb300/) never calls it, and the two share
 * no code: no headers, no helpers, no tables.
 *
 * Every loop here follows the definition on the pages, one element at a
 * time, in the order the definition states it.  Sources:
 *   [P1] "BitCPM-CANN-8B -> Core AI, ternary 1.58-bit" (coreai-model-zoo
 *        knowledge page bitcpm-ternary-1.58bit): the TQ2_0 format paragraph
 *        (2-bit code q in {0,1,2} meaning q-1, one fp16 scale d per 256-element
 *        block along K), the recovery paragraph (d = max|W| in the block,
 *        code = round(W/d)+1), and the linear-factoring identity
 *        sum_k x_k d_b (q_k-1) = sum_b d_b sum_{k in b} x_k (q_k-1).
 *   [P2] "Custom Metal kernels" (coreai-model-zoo knowledge page
 *        custom-metal-kernels): the note on asymmetric (zero-point) int4,
 *        whose fused matvec factors the zero point out,
 *        acc += s * (dot - z * sum x).
 *   [P3] "gemma4 wNa8o8 requires int8 activations" (coreai-model-zoo
 *        knowledge page): the static fake-quant clamp(round(x/s),-128,127)*s,
 *        its implemented form s*clamp(rint(x*(1/s)),-128,127) ("Implemented"
 *        section), and the reciprocal-multiply note ("Two transferable
 *        engineering notes").
 * Readings where the pages are silent (the byte order of the packed codes,
 * code 3, an all-zero block, ties, NaN) are stated next to the code that
 * takes them.
 *
 * Parity pins: every function below is pinned by the CPU tests against
 * closed forms, invariants, brute force or an independent library
 * (numpy); nothing here is "parity unpinned".
 *
 * Build: plain C99 + the GCC/Clang __int128 extension, -O2 -ffp-contract=off
 * (no fused multiply-add: the fp32 decisions must round every operation).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define TQ2O_FLAG_BAD_CODE 1u
#define TQ2O_FLAG_NONFINITE 2u
#define TQ2O_FLAG_INEXACT 4u

/* ---------------------------------------------------------------------- */
/* IEEE 754 binary16, written from the format's definition.               */
/* ---------------------------------------------------------------------- */

/* Value of a binary16 bit pattern: sign, 5-bit biased exponent (bias 15),
 * 10-bit fraction; exponent 0 is the subnormal range m * 2^-24. */
double tq2o_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even (the IEEE default). */
uint16_t tq2o_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v))
        return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0) /* halfway between 65504 and 2^16 rounds up to Inf */
        return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal: count units of 2^-24; rint rounds half to even. The
         * result 1024 is exactly the smallest normal's bit pattern. */
        double q = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int E;
    double f = frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    double q = rint(ldexp(f, 11)); /* 11 significant bits, in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    int ebits = (E - 1) + 15;
    if (ebits >= 31)
        return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(ebits << 10) | (uint16_t)((int)q - 1024));
}

/* A finite binary16 value as an integer count of 2^-24 (|result| < 2^40).
 * Returns 0 and sets *ok = 0 for Inf/NaN. */
static int64_t half_to_units(uint16_t h, int *ok)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int64_t m = h & 0x3ff;
    int64_t u;
    if (e == 31) {
        *ok = 0;
        return 0;
    }
    if (e == 0)
        u = m;
    else
        u = (1024 + m) << (e - 1);
    return sign ? -u : u;
}

/* ---------------------------------------------------------------------- */
/* Packed layout [P1, TQ2_0 format].  The pages do not print the byte      */
/* order; this library's reading: code k of a row sits in byte k/4 at bits */
/* 2*(k%4) .. 2*(k%4)+1, rows are K/4 bytes, row-major [N, K/4].           */
/* ---------------------------------------------------------------------- */

/* codes [N,K] int8 -> qs [N,K/4].  A code outside {0,1,2} is stored as
 * (code & 3) and raises TQ2O_FLAG_BAD_CODE (the pages list only 0,1,2). */
uint32_t tq2o_pack(const int8_t *codes, int64_t N, int64_t K, uint8_t *qs)
{
    uint32_t flags = 0;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t j = 0; j < K / 4; ++j) {
            unsigned byte = 0;
            for (int i = 0; i < 4; ++i) {
                int8_t c = codes[n * K + 4 * j + i];
                if (c < 0 || c > 2)
                    flags |= TQ2O_FLAG_BAD_CODE;
                byte |= ((unsigned)(uint8_t)c & 3u) << (2 * i);
            }
            qs[n * (K / 4) + j] = (uint8_t)byte;
        }
    }
    return flags;
}

/* qs [N,K/4] -> codes [N,K] int8 (every 2-bit field, 3 included). */
void tq2o_unpack(const uint8_t *qs, int64_t N, int64_t K, int8_t *codes)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (int8_t)((qs[n * (K / 4) + k / 4] >> (2 * (k % 4))) & 3);
}

/* One code from the packed matrix. */
static int code_at(const uint8_t *qs, int64_t K, int64_t n, int64_t k)
{
    return (qs[n * (K / 4) + k / 4] >> (2 * (k % 4))) & 3;
}

/* Dequantised weight W[n,k] = d_b * (q - 1) in fp32 (exact for q in {0,1,2}:
 * the product is +-d or 0) [P1, TQ2_0 format]. */
void tq2o_dequant(const uint8_t *qs, const uint16_t *d, int64_t N, int64_t K, float *W)
{
    int64_t B = K / 256;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            double db = tq2o_half_to_double(d[n * B + k / 256]);
            W[n * K + k] = (float)(db * (double)(code_at(qs, K, n, k) - 1));
        }
}

/* ---------------------------------------------------------------------- */
/* Recovery from a dequantised W [P1, recovery paragraph]:                 */
/*   d_block = max |W| over the block, code = round(W / d) + 1.            */
/* Readings: d is stored as fp16 (round to nearest even from the fp32       */
/* maximum); the division uses that stored d, in fp32 (the pages work on    */
/* fp32 numpy/torch tensors), rounding half to even (torch.round /          */
/* numpy.round), clamped to [-1, 1].  d == 0 (all-zero block): every code   */
/* is 1.  W/d that is NaN (NaN in W, Inf/Inf): code 1.  Flags: NONFINITE    */
/* for NaN/Inf in W or a maximum that overflows fp16; INEXACT when some     */
/* W != d*(code-1) (recovery was lossy).                                    */
/* ---------------------------------------------------------------------- */
static uint32_t from_dense_block(const float *w, uint8_t *qrow, int64_t k0, uint16_t *dout)
{
    uint32_t flags = 0;
    float amax = 0.0f;
    for (int i = 0; i < 256; ++i) {
        float v = w[i];
        if (!isfinite(v))
            flags |= TQ2O_FLAG_NONFINITE;
        float a = fabsf(v);
        if (a > amax) /* NaN compares false and is skipped */
            amax = a;
    }
    uint16_t dh = tq2o_double_to_half((double)amax);
    float dv = (float)tq2o_half_to_double(dh);
    if (!isfinite(dv))
        flags |= TQ2O_FLAG_NONFINITE;
    *dout = dh;
    for (int i = 0; i < 256; ++i) {
        float v = w[i];
        int code;
        if (dv == 0.0f) {
            code = 1;
        } else {
            volatile float r = v / dv; /* one fp32 division, rounded */
            if (isnan(r)) {
                code = 1;
            } else {
                float rr = rintf(r);
                if (rr < -1.0f)
                    rr = -1.0f;
                if (rr > 1.0f)
                    rr = 1.0f;
                code = (int)rr + 1;
            }
        }
        volatile float back = dv * (float)(code - 1);
        if (!(back == v))
            flags |= TQ2O_FLAG_INEXACT;
        int64_t k = k0 + i;
        uint8_t *byte = &qrow[k / 4];
        int sh = 2 * (int)(k % 4);
        *byte = (uint8_t)((*byte & ~(3u << sh)) | ((unsigned)code << sh));
    }
    return flags;
}

uint32_t tq2o_from_dense_f32(const float *W, int64_t N, int64_t K, uint8_t *qs, uint16_t *d)
{
    uint32_t flags = 0;
    int64_t B = K / 256;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < B; ++b)
            flags |= from_dense_block(W + n * K + b * 256, qs + n * (K / 4), b * 256, &d[n * B + b]);
    return flags;
}

uint32_t tq2o_from_dense_f16(const uint16_t *W, int64_t N, int64_t K, uint8_t *qs, uint16_t *d)
{
    uint32_t flags = 0;
    int64_t B = K / 256;
    float blk[256];
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < B; ++b) {
            for (int i = 0; i < 256; ++i) /* fp16 -> fp32 is exact */
                blk[i] = (float)tq2o_half_to_double(W[n * K + b * 256 + i]);
            flags |= from_dense_block(blk, qs + n * (K / 4), b * 256, &d[n * B + b]);
        }
    return flags;
}

/* ---------------------------------------------------------------------- */
/* Static int8 activation fake-quant [P3].                                 */
/* The definition is clamp(round(x/s), -128, 127) * s.  The pages'         */
/* implemented form takes the integer decision as rint(x * (1/s)) in fp32   */
/* (reciprocal multiply; "Implemented" and the engineering notes).  Both    */
/* are provided; the matvec below uses the implemented fp32 form, the       */
/* precision in which the CUDA path takes the same decision.  NaN -> 0.     */
/* ---------------------------------------------------------------------- */
static int clamp_i8(double r)
{
    if (isnan(r))
        return 0;
    if (r < -128.0)
        return -128;
    if (r > 127.0)
        return 127;
    return (int)r;
}

/* Integer code of one fp16 activation: rint(fp32(x) * fp32(1/s)), in fp32. */
static int fq_code_recip_f32(uint16_t xh, float s)
{
    volatile float inv = 1.0f / s;
    volatile float xf = (float)tq2o_half_to_double(xh);
    volatile float t = xf * inv;
    return clamp_i8((double)rintf(t));
}

/* Integer code by the definition, rint(x / s) in fp64. */
static int fq_code_div_f64(uint16_t xh, float s)
{
    double t = tq2o_half_to_double(xh) / (double)s;
    return clamp_i8(rint(t));
}

/* Integer codes [n] of the fake-quant.  mode 0: the implemented fp32
 * reciprocal form; mode 1: the fp64 divide form of the definition. */
void tq2o_fakequant_codes(const uint16_t *x, int64_t n, float s, int mode, int8_t *q)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = (int8_t)(mode == 0 ? fq_code_recip_f32(x[i], s) : fq_code_div_f64(x[i], s));
}

/* Fake-quantised activations x' = q * s in fp64, for the given mode. */
void tq2o_fakequant(const uint16_t *x, int64_t n, float s, int mode, double *xq)
{
    for (int64_t i = 0; i < n; ++i) {
        int q = mode == 0 ? fq_code_recip_f32(x[i], s) : fq_code_div_f64(x[i], s);
        xq[i] = (double)q * (double)s;
    }
}

/* ---------------------------------------------------------------------- */
/* Static int8 output requantisation at store [P3]: the fake-quant at a     */
/* linear's output boundary ("Implemented": fake-quant at every linear      */
/* boundary, input post-norm and output at store; the recipe's "requantize  */
/* the result to int8 with output_activation_scale -> dequantize").  The    */
/* same function as the activation fake-quant, applied to the fp32 result:  */
/* code = clamp(rint(fp32(y) * fp32(1/s)), -128, 127) in fp32, y' = code*s. */
/* NaN -> 0, +-Inf saturate (as for the activations).                       */
/* ---------------------------------------------------------------------- */
static int requant_code_f32(double y, float s)
{
    volatile float inv = 1.0f / s;
    volatile float yf = (float)y;
    volatile float t = yf * inv;
    return clamp_i8((double)rintf(t));
}

/* codes[n] and y'[n] = code * s (fp64) of the requantisation of y[n]. */
void tq2o_requant(const double *y, int64_t n, float s, int8_t *codes, double *out)
{
    for (int64_t i = 0; i < n; ++i) {
        int q = requant_code_f32(y[i], s);
        if (codes)
            codes[i] = (int8_t)q;
        if (out)
            out[i] = (double)q * (double)s;
    }
}

/* ---------------------------------------------------------------------- */
/* The matvec [P1, linear factoring]:                                      */
/*   y[m][n] = sum_b d[n][b] * sum_{k in b} x'[m][k] * (q[n][k] - 1)        */
/* with x' = x (act_scale == 0: no prologue, cf. the checkpoint's "scale 0  */
/* = unquantized" convention [P3]) or x' = fake-quant(x) with s=act_scale.  */
/* Also returns the tolerance sum T[m][n] = sum_b |d_b| sum_{k in b} |x'_k| */
/* (over every k, zero codes included).                                     */
/* ---------------------------------------------------------------------- */
static double xprime(const uint16_t *x, int64_t idx, float act_scale)
{
    if (act_scale == 0.0f)
        return tq2o_half_to_double(x[idx]);
    return (double)fq_code_recip_f32(x[idx], act_scale) * (double)act_scale;
}

void tq2o_matvec_f64(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                     int64_t N, int64_t K, float act_scale, double *y, double *tol_sum)
{
    int64_t B = K / 256;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, bound = 0.0;
            for (int64_t b = 0; b < B; ++b) {
                double db = tq2o_half_to_double(d[n * B + b]);
                double sb = 0.0, ab = 0.0;
                for (int64_t k = b * 256; k < (b + 1) * 256; ++k) {
                    double xv = xprime(x, m * K + k, act_scale);
                    sb += xv * (double)(code_at(qs, K, n, k) - 1);
                    ab += fabs(xv);
                }
                acc += db * sb;
                bound += fabs(db) * ab;
            }
            y[m * N + n] = acc;
            if (tol_sum)
                tol_sum[m * N + n] = bound;
        }
}

/* Same as tq2o_matvec_f64 for a subset of output rows: rows[i] in [0,N),
 * y and tol_sum are [M, nrows]. */
void tq2o_matvec_rows_f64(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                          int64_t N, int64_t K, float act_scale, const int64_t *rows,
                          int64_t nrows, double *y, double *tol_sum)
{
    (void)N;
    int64_t B = K / 256;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t n = rows[i];
            double acc = 0.0, bound = 0.0;
            for (int64_t b = 0; b < B; ++b) {
                double db = tq2o_half_to_double(d[n * B + b]);
                double sb = 0.0, ab = 0.0;
                for (int64_t k = b * 256; k < (b + 1) * 256; ++k) {
                    double xv = xprime(x, m * K + k, act_scale);
                    sb += xv * (double)(code_at(qs, K, n, k) - 1);
                    ab += fabs(xv);
                }
                acc += db * sb;
                bound += fabs(db) * ab;
            }
            y[m * nrows + i] = acc;
            if (tol_sum)
                tol_sum[m * nrows + i] = bound;
        }
}

/* ---------------------------------------------------------------------- */
/* Exact matvec, the oracle's own check.  Every finite fp16 value is an     */
/* integer multiple of 2^-24 below 2^40 in magnitude, so d*x*(q-1) is an    */
/* integer multiple of 2^-48 below 2^80 and the K-term sum (K <= 2^14)      */
/* stays below 2^94: it fits __int128 exactly.  With the prologue, x' = q_x */
/* * s and s = S * 2^e with a 24-bit integer S, so the sum of d*q_x*(q-1)*S */
/* is exact too.  The only rounding is the final conversion to double.      */
/* Returns the number of outputs that were not finite (Inf/NaN inputs).     */
/* ---------------------------------------------------------------------- */
int64_t tq2o_matvec_exact(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                          int64_t N, int64_t K, float act_scale, double *y)
{
    int64_t B = K / 256, bad = 0;
    int sexp = 0;
    int64_t sint = 0;
    if (act_scale != 0.0f) {
        double f = frexp((double)act_scale, &sexp); /* s = f * 2^sexp */
        sint = (int64_t)ldexp(f, 24);               /* exact: fp32 has 24 bits */
        sexp -= 24;                                 /* s = sint * 2^sexp */
    }
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            __int128 acc = 0;
            int ok = 1;
            for (int64_t b = 0; b < B; ++b) {
                int64_t du = half_to_units(d[n * B + b], &ok);
                for (int64_t k = b * 256; k < (b + 1) * 256; ++k) {
                    int w = code_at(qs, K, n, k) - 1;
                    if (act_scale == 0.0f) {
                        int64_t xu = half_to_units(x[m * K + k], &ok);
                        acc += (__int128)du * (__int128)xu * w;
                    } else {
                        int qx = fq_code_recip_f32(x[m * K + k], act_scale);
                        acc += (__int128)du * (__int128)qx * (__int128)sint * w;
                    }
                }
            }
            double v;
            if (!ok) {
                v = NAN;
                ++bad;
            } else if (act_scale == 0.0f) {
                v = ldexp((double)acc, -48);
            } else {
                v = ldexp((double)acc, -24 + sexp);
            }
            y[m * N + n] = v;
        }
    return bad;
}

/* ---------------------------------------------------------------------- */
/* Affine int4 matvec (zero-point factoring).                              */
/* [P2] "Custom Metal kernels" (coreai-model-zoo knowledge page             */
/* custom-metal-kernels), the note on asymmetric (zero-point) int4: a fused */
/* affine-int4 matvec factors the zero point out of the dot product,        */
/* acc += s * (dot - z * sum x), per group of the reduction axis.           */
/* Readings (the note gives the identity only): W[n][k] = s[n][g] *         */
/* (q[n][k] - z[n][g]) with a 4-bit unsigned code q in [0, 15] and g = k/G; */
/* code k sits at bits 4*(k%2) of byte k/2 of row n (low nibble first);     */
/* s and z are fp16 arrays [N][K/G]; z is a real zero point in code units.  */
/* ---------------------------------------------------------------------- */
static int nibble_at(const uint8_t *qs, int64_t K, int64_t n, int64_t k)
{
    return (qs[n * (K / 2) + k / 2] >> (4 * (k % 2))) & 15;
}

/* y[m][n] = sum_g s_g * (sum_{k in g} x_k q_k - z_g * sum_{k in g} x_k),  */
/* fp64, the groups and the terms in order.  tol_sum[m][n] =                */
/* sum_g |s_g| sum_{k in g} |x_k| (q_k + |z_g|): the magnitude of the two   */
/* factored sums, which is what their rounding error scales with.           */
static void affine4_row(const uint16_t *x, int64_t m, const uint8_t *qs, const uint16_t *s,
                        const uint16_t *z, int64_t n, int64_t K, int64_t G, double *y, double *t)
{
    int64_t ng = K / G;
    double acc = 0.0, bound = 0.0;
    for (int64_t g = 0; g < ng; ++g) {
        double sg = tq2o_half_to_double(s[n * ng + g]);
        double zg = tq2o_half_to_double(z[n * ng + g]);
        double dot = 0.0, sx = 0.0, ab = 0.0;
        for (int64_t k = g * G; k < (g + 1) * G; ++k) {
            double xv = tq2o_half_to_double(x[m * K + k]);
            int q = nibble_at(qs, K, n, k);
            dot += xv * (double)q;
            sx += xv;
            ab += fabs(xv) * ((double)q + fabs(zg));
        }
        acc += sg * (dot - zg * sx);
        bound += fabs(sg) * ab;
    }
    *y = acc;
    if (t)
        *t = bound;
}

void tq2o_affine4_f64(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *s,
                      const uint16_t *z, int64_t N, int64_t K, int64_t G, double *y, double *tol_sum)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            affine4_row(x, m, qs, s, z, n, K, G, &y[m * N + n], tol_sum ? &tol_sum[m * N + n] : 0);
}

/* The same for the output rows rows[0..nrows): y, tol_sum are [M, nrows]. */
void tq2o_affine4_rows_f64(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *s,
                           const uint16_t *z, int64_t N, int64_t K, int64_t G, const int64_t *rows,
                           int64_t nrows, double *y, double *tol_sum)
{
    (void)N;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < nrows; ++i)
            affine4_row(x, m, qs, s, z, rows[i], K, G, &y[m * nrows + i],
                        tol_sum ? &tol_sum[m * nrows + i] : 0);
}

/* Exact dense form, the oracle's own check: sum_k W[n][k] x_k with W =     */
/* s * (q - z) taken element by element (no factoring).  In units of 2^-24  */
/* every fp16 value is an integer, so each term is s_u * (q * 2^24 - z_u) * */
/* x_u * 2^-72, summed in __int128.  A term that could push the sum past    */
/* 2^126 (|term| >= 2^112 with K <= 2^14) marks the output NaN instead;     */
/* returns the number of such (or non-finite) outputs.                      */
static int bitlen128(__int128 v)
{
    unsigned __int128 u = v < 0 ? (unsigned __int128)(-v) : (unsigned __int128)v;
    int b = 0;
    while (u) {
        u >>= 1;
        ++b;
    }
    return b;
}

int64_t tq2o_affine4_exact(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *s,
                           const uint16_t *z, int64_t N, int64_t K, int64_t G, double *y)
{
    int64_t ng = K / G, bad = 0;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            __int128 acc = 0;
            int ok = K <= (1 << 14);
            for (int64_t k = 0; k < K && ok; ++k) {
                int64_t g = k / G;
                int64_t su = half_to_units(s[n * ng + g], &ok);
                int64_t zu = half_to_units(z[n * ng + g], &ok);
                int64_t xu = half_to_units(x[m * K + k], &ok);
                __int128 w = (__int128)su * ((__int128)nibble_at(qs, K, n, k) * ((__int128)1 << 24) - zu);
                if (bitlen128(w) + bitlen128(xu) >= 112) {
                    ok = 0;
                    break;
                }
                acc += w * xu;
            }
            if (!ok) {
                y[m * N + n] = NAN;
                ++bad;
            } else {
                y[m * N + n] = ldexp((double)acc, -72);
            }
        }
    return bad;
}
