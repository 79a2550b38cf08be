/*
 * oracle.c -- the plain, slow CPU oracle for the half-precision GEMM and
 * the BF16 linear layer (decode GEMV / prefill GEMM).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file.  It is used by the tests, by the package smoke check and
 * by the benchmark's timed CPU baseline, and by nothing else.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * What it computes, and where that is stated:
 *
 *  - "MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘", section 2 (GEMM入门):
 *    C[m,n] = sum_k A[m,k] * B[k,n], written there as a triple loop with one
 *    accumulator per output entry that runs over k in increasing order, and
 *    the column-major addressing A(m,k) = A[m + k*M], B(k,n) = B[k + n*K],
 *    C(m,n) = C[m + n*M].  Section 1 (规则分析) fixes the precision: FP16
 *    inputs, FP32 accumulation, FP16 output.
 *  - DCU decode-GEMV article (forum.sourcefind.cn), section 6.1: the linear
 *    layer Y = X W^T with X:[n,k], W:[m,k], Y:[n,m] (all row-major), i.e.
 *    Y[t,j] = sum_k X[t,k] * W[j,k]; section 6.2: each Y[j] is one
 *    independent dot product over the whole k range.  BF16 in, BF16 out.
 *  - Same article, sections 6.1 and 7: decode attention over a paged KV
 *    cache (see orc_decode_attention_bf16 at the end of this file).
 *  - The FP8 GEMM (orc_gemm_fp8): E4M3 or E5M2 inputs, FP32 accumulator,
 *    the FP8 row of the matrix-instruction table in "Hygon 优化", section
 *    DUMMA 矩阵指令形状.
 *  - The FP16 GEMM in other storage forms (transposed operands, row-major
 *    storage, any leading dimension) with an optional bias: the BLAS reading
 *    of section 2's GEMM, with the bias the DCU article's section 6.1 names
 *    as a property of the linear call (see orc_gemm_f16_general).
 *
 * How the oracle evaluates it:
 *  - Inputs arrive as raw 16-bit patterns and are decoded by this file's own
 *    IEEE binary16 / bfloat16 decoders (exact in double).
 *  - Every product of two decoded inputs is exact in double (11+11 or 8+8
 *    significand bits), and the sum is accumulated in double, k ascending,
 *    exactly as the definition's loop runs.  The accumulated error is below
 *    K * 2^-53 * sum|a*b|, far below any FP32 accumulation error.
 *  - The exact-ish double result is rounded ONCE, round-to-nearest-even,
 *    straight from double to FP16 (GEMM) or BF16 (linear).  Going through
 *    float first would round twice; this file never does.  Overflow goes to
 *    +-Inf; NaN stays NaN.
 *
 * The pages state no output rounding mode; this oracle takes the IEEE default
 * (round to nearest, ties to even).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* IEEE binary16 and bfloat16 codecs, written from the format definitions.   */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_decode(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);  /* (1.f) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double orc_bf16_decode(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);             /* subnormal: f * 2^-133 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134);  /* (1.f) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/*
 * Round a double to a binary format with `frac_bits` fraction bits, exponent
 * bias `bias`, all-ones exponent `emax_field` and the sign at bit `sign_bit`,
 * nearest-even.
 *
 * |x| is written as n * q where q is the spacing of representable values in
 * x's binade (or the subnormal spacing below the normal range).  x / q is an
 * exact power-of-two rescale in double, and rint() in the default rounding
 * mode rounds it to the nearest integer with ties to even.  n == 2^(frac+1)
 * means the value rounded up into the next binade.
 */
static uint32_t orc_round_bits(double x, int frac_bits, int bias, int emax_field, int sign_bit)
{
    uint32_t sign = signbit(x) ? (1u << sign_bit) : 0u;
    uint32_t inf = (uint32_t)emax_field << frac_bits;
    if (isnan(x)) return sign | inf | (1u << (frac_bits - 1));
    double a = fabs(x);
    if (isinf(a)) return sign | inf;
    if (a == 0.0) return sign;

    int ex;
    frexp(a, &ex);             /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;            /* a in [2^E, 2^(E+1)) */
    int emin = 1 - bias;       /* exponent of the smallest normal */
    if (E < emin) {
        /* subnormal range: spacing 2^(emin - frac_bits) */
        double n = rint(ldexp(a, frac_bits - emin));
        /* n == 2^frac_bits is exactly the smallest normal's encoding */
        return sign | (uint32_t)n;
    }
    double n = rint(ldexp(a, frac_bits - E));   /* in [2^frac, 2^(frac+1)] */
    if (n >= ldexp(1.0, frac_bits + 1)) {
        n = ldexp(1.0, frac_bits);
        E += 1;
    }
    int field = E + bias;
    if (field >= emax_field) return sign | inf;
    uint32_t frac = (uint32_t)n - (1u << frac_bits);
    return sign | ((uint32_t)field << frac_bits) | frac;
}

static uint16_t orc_round_to_format(double x, int frac_bits, int bias, int emax_field)
{
    return (uint16_t)orc_round_bits(x, frac_bits, bias, emax_field, 15);
}

uint16_t orc_f16_encode_rn(double x) { return orc_round_to_format(x, 10, 15, 31); }
uint16_t orc_bf16_encode_rn(double x) { return orc_round_to_format(x, 7, 127, 255); }
/* binary32: 1 sign bit, 8 exponent bits (bias 127), 23 fraction bits. */
uint32_t orc_f32_encode_rn(double x) { return orc_round_bits(x, 23, 127, 255, 31); }

/*
 * The two FP8 formats of the matrix-instruction table ("Hygon 优化", section
 * DUMMA 矩阵指令形状), in their common (OCP 8-bit floating point) definition:
 *   E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; exponent
 *         field 0 is subnormal (f/8 * 2^-6); there is no infinity, and only
 *         exponent 15 with fraction 7 is NaN, so the largest value is 448.
 *   E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits, IEEE-style:
 *         field 0 subnormal (f/4 * 2^-14), field 31 infinity (f = 0) or NaN.
 */
double orc_fp8_decode(uint8_t c, int e5m2)
{
    int sign = (c >> 7) & 1;
    double v;
    if (e5m2) {
        int e = (c >> 2) & 0x1f;
        int f = c & 0x3;
        if (e == 0) v = ldexp((double)f, -16);                 /* f/4 * 2^-14 */
        else if (e == 31) v = f ? NAN : INFINITY;
        else v = ldexp((double)(4 + f), e - 17);               /* (1.f) * 2^(e-15) */
    } else {
        int e = (c >> 3) & 0xf;
        int f = c & 0x7;
        if (e == 0) v = ldexp((double)f, -9);                  /* f/8 * 2^-6 */
        else if (e == 15 && f == 7) v = NAN;
        else v = ldexp((double)(8 + f), e - 10);               /* (1.f) * 2^(e-7) */
    }
    return sign ? -v : v;
}

/* Bulk versions for the Python side. */
void orc_f16_decode_n(const uint16_t* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_decode(in[i]);
}
void orc_bf16_decode_n(const uint16_t* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_decode(in[i]);
}
void orc_f16_encode_n(const double* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_encode_rn(in[i]);
}
void orc_bf16_encode_n(const double* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_encode_rn(in[i]);
}
void orc_f32_encode_n(const double* in, uint32_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_encode_rn(in[i]);
}
void orc_fp8_decode_n(const uint8_t* in, double* out, int64_t n, int e5m2)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_decode(in[i], e5m2);
}

/* ------------------------------------------------------------------------ */
/* Helpers                                                                   */
/* ------------------------------------------------------------------------ */

/* Decode table for all 65536 patterns, built with the decoder above; a table
 * lookup is the same value as calling the decoder, just cheaper. */
static void orc_build_table(double* lut, int bf16)
{
    for (uint32_t i = 0; i < 65536u; ++i)
        lut[i] = bf16 ? orc_bf16_decode((uint16_t)i) : orc_f16_decode((uint16_t)i);
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static void orc_set_threads(int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

/* ------------------------------------------------------------------------ */
/* Column-major FP16 GEMM: C(m,n) = sum_k A(m,k) B(k,n)                      */
/* ------------------------------------------------------------------------ */

/*
 * Computes the output columns listed in `cols` (all N columns when cols is
 * NULL).  Column j of the result goes to ref[m + j*M] (double, before
 * rounding) and out[m + j*M] (FP16 bits after the one rounding); either
 * pointer may be NULL.
 *
 * Loop order: for each column n, one double accumulator per row m, and k runs
 * 0..K-1 in the outer loop so that every accumulator sees its terms in the
 * definition's order (k ascending); the inner loop over m walks A's column k,
 * which is contiguous in the column-major layout.
 */
int orc_gemm_f16_colmajor_cols(const uint16_t* A, const uint16_t* B,
                               int64_t M, int64_t N, int64_t K,
                               const int64_t* cols, int64_t ncols,
                               double* ref, uint16_t* out, int threads)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    int64_t nc = cols ? ncols : N;
    double* lut = (double*)malloc(65536 * sizeof(double));
    if (!lut) return 2;
    orc_build_table(lut, 0);
    orc_set_threads(threads);
    int fail = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            fail = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < nc; ++j) {
            if (!acc) continue;
            int64_t n = cols ? cols[j] : j;
            for (int64_t m = 0; m < M; ++m) acc[m] = 0.0;
            if (n >= 0 && n < N) {
                for (int64_t k = 0; k < K; ++k) {
                    double b = lut[B[k + n * K]];
                    const uint16_t* a_col = A + k * M;
                    for (int64_t m = 0; m < M; ++m) acc[m] += lut[a_col[m]] * b;
                }
            }
            for (int64_t m = 0; m < M; ++m) {
                if (ref) ref[m + j * M] = acc[m];
                if (out) out[m + j * M] = orc_f16_encode_rn(acc[m]);
            }
        }
        free(acc);
    }
    free(lut);
    return fail;
}

/*
 * Computes the output rows listed in `rows`.  Row i of the result goes to
 * ref[i + n*nrows] / out[i + n*nrows] (column-major over the selected rows).
 * Each entry is one dot product over k ascending of row m of A (gathered
 * once, it is strided in memory) and column n of B.
 */
int orc_gemm_f16_colmajor_rows(const uint16_t* A, const uint16_t* B,
                               int64_t M, int64_t N, int64_t K,
                               const int64_t* rows, int64_t nrows,
                               double* ref, uint16_t* out, int threads)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    double* lut = (double*)malloc(65536 * sizeof(double));
    if (!lut) return 2;
    orc_build_table(lut, 0);
    orc_set_threads(threads);
    double* arow = (double*)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    if (!arow) { free(lut); return 2; }
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows[i];
        for (int64_t k = 0; k < K; ++k) arow[k] = (m >= 0 && m < M) ? lut[A[m + k * M]] : 0.0;
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            const uint16_t* b_col = B + n * K;
            for (int64_t k = 0; k < K; ++k) acc += arow[k] * lut[b_col[k]];
            if (ref) ref[i + n * nrows] = acc;
            if (out) out[i + n * nrows] = orc_f16_encode_rn(acc);
        }
    }
    free(arow);
    free(lut);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* General FP16 GEMM: C = op(A) op(B) [+ bias], any storage order and strides */
/* ------------------------------------------------------------------------ */

/*
 * Element addressing of a stored matrix.  `row_major` == 0: entry (r, c) at
 * P[r + c*ld] (the column-major storage of the MTT article, section 2);
 * `row_major` == 1: entry (r, c) at P[c + r*ld].
 */
static int64_t orc_at(int row_major, int64_t r, int64_t c, int64_t ld)
{
    return row_major ? c + r * ld : r + c * ld;
}

/*
 * The BLAS reading of the layouts (one FP16 GEMM, other storage forms):
 *   op(A)(m,k) = A_stored(m,k) when transa == 0, A_stored(k,m) when transa == 1;
 *   op(B)(k,n) = B_stored(k,n) when transb == 0, B_stored(n,k) when transb == 1;
 * every stored matrix addressed through orc_at with the call's storage order
 * and its leading dimension.  The optional bias (FP16 bits) is bias[m]
 * (bias_mode 1, one value per row of C) or bias[n] (bias_mode 2, one value
 * per column); it is added to the exact double sum, so the entry is still
 * rounded once:
 *   C(m,n) = fp16_rn( sum_{k ascending} op(A)(m,k) op(B)(k,n) + bias ).
 *
 * Computes rows `rows[0..nrows)` (all M when rows is NULL) of columns
 * `cols[0..ncols)` (all N when cols is NULL); selected entry (i, j) goes to
 * ref[i + j*nr] / out[i + j*nr], nr the number of selected rows, regardless
 * of `row_major` (the selection is always returned column-major).
 */
int orc_gemm_f16_general(int row_major, int transa, int transb,
                         const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                         int64_t M, int64_t N, int64_t K,
                         const uint16_t* bias, int bias_mode,
                         const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                         double* ref, uint16_t* out, int threads)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (bias_mode < 0 || bias_mode > 2 || (bias_mode != 0 && !bias)) return 1;
    int64_t nr = rows ? nrows : M;
    int64_t nc = cols ? ncols : N;
    double* lut = (double*)malloc(65536 * sizeof(double));
    if (!lut) return 2;
    orc_build_table(lut, 0);
    orc_set_threads(threads);
    int fail = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc((size_t)(nr > 0 ? nr : 1) * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            fail = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < nc; ++j) {
            if (!acc) continue;
            int64_t n = cols ? cols[j] : j;
            for (int64_t i = 0; i < nr; ++i) acc[i] = 0.0;
            if (n >= 0 && n < N) {
                for (int64_t k = 0; k < K; ++k) {
                    int64_t bi = transb ? orc_at(row_major, n, k, ldb) : orc_at(row_major, k, n, ldb);
                    double b = lut[B[bi]];
                    for (int64_t i = 0; i < nr; ++i) {
                        int64_t m = rows ? rows[i] : i;
                        if (m < 0 || m >= M) continue;
                        int64_t ai = transa ? orc_at(row_major, k, m, lda) : orc_at(row_major, m, k, lda);
                        acc[i] += lut[A[ai]] * b;
                    }
                }
            }
            for (int64_t i = 0; i < nr; ++i) {
                int64_t m = rows ? rows[i] : i;
                double v = acc[i];
                if (bias_mode == 1 && m >= 0 && m < M) v += lut[bias[m]];
                if (bias_mode == 2 && n >= 0 && n < N) v += lut[bias[n]];
                if (ref) ref[i + j * nr] = v;
                if (out) out[i + j * nr] = orc_f16_encode_rn(v);
            }
        }
        free(acc);
    }
    free(lut);
    return fail;
}

/* ------------------------------------------------------------------------ */
/* FP8 GEMM: C(m,n) = alpha * sum_k A(m,k) B(k,n), FP32 accumulator          */
/* ------------------------------------------------------------------------ */

/*
 * The FP8 row of the matrix-instruction table ("Hygon 优化", section DUMMA
 * 矩阵指令形状): FP8 (E4M3 or E5M2) inputs, FP32 accumulator; the product is
 * the GEMM of "MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘", section 2.
 * Both operands are stored K-major (the k values of one row of A, or of one
 * column of B, contiguous): A(m,k) = A[k + m*lda], B(k,n) = B[k + n*ldb].
 * Every product of two FP8 values is exact in double and the sum runs over k
 * ascending in double; the result is scaled by alpha and rounded once to the
 * output format: out_type 0 = FP32 (written to out32), 1 = BF16 (out16).
 * Rows `rows` (all M when NULL) x columns `cols` (all N when NULL); entry
 * (i, j) of the selection at index i + j*nr.
 */
int orc_gemm_fp8(int e5m2, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                 int64_t M, int64_t N, int64_t K, double alpha, int out_type,
                 const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                 double* ref, uint32_t* out32, uint16_t* out16, int threads)
{
    if (M < 0 || N < 0 || K < 0 || out_type < 0 || out_type > 1) return 1;
    int64_t nr = rows ? nrows : M;
    int64_t nc = cols ? ncols : N;
    double lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = orc_fp8_decode((uint8_t)c, e5m2);
    orc_set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < nc; ++j) {
        int64_t n = cols ? cols[j] : j;
        for (int64_t i = 0; i < nr; ++i) {
            int64_t m = rows ? rows[i] : i;
            double acc = 0.0;
            if (n >= 0 && n < N && m >= 0 && m < M) {
                const uint8_t* a_row = A + m * lda;
                const uint8_t* b_col = B + n * ldb;
                for (int64_t k = 0; k < K; ++k) acc += lut[a_row[k]] * lut[b_col[k]];
            }
            double v = alpha * acc;
            if (ref) ref[i + j * nr] = v;
            if (out_type == 0 && out32) out32[i + j * nr] = orc_f32_encode_rn(v);
            if (out_type == 1 && out16) out16[i + j * nr] = orc_bf16_encode_rn(v);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* BF16 linear layer: Y[t,j] = sum_k X[t,k] W[j,k]                           */
/* ------------------------------------------------------------------------ */

/*
 * W is [M,K] row-major, X is [n,K] row-major, Y is [n,M] row-major.  Computes
 * the output features j listed in `js` (all M when js is NULL) for every
 * token t; entry (t, i) of the selection goes to ref[t*nj + i] / out[t*nj + i].
 * Each entry is one dot product over k ascending, accumulated in double and
 * rounded once to BF16.
 */
int orc_linear_bf16(const uint16_t* W, const uint16_t* X,
                    int64_t M, int64_t K, int64_t n,
                    const int64_t* js, int64_t njs,
                    double* ref, uint16_t* out, int threads)
{
    if (M < 0 || K < 0 || n < 0) return 1;
    int64_t nj = js ? njs : M;
    double* lut = (double*)malloc(65536 * sizeof(double));
    if (!lut) return 2;
    orc_build_table(lut, 1);
    orc_set_threads(threads);
    /* decode X once: n*K doubles (small: X is the activation side) */
    double* xd = (double*)malloc((size_t)((n * K) > 0 ? n * K : 1) * sizeof(double));
    if (!xd) { free(lut); return 2; }
    for (int64_t i = 0; i < n * K; ++i) xd[i] = lut[X[i]];
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < nj; ++i) {
        int64_t j = js ? js[i] : i;
        const uint16_t* wrow = W + j * K;
        for (int64_t t = 0; t < n; ++t) {
            double acc = 0.0;
            if (j >= 0 && j < M) {
                const double* xr = xd + t * K;
                for (int64_t k = 0; k < K; ++k) acc += xr[k] * lut[wrow[k]];
            }
            if (ref) ref[t * nj + i] = acc;
            if (out) out[t * nj + i] = orc_bf16_encode_rn(acc);
        }
    }
    free(xd);
    free(lut);
    return 0;
}

/*
 * Same linear layer, restricted to the tokens listed in `ts` (rows of X) for
 * every output feature j: entry (i, j) goes to ref[i*M + j] / out[i*M + j].
 */
int orc_linear_bf16_tokens(const uint16_t* W, const uint16_t* X,
                           int64_t M, int64_t K, int64_t n,
                           const int64_t* ts, int64_t nts,
                           double* ref, uint16_t* out, int threads)
{
    if (M < 0 || K < 0 || n < 0) return 1;
    double* lut = (double*)malloc(65536 * sizeof(double));
    if (!lut) return 2;
    orc_build_table(lut, 1);
    orc_set_threads(threads);
    double* xd = (double*)malloc((size_t)((nts * K) > 0 ? nts * K : 1) * sizeof(double));
    if (!xd) { free(lut); return 2; }
    for (int64_t i = 0; i < nts; ++i)
        for (int64_t k = 0; k < K; ++k)
            xd[i * K + k] = (ts[i] >= 0 && ts[i] < n) ? lut[X[ts[i] * K + k]] : 0.0;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t j = 0; j < M; ++j) {
        const uint16_t* wrow = W + j * K;
        for (int64_t i = 0; i < nts; ++i) {
            double acc = 0.0;
            const double* xr = xd + i * K;
            for (int64_t k = 0; k < K; ++k) acc += xr[k] * lut[wrow[k]];
            if (ref) ref[i * M + j] = acc;
            if (out) out[i * M + j] = orc_bf16_encode_rn(acc);
        }
    }
    free(xd);
    free(lut);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention over a paged BF16 KV cache                               */
/* ------------------------------------------------------------------------ */

/*
 * DCU decode-GEMV article (forum.sourcefind.cn), section 6.1: for one query
 * head, scores[1,L] = Q K^T, prob = softmax(scores), out[1,D] = prob V, with K
 * and V stored in a paged cache [block, token_in_block, kv_head, head_dim];
 * section 7: 16 query heads share 4 KV heads (query head h reads KV head
 * h / (num_q_heads / num_kv_heads)).  The page omits the score scale; it is an
 * argument here (scores = scale * q.k).
 *
 * The oracle computes the definition directly, over the whole sequence, in
 * double: the maximum score is subtracted before exponentiating (the same
 * value mathematically), the weighted sum of V rows and the normaliser run over
 * tokens in increasing order, and each output is rounded once to BF16.  A
 * sequence of length 0 gives zeros.  Returns 3 if a block-table entry is out
 * of range.
 *
 * q: [num_seqs, num_q_heads, hd]; out/ref: same shape;
 * block_tables: [num_seqs, max_blocks]; seq_lens: [num_seqs].
 */
int orc_decode_attention_bf16(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                              const int32_t* block_tables, const int32_t* seq_lens,
                              int64_t num_seqs, int64_t num_q_heads, int64_t num_kv_heads, int64_t hd,
                              int64_t block_size, int64_t max_blocks, int64_t num_blocks, double scale,
                              double* ref, uint16_t* out, int threads)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || hd <= 0 || block_size <= 0) return 1;
    if (num_q_heads % num_kv_heads != 0) return 1;
    const int64_t group = num_q_heads / num_kv_heads;
    double* lut = (double*)malloc(65536 * sizeof(double));
    if (!lut) return 2;
    orc_build_table(lut, 1);
    orc_set_threads(threads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t s = 0; s < num_seqs; ++s) {
        for (int64_t h = 0; h < num_q_heads; ++h) {
            const int64_t L = seq_lens[s];
            const int64_t g = h / group;
            const uint16_t* qh = q + (s * num_q_heads + h) * hd;
            double* acc = (double*)calloc((size_t)hd, sizeof(double));
            double* sc = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
            int64_t* rowbase = (int64_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int64_t));
            if (!acc || !sc || !rowbase) {
#pragma omp atomic write
                bad = 2;
            } else {
                double mx = -INFINITY;
                for (int64_t t = 0; t < L; ++t) {
                    const int64_t blk = block_tables[s * max_blocks + t / block_size];
                    if (blk < 0 || blk >= num_blocks) {
#pragma omp atomic write
                        bad = 3;
                        sc[t] = -INFINITY;
                        rowbase[t] = -1;
                        continue;
                    }
                    const int64_t base = ((blk * block_size + t % block_size) * num_kv_heads + g) * hd;
                    rowbase[t] = base;
                    double d = 0.0;
                    for (int64_t e = 0; e < hd; ++e) d += lut[qh[e]] * lut[k_cache[base + e]];
                    sc[t] = scale * d;
                    if (sc[t] > mx) mx = sc[t];
                }
                double l = 0.0;
                for (int64_t t = 0; t < L; ++t) {
                    if (rowbase[t] < 0) continue;
                    const double p = exp(sc[t] - mx);
                    l += p;
                    for (int64_t e = 0; e < hd; ++e) acc[e] += p * lut[v_cache[rowbase[t] + e]];
                }
                for (int64_t e = 0; e < hd; ++e) {
                    const double o = (L > 0 && l > 0.0) ? acc[e] / l : 0.0;
                    const int64_t idx = (s * num_q_heads + h) * hd + e;
                    if (ref) ref[idx] = o;
                    if (out) out[idx] = orc_bf16_encode_rn(o);
                }
            }
            free(acc);
            free(sc);
            free(rowbase);
        }
    }
    free(lut);
    return bad;
}
