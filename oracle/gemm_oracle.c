/*
 * gemm_oracle.c -- the parity oracle for the two dense matrix products.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, load or call this file.  Only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of each product, written out as
 * nested loops with one float64 accumulator per output element, summed in
 * ascending k.  There is no blocking, no reordering of the sum and no fusion;
 * the only preparation steps are exact conversions of the inputs to double
 * (half -> double and float -> double are both exact) and, for the SGEMM,
 * a copy of B into k-contiguous order so that each dot product walks memory
 * linearly.  Neither step changes a single rounding.
 *
 * Sources (the pages the method is taken from):
 *  - fp16 NT product: "从零开始的 AI Infra: 算子基础与GPU架构"
 *    (qi-zhan.github.io/blog/2026/cuda-gemm), section "0. Naive
 *    Implementation": C[m][n] = sum_k float(A[m*K+k]) * float(B[n*K+k]),
 *    stored as half(acc); and section "19. 去掉转置" for the reading of
 *    B[N,K] row-major as the transposed right operand.
 *  - fp32 SGEMM: "异步拷贝与 Hopper/Blackwell 新特性"
 *    (anrans.github.io/ai-infra-handbooks/cuda/advanced/async-hopper),
 *    section "cp.async 与多级流水 sm_80+", the gemm_cp_async listing's
 *    epilogue c = alpha*acc + beta*c over row-major A[M,K], B[K,N], C[M,N],
 *    and the CPU reference loop of its host harness.
 *  - block-scaled FP8 (MXFP8) NT product: the same page, section
 *    "Blackwell 概览 sm_100" (32 elements share one 8-bit exponent scale).
 *  - block-scaled FP4 (NVFP4) NT product: the same section (16 elements
 *    share one FP8 scale, plus a tensor-level FP32 scale).
 *
 * Precision: the pages accumulate in float; this oracle accumulates in
 * float64 and keeps the result unrounded, so that the GPU result can be
 * judged against the exact-ish value with a tolerance scaled by
 * S[i][j] = |alpha| * sum_k |A[i][k] * B'[k][j]|, which is also returned.
 *
 * Build: plain C99 + OpenMP, no fast-math, no FP contraction:
 *   gcc -O2 -std=c99 -fopenmp -ffp-contract=off -fPIC -shared
 */
#define _USE_MATH_DEFINES
#include <math.h>
#include <stdint.h>
#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* IEEE 754 binary16, from its definition: 1 sign bit, 5 exponent bits     */
/* with bias 15, 10 fraction bits; exponent 0 = zero/subnormal, 31 = inf or */
/* NaN.                                                                     */
/* ---------------------------------------------------------------------- */

double oracle_half_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);              /* 2^-14 * frac/2^10 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* 2^(e-15) * (1024+f)/2^10 */
    }
    return sign ? -v : v;
}

/* Round-to-nearest-even of a double to binary16, returned as its bits.
 * Values at or beyond 65520 (the midpoint between the largest finite half,
 * 65504, and 2^16) round to infinity. */
uint16_t oracle_f64_to_half_rn(double x)
{
    if (isnan(x)) return (uint16_t)0x7e00;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    const double a = fabs(x);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: multiples of 2^-24; 1024 * 2^-24 is the smallest
         * normal, whose encoding 0x0400 is also the integer 1024. */
        const double n = nearbyint(ldexp(a, 24));   /* ties to even */
        return (uint16_t)(sign | (uint16_t)n);
    }
    int ex;
    (void)frexp(a, &ex);             /* a = m * 2^ex, m in [0.5, 1) */
    int E = ex - 1;                  /* a in [2^E, 2^(E+1)) */
    double r = nearbyint(ldexp(a, 10 - E));   /* in [1024, 2048] */
    if (r >= 2048.0) { r = 1024.0; E += 1; }
    if (E + 15 >= 31) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(r - 1024.0));
}

void oracle_half_to_f64_array(int64_t n, const uint16_t *h, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_f64(h[i]);
}

void oracle_f64_to_half_rn_array(int64_t n, const double *x, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_half_rn(x[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* fp16 NT: C[i][j] = sum_{k<K} A[i][k] * B[j][k]                           */
/*   A: half [M,K] row-major, B: half [N,K] row-major (= B^T [K,N]          */
/*   column-major), C, S: double [M,N] row-major.  S may be NULL.           */
/* ---------------------------------------------------------------------- */

static double *decode_half_matrix(int64_t rows, int64_t cols, const uint16_t *h)
{
    const int64_t n = rows * cols;
    double *d = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!d) return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) d[i] = oracle_half_to_f64(h[i]);
    return d;
}

static void dot_nt(const double *a_row, const double *b_row, int64_t K,
                   double *acc_out, double *mag_out)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        /* exact: two halves (11-bit significands) or two scaled E4M3 values
         * (4-bit significands, exponents far inside double's range) */
        const double p = a_row[k] * b_row[k];
        acc += p;
        mag += fabs(p);
    }
    *acc_out = acc;
    *mag_out = mag;
}

int oracle_gemm_f16_nt(int64_t M, int64_t N, int64_t K,
                       const uint16_t *A, const uint16_t *B,
                       double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    double *a = decode_half_matrix(M, K, A);
    double *b = decode_half_matrix(N, K, B);
    if (!a || !b) { free(a); free(b); return -2; }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc, mag;
            dot_nt(a + i * K, b + j * K, K, &acc, &mag);
            C[i * N + j] = acc;
            if (S) S[i * N + j] = mag;
        }
    }
    free(a);
    free(b);
    return 0;
}

/* The same product at n listed positions (rows[t], cols[t]) only. */
int oracle_gemm_f16_nt_sampled(int64_t M, int64_t N, int64_t K,
                               const uint16_t *A, const uint16_t *B,
                               int64_t n, const int64_t *rows, const int64_t *cols,
                               double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#pragma omp parallel
    {
        double *a = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double *b = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            for (int64_t k = 0; k < K; ++k) {
                a[k] = oracle_half_to_f64(A[rows[t] * K + k]);
                b[k] = oracle_half_to_f64(B[cols[t] * K + k]);
            }
            double acc, mag;
            dot_nt(a, b, K, &acc, &mag);
            C[t] = acc;
            if (S) S[t] = mag;
        }
        free(a);
        free(b);
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* fp32 SGEMM: C[i][j] = alpha * sum_{k<K} A[i][k] * B[k][j] + beta * C0[i][j] */
/*   A: float [M,K], B: float [K,N], C0: float [M,N], all row-major.        */
/*   beta == 0 follows the BLAS convention: C0 is not read (may be NULL).   */
/*   C, S: double [M,N].  S = |alpha| * sum_k |A[i][k] * B[k][j]|.          */
/* ---------------------------------------------------------------------- */

static void dot_sgemm(const float *a_row, const double *b_col, int64_t K,
                      double *acc_out, double *mag_out)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double p = (double)a_row[k] * b_col[k];  /* exact: 24 x 24 bits */
        acc += p;
        mag += fabs(p);
    }
    *acc_out = acc;
    *mag_out = mag;
}

int oracle_sgemm(int64_t M, int64_t N, int64_t K, double alpha,
                 const float *A, const float *B, double beta, const float *C0,
                 double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (beta != 0.0 && !C0) return -1;
    /* B gathered column by column (bt[j*K + k] = B[k][j]); values unchanged. */
    double *bt = (double *)malloc((size_t)(N * K > 0 ? N * K : 1) * sizeof(double));
    if (!bt) return -2;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k) bt[j * K + k] = (double)B[k * N + j];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc, mag;
            dot_sgemm(A + i * K, bt + j * K, K, &acc, &mag);
            double c = alpha * acc;
            if (beta != 0.0) c += beta * (double)C0[i * N + j];
            C[i * N + j] = c;
            if (S) S[i * N + j] = fabs(alpha) * mag;
        }
    }
    free(bt);
    return 0;
}

int oracle_sgemm_sampled(int64_t M, int64_t N, int64_t K, double alpha,
                         const float *A, const float *B, double beta, const float *C0,
                         int64_t n, const int64_t *rows, const int64_t *cols,
                         double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    if (beta != 0.0 && !C0) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#pragma omp parallel
    {
        double *b = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            const int64_t i = rows[t], j = cols[t];
            for (int64_t k = 0; k < K; ++k) b[k] = (double)B[k * N + j];
            double acc, mag;
            dot_sgemm(A + i * K, b, K, &acc, &mag);
            double c = alpha * acc;
            if (beta != 0.0) c += beta * (double)C0[i * N + j];
            C[t] = c;
            if (S) S[t] = fabs(alpha) * mag;
        }
        free(b);
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Fused epilogue of the fp16 product ("第 6 章 · Shared Memory & Tile",    */
/* section "6.5.4 Epilogue 融合": Y = activation(GEMM(X, W) + bias)), with   */
/* the scalars and residual of the usual GEMM epilogue:                     */
/*   Y[i][j] = act(alpha * sum_k A[i][k] B[j][k] + bias[j] + beta * R[i][j]) */
/* act: 0 none, 1 ReLU max(v, 0), 2 SiLU v / (1 + e^-v), 3 GELU with the    */
/* tanh approximation 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))).       */
/* bias (half [N]) and R (half [M,N]) may be NULL (no term).  Y, S: double  */
/* [M,N]; S = |alpha| sum_k |A B| + |bias[j]| + |beta R[i][j]|, the          */
/* pre-activation magnitude.                                                 */
/* ---------------------------------------------------------------------- */

double oracle_activation(double v, int act)
{
    switch (act) {
    case 0: return v;
    case 1: return v > 0.0 ? v : 0.0;
    case 2: return v / (1.0 + exp(-v));
    case 3: return 0.5 * v * (1.0 + tanh(sqrt(2.0 / M_PI) * (v + 0.044715 * v * v * v)));
    default: return NAN;
    }
}

/* One output of the epilogue from its product acc and scale mag:
 * Y = act(alpha*acc + bias[j] + beta*R[i][j]), S = |alpha|*mag + |bias[j]| + |beta*R[i][j]|. */
static void epilogue_at(double acc, double mag, int64_t i, int64_t j, int64_t N,
                        double alpha, const uint16_t *bias, double beta, const uint16_t *R,
                        int act, double *y, double *s)
{
    double v = alpha * acc;
    double scale = fabs(alpha) * mag;
    if (bias) {
        const double b = oracle_half_to_f64(bias[j]);
        v += b;
        scale += fabs(b);
    }
    if (R) {
        const double r = beta * oracle_half_to_f64(R[i * N + j]);
        v += r;
        scale += fabs(r);
    }
    *y = oracle_activation(v, act);
    *s = scale;
}

int oracle_gemm_f16_nt_epilogue(int64_t M, int64_t N, int64_t K,
                                const uint16_t *A, const uint16_t *B,
                                double alpha, const uint16_t *bias,
                                double beta, const uint16_t *R, int act,
                                double *Y, double *S)
{
    if (act < 0 || act > 3) return -1;
    int rc = oracle_gemm_f16_nt(M, N, K, A, B, Y, S);
    if (rc != 0) return rc;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            epilogue_at(Y[i * N + j], S[i * N + j], i, j, N, alpha, bias, beta, R, act,
                        &Y[i * N + j], &S[i * N + j]);
    return 0;
}

/* The same epilogue at n listed positions (rows[t], cols[t]) only. */
int oracle_gemm_f16_nt_epilogue_sampled(int64_t M, int64_t N, int64_t K,
                                        const uint16_t *A, const uint16_t *B,
                                        double alpha, const uint16_t *bias,
                                        double beta, const uint16_t *R, int act,
                                        int64_t n, const int64_t *rows, const int64_t *cols,
                                        double *Y, double *S)
{
    if (act < 0 || act > 3) return -1;
    int rc = oracle_gemm_f16_nt_sampled(M, N, K, A, B, n, rows, cols, Y, S);
    if (rc != 0) return rc;
    for (int64_t t = 0; t < n; ++t)
        epilogue_at(Y[t], S[t], rows[t], cols[t], N, alpha, bias, beta, R, act, &Y[t], &S[t]);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Block-scaled FP8 (MXFP8): "异步拷贝与 Hopper/Blackwell 新特性", section   */
/* "Blackwell 概览 sm_100": in MXFP8 every 32 consecutive elements share   */
/* one 8-bit exponent scale factor.  The element format is FP8 E4M3 and    */
/* the scale UE8M0 (the OCP microscaling formats Blackwell's block-scaled   */
/* MMA reads):                                                               */
/*   E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;        */
/*         exponent 0 = subnormal m/8 * 2^-6; S.1111.111 = NaN; no inf.     */
/*   UE8M0: an unsigned exponent alone, 2^(e - 127); 0xFF = NaN.            */
/* The product of one row of A with one row of B (both K-major):            */
/*   C[m][n] = sum_k e4m3(A[m][k]) 2^(SA[m][k/32] - 127)                    */
/*                   * e4m3(B[n][k]) 2^(SB[n][k/32] - 127)                  */
/* with SA [M][K/32], SB [N][K/32] row-major.  Each term is exact in        */
/* double (4 + 4 significant bits, exponents within range).                 */
/* ---------------------------------------------------------------------- */

double oracle_e4m3_to_f64(uint8_t c)
{
    const int sign = (c >> 7) & 1;
    const int expo = (c >> 3) & 0xf;
    const int mant = c & 0x7;
    double v;
    if (expo == 0xf && mant == 0x7) return NAN;
    if (expo == 0)
        v = ldexp((double)mant / 8.0, -6);
    else
        v = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -v : v;
}

double oracle_ue8m0_to_f64(uint8_t e)
{
    if (e == 0xff) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* Row r of an MXFP8 matrix (K codes, K/32 scales) decoded to doubles. */
static void decode_mx_row(const uint8_t *codes, const uint8_t *scales, int64_t K, double *out)
{
    for (int64_t k = 0; k < K; ++k)
        out[k] = oracle_e4m3_to_f64(codes[k]) * oracle_ue8m0_to_f64(scales[k / 32]);
}

static double *decode_mx_matrix(int64_t rows, int64_t K, const uint8_t *codes, const uint8_t *scales)
{
    double *d = (double *)malloc((size_t)(rows > 0 ? rows : 1) * (size_t)(K > 0 ? K : 1) * sizeof(double));
    if (!d) return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        decode_mx_row(codes + r * K, scales + r * (K / 32), K, d + r * K);
    return d;
}

int oracle_gemm_mxfp8_nt(int64_t M, int64_t N, int64_t K,
                         const uint8_t *A, const uint8_t *SA,
                         const uint8_t *B, const uint8_t *SB,
                         double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0) return -1;
    double *a = decode_mx_matrix(M, K, A, SA);
    double *b = decode_mx_matrix(N, K, B, SB);
    if (!a || !b) {
        free(a);
        free(b);
        return -2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double acc, mag;
            dot_nt(a + i * K, b + j * K, K, &acc, &mag);
            C[i * N + j] = acc;
            if (S) S[i * N + j] = mag;
        }
    free(a);
    free(b);
    return 0;
}

/* The same product at n listed positions (rows[t], cols[t]) only. */
int oracle_gemm_mxfp8_nt_sampled(int64_t M, int64_t N, int64_t K,
                                 const uint8_t *A, const uint8_t *SA,
                                 const uint8_t *B, const uint8_t *SB,
                                 int64_t n, const int64_t *rows, const int64_t *cols,
                                 double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || n < 0) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#pragma omp parallel
    {
        double *a = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double *b = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            decode_mx_row(A + rows[t] * K, SA + rows[t] * (K / 32), K, a);
            decode_mx_row(B + cols[t] * K, SB + cols[t] * (K / 32), K, b);
            double acc, mag;
            dot_nt(a, b, K, &acc, &mag);
            C[t] = acc;
            if (S) S[t] = mag;
        }
        free(a);
        free(b);
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Block-scaled FP4 (NVFP4): "异步拷贝与 Hopper/Blackwell 新特性", section    */
/* "Blackwell 概览 sm_100": every 16 elements share one FP8 scale factor,   */
/* and a tensor-level FP32 scale applies on top.  Read here as:             */
/*   elements FP4 E2M1: 1 sign bit, 2 exponent bits with bias 1, 1          */
/*     mantissa bit; exponent 0 = subnormal m/2; no inf or NaN.  Two per    */
/*     byte, element 2i in the low nibble of byte i, 2i+1 in the high one.  */
/*   block scales UE4M3: the E4M3 value of the byte (positive codes);       */
/*   C[m][n] = alpha * sum_k a(m,k) SA[m][k/16] * b(n,k) SB[n][k/16],       */
/*     alpha the product of the two tensor-level scales.                    */
/* Each term is exact in double (2 x 2 significant bits, 4 x 4 for the      */
/* scales).                                                                  */
/* ---------------------------------------------------------------------- */

double oracle_e2m1_to_f64(uint8_t nibble)
{
    const int sign = (nibble >> 3) & 1;
    const int expo = (nibble >> 1) & 3;
    const int mant = nibble & 1;
    double v;
    if (expo == 0)
        v = 0.5 * (double)mant;
    else
        v = ldexp(1.0 + 0.5 * (double)mant, expo - 1);
    return sign ? -v : v;
}

static void decode_nvfp4_row(const uint8_t *packed, const uint8_t *scales, int64_t K, double *out)
{
    for (int64_t k = 0; k < K; ++k) {
        const uint8_t byte = packed[k / 2];
        const uint8_t nib = (k % 2 == 0) ? (uint8_t)(byte & 0xf) : (uint8_t)(byte >> 4);
        out[k] = oracle_e2m1_to_f64(nib) * oracle_e4m3_to_f64(scales[k / 16]);
    }
}

int oracle_gemm_nvfp4_nt(int64_t M, int64_t N, int64_t K,
                         const uint8_t *A, const uint8_t *SA,
                         const uint8_t *B, const uint8_t *SB, double alpha,
                         double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % 16 != 0) return -1;
    double *a = (double *)malloc((size_t)(M > 0 ? M : 1) * (size_t)(K > 0 ? K : 1) * sizeof(double));
    double *b = (double *)malloc((size_t)(N > 0 ? N : 1) * (size_t)(K > 0 ? K : 1) * sizeof(double));
    if (!a || !b) {
        free(a);
        free(b);
        return -2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) decode_nvfp4_row(A + r * (K / 2), SA + r * (K / 16), K, a + r * K);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) decode_nvfp4_row(B + r * (K / 2), SB + r * (K / 16), K, b + r * K);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double acc, mag;
            dot_nt(a + i * K, b + j * K, K, &acc, &mag);
            C[i * N + j] = alpha * acc;
            if (S) S[i * N + j] = fabs(alpha) * mag;
        }
    free(a);
    free(b);
    return 0;
}

/* The same product at n listed positions (rows[t], cols[t]) only. */
int oracle_gemm_nvfp4_nt_sampled(int64_t M, int64_t N, int64_t K,
                                 const uint8_t *A, const uint8_t *SA,
                                 const uint8_t *B, const uint8_t *SB, double alpha,
                                 int64_t n, const int64_t *rows, const int64_t *cols,
                                 double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % 16 != 0 || n < 0) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#pragma omp parallel
    {
        double *a = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double *b = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            decode_nvfp4_row(A + rows[t] * (K / 2), SA + rows[t] * (K / 16), K, a);
            decode_nvfp4_row(B + cols[t] * (K / 2), SB + cols[t] * (K / 16), K, b);
            double acc, mag;
            dot_nt(a, b, K, &acc, &mag);
            C[t] = alpha * acc;
            if (S) S[t] = fabs(alpha) * mag;
        }
        free(a);
        free(b);
    }
    return 0;
}
