/*
 * oracle.c - plain CPU reference for C = epilogue(A . B) on bf16 or fp16 inputs.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or helper with the CUDA
 * path, and it includes nothing from it.
 *
 * What it computes (page "How We Built TLX: A Hardware-Native GPU Compiler
 * for Production ML at Scale", section "Introducing TLX", first listing: the
 * standard Triton tiled matmul; and the fused "multiply, add bias, apply
 * GELU in one pass" kernel of the TileGym/cuTile tutorial page):
 *
 *     x_ij = sum_{k < K} a_ik * b_kj          (the accumulation over K)
 *     y_ij = x_ij                             epilogue "none"
 *          = x_ij + bias_j                    epilogue "bias"
 *          = gelu_tanh(x_ij + bias_j)         epilogue "bias + GELU"
 *
 * The listing accumulates in fp32 over BLOCK_K steps; the oracle is the
 * plain definition that result approximates: every input is widened
 * exactly to double, every product a_ik*b_kj is exact in double (8+8
 * significand bits for bf16, 11+11 for fp16), and the sum runs over k in
 * ascending order in double.
 * No blocking, no reordering: one output element is one dot product.
 *
 * Beside y it returns s_ij = sum_k |a_ik * b_kj|, the magnitude that the
 * per-element tolerance |err| <= 1e-2 * s_ij + 1e-5 is stated against.
 *
 * GELU: the pages name GELU without a formula; the workload names the tanh
 * form, so gelu_tanh(z) = z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3)))
 * (Hendrycks & Gimpel, "Gaussian Error Linear Units"), in double with the C
 * library's tanh.
 *
 * Row normalisation (optional, the "fuse the norm into the GEMM" idea of the
 * TLX pages): with row_norm set, A is first replaced by rmsnorm(A),
 *     a'_ik = a_ik / sqrt((1/K) sum_k a_ik^2 + eps),
 * in double, and the product, bias and GELU follow on a'.  (A gain vector
 * gamma folds into B: rmsnorm_gamma(A) . B = rmsnorm(A) . diag(gamma) B.)
 *
 * Element types: A, B and bias are all bf16 or all IEEE binary16 (fp16, the
 * TLX listing's type); both widen exactly to double.
 *
 * Layouts: A is M x K, row-major (element (i,k) at A[i*lda + k]) or
 * column-major (at A[k*lda + i]); B is K x N, row-major (B[k*ldb + j]) or
 * column-major (B[j*ldb + k]).  Inputs are bit patterns (uint16).
 *
 * Rows: the caller may ask for a subset of output rows (rows != NULL), so a
 * full-size problem can be checked on a sample; row r of Y/S then holds
 * output row rows[r].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_EPI_NONE = 0, ORACLE_EPI_BIAS = 1, ORACLE_EPI_BIAS_GELU = 2 };

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal: (-1)^s * 2^(e-15) * (1 + f/1024); subnormal (e = 0): (-1)^s * 2^-14 * f/1024;
 * e = 31: infinity (f = 0) or NaN.  Every value is exact in double. */
double oracle_f16_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

enum { ORACLE_IN_BF16 = 0, ORACLE_IN_F16 = 1 };

static double widen(uint16_t h, int in_dtype)
{
    return in_dtype == ORACLE_IN_F16 ? oracle_f16_to_double(h) : oracle_bf16_to_double(h);
}

double oracle_gelu_tanh(double z)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)));
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Returns 0 on success, -1 on a bad argument, -2 when scratch memory for the
 * widened operands cannot be had.
 */
int oracle_gemm_norm(const uint16_t *A, int a_col_major, int64_t lda,
                     const uint16_t *B, int b_col_major, int64_t ldb,
                     const uint16_t *bias, int epi, int in_dtype,
                     int row_norm, double eps,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t *rows, int64_t n_rows,
                     double *Y, double *S)
{
    if (M < 0 || N < 0 || K < 0 || !Y || !S) return -1;
    if (in_dtype != ORACLE_IN_BF16 && in_dtype != ORACLE_IN_F16) return -1;
    if (epi != ORACLE_EPI_NONE && epi != ORACLE_EPI_BIAS && epi != ORACLE_EPI_BIAS_GELU) return -1;
    if (epi != ORACLE_EPI_NONE && N > 0 && !bias) return -1;
    if (K > 0 && M > 0 && !A) return -1;
    if (K > 0 && N > 0 && !B) return -1;
    if (!rows) n_rows = M;
    for (int64_t r = 0; rows && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;

    /* B widened once into a K x N row-major double array (b[k*N + j]), so
     * the inner loop runs along j whatever B's storage order is. */
    double *b = NULL;
    if (K > 0 && N > 0) {
        b = (double *)malloc((size_t)K * (size_t)N * sizeof(double));
        if (!b) return -2;
        for (int64_t k = 0; k < K; ++k)
            for (int64_t j = 0; j < N; ++j)
                b[k * N + j] = widen(b_col_major ? B[j * ldb + k] : B[k * ldb + j], in_dtype);
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *y = Y + r * N;
        double *s = S + r * N;
        for (int64_t j = 0; j < N; ++j) { y[j] = 0.0; s[j] = 0.0; }
        /* rmsnorm scale of row i (1 without normalisation) */
        double scale = 1.0;
        if (row_norm && K > 0) {
            double ss = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = widen(a_col_major ? A[k * lda + i] : A[i * lda + k], in_dtype);
                ss += a * a;
            }
            scale = 1.0 / sqrt(ss / (double)K + eps);
        }
        /* k ascending, the same order for every element: y_ij accumulates
         * a'_ik*b_kj for k = 0, 1, ..., K-1. */
        for (int64_t k = 0; k < K; ++k) {
            const double a = scale * widen(a_col_major ? A[k * lda + i] : A[i * lda + k], in_dtype);
            const double *bk = b + k * N;
            for (int64_t j = 0; j < N; ++j) {
                const double p = a * bk[j];
                y[j] += p;
                s[j] += fabs(p);
            }
        }
        if (epi != ORACLE_EPI_NONE) {
            for (int64_t j = 0; j < N; ++j) {
                const double z = y[j] + widen(bias[j], in_dtype);
                y[j] = (epi == ORACLE_EPI_BIAS_GELU) ? oracle_gelu_tanh(z) : z;
            }
        }
    }
    free(b);
    return 0;
}

/* The GEMM without row normalisation. */
int oracle_gemm(const uint16_t *A, int a_col_major, int64_t lda,
                const uint16_t *B, int b_col_major, int64_t ldb,
                const uint16_t *bias, int epi, int in_dtype,
                int64_t M, int64_t N, int64_t K,
                const int64_t *rows, int64_t n_rows,
                double *Y, double *S)
{
    return oracle_gemm_norm(A, a_col_major, lda, B, b_col_major, ldb, bias, epi, in_dtype, 0, 0.0,
                            M, N, K, rows, n_rows, Y, S);
}
