/*
 * FP64 CPU oracle for the FP16 GEMM  C = A * B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * execute this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table
 * or helper with the CUDA path.
 *
 * What it computes (the plain definition of the product the GPU path
 * approximates; "Xe2 ESIMD GEMM" page, section "Correctness testing", which
 * asks for a CPU reference of C = A*B over the same half-precision inputs):
 *
 *     R[i][j] = sum_{k=0}^{K-1} double(a_ik) * double(b_kj)
 *
 * where a_ik and b_kj are the IEEE binary16 inputs widened exactly to
 * binary64.  The page asks for an FP32 reference; this oracle uses FP64,
 * which is stricter (every product of two binary16 values is exact in
 * binary64, so the only rounding is in the running sum).
 *
 * The loop is the textbook triple loop in i-k-j order (so the innermost
 * loop walks a row of B and a row of R contiguously), with the rows of R
 * shared out over OpenMP threads.  There is no blocking, no reordering of
 * the k sum and no fusion: for each (i, j) the k terms are added in
 * increasing k, starting from +0.0.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

/*
 * Exact widening of one IEEE 754 binary16 bit pattern to binary64.
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   exponent field 0        -> zero or subnormal: fraction * 2^-24
 *   exponent field 1..30    -> normal: (1024 + fraction) * 2^(e - 25)
 *   exponent field 31       -> infinity (fraction 0) or NaN
 */
double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Widen n binary16 patterns (contiguous) into dst. */
void oracle_widen_f16(int64_t n, const uint16_t *src, double *dst)
{
    for (int64_t t = 0; t < n; ++t)
        dst[t] = oracle_f16_to_f64(src[t]);
}

/*
 * R (M x N, row stride ldr) = A (M x K, row stride lda) * B (K x N, row
 * stride ldb), all row-major binary64, entries of A and B being widened
 * binary16 values.
 */
void oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                     const double *A, int64_t lda,
                     const double *B, int64_t ldb,
                     double *R, int64_t ldr)
{
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < M; ++i) {
        double *r = R + i * ldr;
        for (int64_t j = 0; j < N; ++j)
            r[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[i * lda + k];
            const double *b = B + k * ldb;
            for (int64_t j = 0; j < N; ++j)
                r[j] += a * b[j];
        }
    }
}

/* Number of OpenMP threads the oracle will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
