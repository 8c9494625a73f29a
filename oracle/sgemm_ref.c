/*
 * fp64 CPU oracle for the FP32 general matrix multiply
 *
 *     C_out[i][j] = alpha * sum_{k<K} A[i][k] * B[k][j] + beta * C_in[i][j]
 *
 * on row-major A[M,K] (row pitch lda), B[K,N] (ldb), C[M,N] (ldc).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file;
 * only the tests, the package's smoke check and the bench's CPU-baseline leg
 * load it.  It shares no code, header or constant with the CUDA library.
 *
 * Where the definition comes from
 *   - "Matmul I: tiling and shared memory" (notes.ybc.sh cap-07), section 1:
 *     C = A.B with A [M,K], B [K,N], C [M,N], all row major, FP32; each output
 *     is a length-K dot product, 2MNK FLOPs in total.
 *   - "2D Register Tiling: The Outer Product" (maxxfuu article4/page8), "The
 *     Kernel": the epilogue writes alpha * acc + beta * C.
 *   - "The Final Kernel" (maxxfuu article4/page14), "Skipping The Read Of C":
 *     with beta == 0 the old C is not read at all.
 *
 * Readings where the pages are silent (BLAS conventions):
 *   - beta == 0: C_in is never read (NaN/Inf in it cannot reach the output).
 *   - alpha == 0 or K == 0: the product term is skipped and A, B are not read,
 *     so C_out = beta * C_in (or 0 when beta == 0).
 *   - M == 0 or N == 0: nothing is written.
 *   - Only the first N entries of each output row are written; the ldc
 *     padding is left as it was.
 *
 * Arithmetic: every fp32 input is widened to double; the product of two fp32
 * values is exact in double (24 + 24 <= 53 significand bits); the K products
 * are summed in double in ascending k; then alpha * s + beta * c is formed in
 * double.  Loop order is i (rows, optionally split over OpenMP threads), k,
 * j: a plain triple loop with one double accumulator row, no blocking.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Full oracle.  out is [M, ldo] doubles; C_in may be NULL when beta == 0. */
int oracle_sgemm_f64(int64_t M, int64_t N, int64_t K, double alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb,
                     double beta, const float *C_in, int64_t ldc,
                     double *out, int64_t ldo, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (M == 0 || N == 0) return 0;
    if (beta != 0.0 && C_in == NULL) return 2;
    const int use_product = (alpha != 0.0 && K > 0);
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(|| : failed)
#endif
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (acc == NULL) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
            for (int64_t i = 0; i < M; ++i) {
                for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
                if (use_product) {
                    for (int64_t k = 0; k < K; ++k) {
                        const double a = (double)A[i * lda + k];
                        const float *brow = B + k * ldb;
                        for (int64_t j = 0; j < N; ++j)
                            acc[j] += a * (double)brow[j];
                    }
                }
                double *orow = out + i * ldo;
                if (beta != 0.0) {
                    const float *crow = C_in + i * ldc;
                    for (int64_t j = 0; j < N; ++j)
                        orow[j] = alpha * acc[j] + beta * (double)crow[j];
                } else {
                    for (int64_t j = 0; j < N; ++j)
                        orow[j] = alpha * acc[j];
                }
            }
            free(acc);
        }
    }
    return failed ? 3 : 0;
}

/* Selected entries (rows[t], cols[t]), t < count, each one length-K fp64 dot
 * product followed by the same epilogue as above. */
int oracle_sgemm_entries_f64(int64_t K, double alpha,
                             const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             double beta, const float *C_in, int64_t ldc,
                             int64_t count, const int64_t *rows,
                             const int64_t *cols, double *out, int nthreads)
{
    if (K < 0 || count < 0) return 1;
    if (beta != 0.0 && C_in == NULL) return 2;
    const int use_product = (alpha != 0.0 && K > 0);
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double s = 0.0;
        if (use_product) {
            for (int64_t k = 0; k < K; ++k)
                s += (double)A[i * lda + k] * (double)B[k * ldb + j];
        }
        double v = alpha * s;
        if (beta != 0.0) v += beta * (double)C_in[i * ldc + j];
        out[t] = v;
    }
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
