/*
 * sgemm_oracle.c -- CPU oracle for C = alpha * op(A) * op(B) + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library; the CUDA library never links, includes
 * or calls it, and it shares no code with the CUDA path.
 *
 * What it computes is the plain definition stated at the top of the GEMM
 * handbook page ("GEMM 优化之路", section 问题定义与性能上限): A is M x K, B is
 * K x N, C is M x N, all row-major FP32, and the result is alpha*A*B + beta*C.
 * Tiling, register blocking and pipelining on the pages only reorder the same
 * multiply-adds, so no blocking is written here.
 *
 * Choices (readings of points the pages leave open):
 *  - Every product and sum is taken in double (the pages' own CPU reference
 *    accumulates in float; double makes the oracle far more accurate than any
 *    FP32 result it checks).
 *  - Loop order is i-k-j with a per-row accumulator, the order of the
 *    handbook's CPU reference (section 完整代码, gemm_cpu); rows are independent,
 *    so OpenMP splits them across cores without changing any sum.
 *  - beta == 0 means C is write-only: C_in is not read, so NaN/Inf there do not
 *    propagate (reference-BLAS convention; the pages are silent).
 *  - alpha == 0 or K == 0 means A and B are not read.
 *  - op(X) is X or its transpose (the optimisation guide, step 8: A^T*B and
 *    A*B^T cases).
 *
 * Besides the result it returns, per element, the elementwise error budget
 *     bound_ij = 2*K*2^-24 * (|alpha| * sum_k |a_ik||b_kj| + |beta * c_ij|) + 1e-6
 * used to check an FP32 result, and the number of multiply-adds it performed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_U (1.0 / 16777216.0) /* 2^-24, FP32 unit roundoff */

static inline float opA(int transA, const float *A, int64_t lda, int64_t i, int64_t k) {
    return transA ? A[k * lda + i] : A[i * lda + k];
}

static inline float opB(int transB, const float *B, int64_t ldb, int64_t k, int64_t j) {
    return transB ? B[j * ldb + k] : B[k * ldb + j];
}

/*
 * Full product.  ref and bound are M x N row-major doubles (leading dim N).
 * Returns the number of multiply-adds performed (M*N*K when alpha != 0).
 */
int64_t oracle_sgemm(int transA, int transB, int M, int N, int K, double alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                     const float *C, int64_t ldc, double *ref, double *bound, int threads) {
    int64_t fmas = 0;
    if (M <= 0 || N <= 0) return 0;
    const int use_ab = (alpha != 0.0 && K > 0);
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel reduction(+ : fmas)
#endif
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        double *mag = (double *)malloc(sizeof(double) * (size_t)N);
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int i = 0; i < M; ++i) {
            for (int j = 0; j < N; ++j) acc[j] = 0.0, mag[j] = 0.0;
            if (use_ab) {
                for (int k = 0; k < K; ++k) {
                    const double a = (double)opA(transA, A, lda, i, k);
                    const double aa = fabs(a);
                    if (!transB) {
                        const float *brow = B + (int64_t)k * ldb;
                        for (int j = 0; j < N; ++j) {
                            acc[j] += a * (double)brow[j];
                            mag[j] += aa * fabs((double)brow[j]);
                        }
                    } else {
                        for (int j = 0; j < N; ++j) {
                            const double b = (double)opB(transB, B, ldb, k, j);
                            acc[j] += a * b;
                            mag[j] += aa * fabs(b);
                        }
                    }
                }
                fmas += (int64_t)N * K;
            }
            for (int j = 0; j < N; ++j) {
                const double c = (beta != 0.0) ? (double)C[(int64_t)i * ldc + j] : 0.0;
                const double bc = beta * c;
                ref[(int64_t)i * N + j] = (use_ab ? alpha * acc[j] : 0.0) + bc;
                if (bound)
                    bound[(int64_t)i * N + j] =
                        2.0 * (double)K * ORACLE_U * (fabs(alpha) * mag[j] + fabs(bc)) + 1e-6;
            }
        }
        free(acc);
        free(mag);
    }
    return fmas;
}

/*
 * Selected entries only: ref[t], bound[t] for (rows[t], cols[t]), t < count.
 * Each entry is the same k-ordered double dot product as oracle_sgemm.
 */
int64_t oracle_sgemm_entries(int transA, int transB, int M, int N, int K, double alpha,
                             const float *A, int64_t lda, const float *B, int64_t ldb,
                             double beta, const float *C, int64_t ldc, int64_t count,
                             const int64_t *rows, const int64_t *cols, double *ref,
                             double *bound, int threads) {
    int64_t fmas = 0;
    const int use_ab = (alpha != 0.0 && K > 0);
    (void)M;
    (void)N;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 16) reduction(+ : fmas)
#endif
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double s = 0.0, m = 0.0;
        if (use_ab) {
            for (int k = 0; k < K; ++k) {
                const double a = (double)opA(transA, A, lda, i, k);
                const double b = (double)opB(transB, B, ldb, k, j);
                s += a * b;
                m += fabs(a) * fabs(b);
            }
            fmas += K;
        }
        const double c = (beta != 0.0) ? (double)C[i * ldc + j] : 0.0;
        const double bc = beta * c;
        ref[t] = (use_ab ? alpha * s : 0.0) + bc;
        if (bound) bound[t] = 2.0 * (double)K * ORACLE_U * (fabs(alpha) * m + fabs(bc)) + 1e-6;
    }
    return fmas;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
