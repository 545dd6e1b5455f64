/*
 * CPU oracle for dense GEMM -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this code.  It shares nothing with the CUDA library: no headers, no
 * helpers, no constants.
 *
 * What it computes is the plain definition of GEMM given in "CUDA 算子工程,
 * ch.10 朴素 GEMM 与 Roofline 分析", section 10.1 (the GEMM equation):
 *
 *     C[m][n] = alpha * sum_{k} A[m][k] * B[k][n] + beta * C0[m][n]
 *
 * with row-major storage as in the naive kernel of section 10.2
 * (A[row*K + k], B[k*N + col], C[row*N + col]), generalised to leading
 * dimensions lda, ldb, ldc.  Everything is in fp64.  For every output element
 * the products are summed in increasing k, one after another (no blocking,
 * no reassociation, FMA contraction disabled at build time).  When beta is 0
 * the C0 term is left out entirely and C0 is never read: the ideal-traffic
 * count in "Kernel 性能从何而来" (section "GEMM") assumes that C is not read
 * when beta = 0, so a NaN in C0 must not reach the result.
 *
 * Work is split over host threads by whole output rows; each row is computed
 * by exactly one thread, so the result does not depend on the thread count.
 */
#include <pthread.h>
#include <stdlib.h>

typedef struct {
    long M, N, K;
    double alpha, beta;
    const double *A, *B, *C0;
    long lda, ldb, ldc0;
    double *R;
    long ldr;
    long row_begin, row_end;
} oracle_job;

static void *oracle_rows(void *arg)
{
    oracle_job *j = (oracle_job *)arg;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    if (!acc) return (void *)1;
    for (long m = j->row_begin; m < j->row_end; ++m) {
        for (long n = 0; n < j->N; ++n) acc[n] = 0.0;
        /* i-k-j order: for a fixed (m, n) the k terms are still added in
         * order k = 0, 1, ..., K-1. */
        for (long k = 0; k < j->K; ++k) {
            const double a = j->A[m * j->lda + k];
            const double *brow = j->B + k * j->ldb;
            for (long n = 0; n < j->N; ++n) acc[n] += a * brow[n];
        }
        double *out = j->R + m * j->ldr;
        for (long n = 0; n < j->N; ++n) {
            double r = j->alpha * acc[n];
            if (j->beta != 0.0) r += j->beta * j->C0[m * j->ldc0 + n];
            out[n] = r;
        }
    }
    free(acc);
    return (void *)0;
}

/* R = alpha * A B + beta * C0 (C0 unread when beta == 0).
 * Returns 0 on success, 1 on bad arguments, 2 on a thread/alloc failure. */
int oracle_gemm(long M, long N, long K, double alpha,
                const double *A, long lda, const double *B, long ldb,
                double beta, const double *C0, long ldc0,
                double *R, long ldr, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (M == 0 || N == 0) return 0;
    if (lda < K || ldb < N || ldr < N) return 1;
    if (beta != 0.0 && (!C0 || ldc0 < N)) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)M;

    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return 2; }
    int rc = 0;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->M = M; j->N = N; j->K = K; j->alpha = alpha; j->beta = beta;
        j->A = A; j->B = B; j->C0 = C0; j->lda = lda; j->ldb = ldb; j->ldc0 = ldc0;
        j->R = R; j->ldr = ldr;
        j->row_begin = M * t / nthreads;
        j->row_end = M * (t + 1) / nthreads;
        if (nthreads == 1) {
            if (oracle_rows(j) != (void *)0) rc = 2;
        } else if (pthread_create(&tids[t], NULL, oracle_rows, j) != 0) {
            rc = 2;
            break;
        } else {
            ++started;
        }
    }
    for (int t = 0; t < started; ++t) {
        void *ret = 0;
        pthread_join(tids[t], &ret);
        if (ret != (void *)0) rc = 2;
    }
    free(jobs);
    free(tids);
    return rc;
}
