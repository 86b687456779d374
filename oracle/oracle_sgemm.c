/*
 * Reference (oracle) for single-precision GEMM, C = alpha * A * B + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test-suite, the package's smoke check and the benchmark's
 * CPU-baseline arm do.  It shares no code, header or constant with the CUDA
 * library, and it includes no CUDA header.
 *
 * What it computes is the plain definition of the product, widened to double:
 *
 *   Cref[i][j] = alpha * sum_{k<K} A[i][k] * B[k][j] + beta * C[i][j]
 *
 * - "Optimizing Matrix Multiply on CUDA, Part 1", section "Counting the Work":
 *   C[i][j] is the dot product of row i of A with column j of B.
 * - "GEMM from Scratch", Module 02 ("One Thread Per Output"): the same dot
 *   product over row-major operands (A[x*K+i], B[i*N+y], C[x*N+y]) followed by
 *   the epilogue alpha*tmp + beta*C.
 * - "Optimizing CUDA matmul, steps 4 to 6", section "Five paths, one table":
 *   every path is checked at every element against a double-precision CPU
 *   reference.
 *
 * Readings where the pages are silent (the BLAS conventions):
 * - beta == 0: C is not read, so a NaN already in C does not reach the result.
 * - alpha == 0 or K == 0: the product is not formed; Cref = beta * C.
 * - Leading dimensions lda, ldb, ldc may exceed the row length; elements in
 *   the gap are never read.
 *
 * Besides Cref the oracle returns absprod[i][j] = sum_k |A[i][k]| * |B[k][j]|,
 * the quantity the elementwise FP32 error bound is stated in.
 *
 * Each product of two floats is exact in double (24 + 24 significand bits),
 * and the double sum of K such products is accurate to K * 2^-53 relative to
 * absprod, far below the FP32 rounding the GPU result is judged against.
 *
 * Loop order is i-k-j (row of Cref held in a double accumulator while the k
 * loop walks rows of B); rows are shared out to POSIX threads.  This is still
 * the textbook triple loop: no blocking, no reordering of the k sum.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    const float *A; int64_t lda;
    const float *B; int64_t ldb;
    const float *C; int64_t ldc;
    const int64_t *rows; int64_t nrows;
    double *out;     /* nrows x N, row stride N */
    double *absprod; /* nrows x N or NULL */
    int64_t first, last; /* this worker's share of [0, nrows) */
} oracle_job;

static void oracle_one_row(const oracle_job *job, int64_t r, double *acc, double *abs_acc)
{
    const int64_t i = job->rows[r];
    const int64_t N = job->N;
    for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; abs_acc[j] = 0.0; }

    if (job->alpha != 0.0) {
        for (int64_t k = 0; k < job->K; ++k) {
            const double a = (double)job->A[i * job->lda + k];
            const double abs_a = fabs(a);
            const float *brow = job->B + k * job->ldb;
            for (int64_t j = 0; j < N; ++j) {
                const double b = (double)brow[j];
                acc[j] += a * b;
                abs_acc[j] += abs_a * fabs(b);
            }
        }
    }

    double *dst = job->out + r * N;
    for (int64_t j = 0; j < N; ++j) {
        double v = job->alpha * acc[j];
        if (job->beta != 0.0) v += job->beta * (double)job->C[i * job->ldc + j];
        dst[j] = v;
    }
    if (job->absprod) memcpy(job->absprod + r * N, abs_acc, (size_t)N * sizeof(double));
}

static void *oracle_worker(void *arg)
{
    const oracle_job *job = (const oracle_job *)arg;
    const int64_t N = job->N > 0 ? job->N : 1;
    double *acc = (double *)malloc((size_t)N * sizeof(double));
    double *abs_acc = (double *)malloc((size_t)N * sizeof(double));
    if (!acc || !abs_acc) { free(acc); free(abs_acc); return (void *)1; }
    for (int64_t r = job->first; r < job->last; ++r) oracle_one_row(job, r, acc, abs_acc);
    free(acc);
    free(abs_acc);
    return NULL;
}

/* Number of threads the oracle uses when asked for 0 (all online cores). */
int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Compute the rows listed in `rows` (each in [0, M)) of the reference result.
 * out and absprod (absprod may be NULL) are nrows x N, row-major, stride N.
 * C may be NULL when beta == 0.  Returns 0 on success, a negative value on a
 * bad argument, 1 if a worker could not allocate its row buffers.
 */
int oracle_sgemm_rows(int64_t M, int64_t N, int64_t K, double alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      double beta, const float *C, int64_t ldc,
                      const int64_t *rows, int64_t nrows,
                      double *out, double *absprod, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (!rows || !out) return -2;
    if (alpha != 0.0 && K > 0 && (!A || !B || lda < K || ldb < N)) return -3;
    if (beta != 0.0 && (!C || ldc < N)) return -4;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -5;

    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > nrows) nthreads = (int)nrows;

    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return 1; }

    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->M = M; j->N = N; j->K = K; j->alpha = alpha; j->beta = beta;
        j->A = A; j->lda = lda; j->B = B; j->ldb = ldb; j->C = C; j->ldc = ldc;
        j->rows = rows; j->nrows = nrows; j->out = out; j->absprod = absprod;
        j->first = nrows * t / nthreads;
        j->last = nrows * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) != 0) break;
        started = t;
    }
    /* Rows of workers that could not be started are done on this thread. */
    if (oracle_worker(&jobs[0]) != NULL) rc = 1;
    for (int t = started + 1; t < nthreads; ++t)
        if (oracle_worker(&jobs[t]) != NULL) rc = 1;
    for (int t = 1; t <= started; ++t) {
        void *ret = NULL;
        pthread_join(tids[t], &ret);
        if (ret != NULL) rc = 1;
    }
    free(jobs);
    free(tids);
    return rc;
}
