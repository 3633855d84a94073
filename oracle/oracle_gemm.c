/*
 * Oracle for the dense GEMM C = A·B.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * may load this library.  The CUDA path neither links nor calls it, and it
 * shares no code, header or constant with the CUDA path.
 *
 * What it computes (the plain definition, nothing more):
 *
 *   C[i][j] = sum_{k=0}^{K-1} A(i,k) * B(k,j)        accumulated in FP64,
 *   S[i][j] = sum_{k=0}^{K-1} |A(i,k) * B(k,j)|      accumulated in FP64,
 *
 * with each sum taken left to right, k = 0, 1, ..., K-1.
 *
 *  - "GEMM 性能优化", section 指标与目标: C = A·B, 2·M·N·K flops.
 *  - "GEMM 性能优化", 台阶 1 (Shared Memory Tiling): the sum runs along K, so
 *    splitting K into slices and adding the partial products gives the same
 *    matrix (blocked-matrix identity).  The oracle does no blocking.
 *  - "PMPP Chapter 06: Performance considerations", section 1 (Corner
 *    Turning example): A and C row-major, B column-major, so element (k,j) of
 *    B lives at B[j*ld + k]; out-of-range rows/columns do not exist and
 *    only C[i][j] with i < M, j < N is written.
 *
 * Layouts: A(i,k) = A[i*lda + k]; B(k,j) = B[k*ldb + j] (row-major, layout 0)
 * or B[j*ldb + k] (column-major, layout 1); C and S row-major with ldc.
 * Inputs are FP64 copies of the exact values the GPU reads (FP32 values, or
 * BF16-rounded values), so every product a*b is exact in FP64.
 *
 * S is the per-element error scale used by the parity tolerance
 * |C_gpu - C| <= tol * S.
 *
 * Work is split over threads by whole rows of C; the k order of every element
 * is the same whatever the thread count, so results do not depend on it.
 * Build with -ffp-contract=off so no compiler fuses a*b+c into an FMA and the
 * results are bit-identical on every host.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

#define ORACLE_B_ROW_MAJOR 0
#define ORACLE_B_COL_MAJOR 1

typedef struct {
    int layout_b;
    int64_t row_begin, row_end, N, K;
    const double *A;
    int64_t lda;
    const double *B;
    int64_t ldb;
    double *C;
    int64_t ldc;
    double *S;
    int64_t lds;
} oracle_rows_t;

static void oracle_rows(const oracle_rows_t *w)
{
    for (int64_t i = w->row_begin; i < w->row_end; ++i) {
        double *c = w->C + i * w->ldc;
        double *s = w->S + i * w->lds;
        for (int64_t j = 0; j < w->N; ++j) {
            c[j] = 0.0;
            s[j] = 0.0;
        }
        /* i-k-j loop order: for a fixed (i, j) the terms are still added in
         * k order 0..K-1; the order only keeps B's rows streaming. */
        for (int64_t k = 0; k < w->K; ++k) {
            const double a = w->A[i * w->lda + k];
            for (int64_t j = 0; j < w->N; ++j) {
                const double b = (w->layout_b == ORACLE_B_ROW_MAJOR)
                                     ? w->B[k * w->ldb + j]
                                     : w->B[j * w->ldb + k];
                const double p = a * b;
                c[j] += p;
                s[j] += fabs(p);
            }
        }
    }
}

static void *oracle_thread(void *arg)
{
    oracle_rows((const oracle_rows_t *)arg);
    return NULL;
}

/* Number of worker threads a call with nthreads <= 0 uses. */
int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * C (M x N, ldc) and S (M x N, lds) <- the sums above.
 * Returns 0, -1 on a bad argument (nothing written), or -2 when the thread
 * bookkeeping could not be allocated (nothing written).  A worker thread that
 * cannot be started has its rows computed on the calling thread instead.
 */
int oracle_gemm_f64(int layout_b, int64_t M, int64_t N, int64_t K,
                    const double *A, int64_t lda,
                    const double *B, int64_t ldb,
                    double *C, int64_t ldc,
                    double *S, int64_t lds,
                    int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (layout_b != ORACLE_B_ROW_MAJOR && layout_b != ORACLE_B_COL_MAJOR) return -1;
    if (M == 0 || N == 0) return 0;
    if (!C || !S || ldc < N || lds < N) return -1;
    if (K > 0) {
        if (!A || !B || lda < K) return -1;
        if (layout_b == ORACLE_B_ROW_MAJOR && ldb < N) return -1;
        if (layout_b == ORACLE_B_COL_MAJOR && ldb < K) return -1;
    }
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > M) nthreads = (int)M;

    oracle_rows_t *work = (oracle_rows_t *)calloc((size_t)nthreads, sizeof(oracle_rows_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int *started = (int *)calloc((size_t)nthreads, sizeof(int));
    if (!work || !tid || !started) {
        free(work); free(tid); free(started);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        oracle_rows_t *w = &work[t];
        w->layout_b = layout_b;
        w->row_begin = M * t / nthreads;
        w->row_end = M * (t + 1) / nthreads;
        w->N = N; w->K = K;
        w->A = A; w->lda = lda;
        w->B = B; w->ldb = ldb;
        w->C = C; w->ldc = ldc;
        w->S = S; w->lds = lds;
        if (t > 0) started[t] = (pthread_create(&tid[t], NULL, oracle_thread, w) == 0);
    }
    oracle_rows(&work[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) {
            pthread_join(tid[t], NULL);
        } else {
            oracle_rows(&work[t]);
        }
    }
    free(work); free(tid); free(started);
    return 0;
}
