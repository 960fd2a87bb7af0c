/*
 * sgemm_oracle.c -- the CPU oracle for C = alpha*A*B + beta*C on row-major
 * float32 matrices.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the bench's CPU-baseline leg call it; the library path never does.  It
 * shares no code, header or table with the CUDA path.
 *
 * What it computes (the plain definition, written out):
 *
 *   C_ref[i][j] = alpha * sum_{p=0}^{K-1} A[i][p] * B[p][j]  +  beta * C0[i][j]
 *   S[i][j]     =         sum_{p=0}^{K-1} |A[i][p]| * |B[p][j]|
 *
 * -- "Learn: Optimizing GEMM", section 3 "Rung 0 -- Naive (recap)": one
 *    output element is the length-K dot product of row i of A and column j
 *    of B, scaled by alpha, plus beta times the old C, all three matrices
 *    row-major (element [i][j] at base + i*ld + j).
 * -- "How a Matmul Kernel Gets Fast", section 1 "The problem, and what
 *    cuBLAS is": GEMM is C = alpha*A*B + beta*C.
 * -- "Writing a Fast Matmul in CUDA, Step by Step", "Step 1: the problem and
 *    the yardstick": results are checked against a float64 dot product on
 *    the CPU.
 *
 * Precision: every product A[i][p]*B[p][j] of two floats is exact in
 * double (24+24 significant bits < 53), and the sum runs in double in
 * ascending p.  The result stays in double (it is not rounded to float).
 * S is the |A||B| matrix that scales the acceptance bound
 * |C - C_ref| <= 4*K*2^-24*S + 1e-6.
 *
 * Conventions the pages leave open (BLAS readings):
 *   beta == 0  : C0 is not read (so NaN in an uninitialised C0 does not
 *                propagate); C_ref = alpha * sum.
 *   K == 0 or alpha == 0 : the sum term is dropped, C_ref = beta*C0.
 *   M == 0 or N == 0     : nothing to do.
 *
 * Two routines compute the same numbers in two loop orders:
 *   oracle_sgemm         i - p - j with a double row accumulator (each
 *                        element still sums its products in ascending p,
 *                        so it is bit-identical to the dot form);
 *   oracle_sgemm_entries one plain dot product per requested (i, j).
 * A third, oracle_fp32_chain_entries, is a diagnostic, not the oracle: the
 * float32 fused-multiply-add chain in ascending k, which any kernel that
 * keeps that order reproduces bit for bit ("Writing a Fast Matmul in CUDA",
 * Step 1: kernels that add the products in the order k = 0 .. n-1 agree to
 * the last bit).
 *
 * Build: plain C11, gcc -O2 -ffp-contract=off -pthread (no fast-math, no
 * intrinsics; the same source builds on x86-64 and aarch64).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_NOMEM (-2)

typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    const float *A, *B, *C0;
    int64_t lda, ldb, ldc;
    double *Cref, *S;
    int64_t ldr;
    int64_t row_begin, row_end;
    uint64_t fma_count;
    int status;
} oracle_job;

static int check_dims(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return ORACLE_ERR_ARG;
    if (lda < (K > 1 ? K : 1)) return ORACLE_ERR_ARG;
    if (ldb < (N > 1 ? N : 1)) return ORACLE_ERR_ARG;
    if (ldc < (N > 1 ? N : 1)) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/* Rows [row_begin, row_end) of the full product, i - p - j order. */
static void *oracle_rows(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int64_t N = job->N, K = job->K;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *sacc = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!acc || !sacc) {
        free(acc);
        free(sacc);
        job->status = ORACLE_ERR_NOMEM;
        return NULL;
    }
    uint64_t fmas = 0;
    const int use_sum = (K > 0 && job->alpha != 0.0);
    for (int64_t i = job->row_begin; i < job->row_end; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            acc[j] = 0.0;
            sacc[j] = 0.0;
        }
        const float *a_row = job->A + i * job->lda;
        for (int64_t p = 0; p < K; ++p) {
            const double a = (double)a_row[p];
            const double abs_a = fabs(a);
            const float *b_row = job->B + p * job->ldb;
            for (int64_t j = 0; j < N; ++j) {
                const double b = (double)b_row[j];
                acc[j] = acc[j] + a * b;            /* product exact in double */
                sacc[j] = sacc[j] + abs_a * fabs(b);
                fmas++;
            }
        }
        double *c_out = job->Cref + i * job->ldr;
        double *s_out = job->S ? job->S + i * job->ldr : NULL;
        for (int64_t j = 0; j < N; ++j) {
            double c = use_sum ? job->alpha * acc[j] : 0.0;
            if (job->beta != 0.0) c = c + job->beta * (double)job->C0[i * job->ldc + j];
            c_out[j] = c;
            if (s_out) s_out[j] = sacc[j];
        }
    }
    free(acc);
    free(sacc);
    job->fma_count = fmas;
    job->status = ORACLE_OK;
    return NULL;
}

/*
 * Full product.  Cref and S (S may be NULL) are M x N doubles with row
 * stride ldr.  nthreads <= 1 runs on the calling thread; otherwise rows are
 * split into nthreads contiguous bands, one POSIX thread each (no thread
 * changes any element's summation order).  If fma_count is not NULL it
 * receives the number of inner multiply-add steps executed (M*N*K).
 */
int oracle_sgemm(int64_t M, int64_t N, int64_t K, double alpha, const float *A, int64_t lda,
                 const float *B, int64_t ldb, double beta, const float *C0, int64_t ldc,
                 double *Cref, double *S, int64_t ldr, int nthreads, uint64_t *fma_count)
{
    int rc = check_dims(M, N, K, lda, ldb, ldc);
    if (rc != ORACLE_OK) return rc;
    if (ldr < (N > 1 ? N : 1)) return ORACLE_ERR_ARG;
    if (fma_count) *fma_count = 0;
    if (M == 0 || N == 0) return ORACLE_OK;
    if ((K > 0 && (!A || !B)) || !Cref || (beta != 0.0 && !C0)) return ORACLE_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)M;

    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ERR_NOMEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->M = M; j->N = N; j->K = K;
        j->alpha = alpha; j->beta = beta;
        j->A = A; j->B = B; j->C0 = C0;
        j->lda = lda; j->ldb = ldb; j->ldc = ldc;
        j->Cref = Cref; j->S = S; j->ldr = ldr;
        j->row_begin = (M * t) / nthreads;
        j->row_end = (M * (t + 1)) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, oracle_rows, &jobs[t]) != 0) break;
        started = t;
    }
    /* Any band whose thread did not start runs here, on the caller. */
    for (int t = started + 1; t < nthreads; ++t) oracle_rows(&jobs[t]);
    oracle_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);

    rc = ORACLE_OK;
    uint64_t total = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (jobs[t].status != ORACLE_OK) rc = jobs[t].status;
        total += jobs[t].fma_count;
    }
    if (fma_count) *fma_count = total;
    free(jobs);
    free(tids);
    return rc;
}

/*
 * Selected entries, one plain dot product each: for e in [0, n),
 * cref[e] = C_ref[rows[e]][cols[e]] and s[e] = S[rows[e]][cols[e]]
 * (s may be NULL).  Cost K per entry, so a sample of a very large product
 * is cheap.  Indices out of range give ORACLE_ERR_ARG.
 */
int oracle_sgemm_entries(int64_t M, int64_t N, int64_t K, double alpha, const float *A, int64_t lda,
                         const float *B, int64_t ldb, double beta, const float *C0, int64_t ldc,
                         int64_t n, const int64_t *rows, const int64_t *cols, double *cref, double *s)
{
    int rc = check_dims(M, N, K, lda, ldb, ldc);
    if (rc != ORACLE_OK) return rc;
    if (n < 0 || (n > 0 && (!rows || !cols || !cref))) return ORACLE_ERR_ARG;
    const int use_sum = (K > 0 && alpha != 0.0);
    for (int64_t e = 0; e < n; ++e) {
        const int64_t i = rows[e], j = cols[e];
        if (i < 0 || i >= M || j < 0 || j >= N) return ORACLE_ERR_ARG;
        double dot = 0.0, sabs = 0.0;
        for (int64_t p = 0; p < K; ++p) {
            const double a = (double)A[i * lda + p];
            const double b = (double)B[p * ldb + j];
            dot = dot + a * b;
            sabs = sabs + fabs(a) * fabs(b);
        }
        double c = use_sum ? alpha * dot : 0.0;
        if (beta != 0.0) c = c + beta * (double)C0[i * ldc + j];
        cref[e] = c;
        if (s) s[e] = sabs;
    }
    return ORACLE_OK;
}

/*
 * Diagnostic: the float32 chain acc = fmaf(A[i][p], B[p][j], acc) for
 * p = 0 .. K-1 from acc = +0, returned unscaled (alpha and beta are not
 * applied).  A kernel that accumulates each output in ascending k with
 * single-rounding fused multiply-adds returns exactly these floats when
 * alpha == 1 and beta == 0.
 */
int oracle_fp32_chain_entries(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                              const float *B, int64_t ldb, int64_t n, const int64_t *rows,
                              const int64_t *cols, float *out)
{
    int rc = check_dims(M, N, K, lda, ldb, N > 1 ? N : 1);
    if (rc != ORACLE_OK) return rc;
    if (n < 0 || (n > 0 && (!rows || !cols || !out))) return ORACLE_ERR_ARG;
    for (int64_t e = 0; e < n; ++e) {
        const int64_t i = rows[e], j = cols[e];
        if (i < 0 || i >= M || j < 0 || j >= N) return ORACLE_ERR_ARG;
        float acc = 0.0f;
        for (int64_t p = 0; p < K; ++p) acc = fmaf(A[i * lda + p], B[p * ldb + j], acc);
        out[e] = acc;
    }
    return ORACLE_OK;
}
