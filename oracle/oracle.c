/*
 * oracle.c -- plain, slow, obviously correct CPU reference for the tiled
 * matrix multiply.  TEST INFRASTRUCTURE ONLY: the product path (libtgemm and
 * its Python binding) never links, loads or calls this file; only the test
 * suite, the smoke check and the bench's CPU-baseline leg do.
 *
 * What it computes (hecess.blogspot.com "[Multi-Core & GPU Programming] CUDA -
 * Matrix Multiplication", section "[Matrix Multiplication]": the triple loop
 * that adds M(i,k)*N(k,j) into P(i,j), and the variant right after it that keeps
 * the running sum in a local "sum" and stores P(i,j) once):
 *
 *     P(i,j) = sum_{k=0}^{K-1} M(i,k) * N(k,j)
 *
 * generalised from the page's square Width x Width case to rectangular
 * row-major m x k times k x n with independent leading dimensions (the page's
 * flattened index M[row*width+k], N[k*width+col] of section "[Coalescing]",
 * with "width" replaced by a leading dimension per matrix).  Indices are
 * 0-based, as in the page's worked 4x4 example.
 *
 * Every product and every partial sum is formed in IEEE double precision
 * (fp64), starting from 0 and adding the terms in ascending k.  Inputs stored
 * as fp32 or as bf16 bit patterns are widened to double exactly before use.
 *
 * Alongside P it returns D(i,j) = sum_k |M(i,k)| * |N(k,j)|, the scale that
 * the error measure |P_gpu - P| / D divides by.
 *
 * Loop order.  oracle_gemm visits (i, k, j) -- for each row i, for k
 * ascending, it adds M(i,k)*N(k,j) into the fp64 accumulator of every j of
 * that row.  For every single (i,j) the terms still enter in ascending k into
 * one fp64 running sum that starts at 0, exactly as in the page's loop; only
 * the interleaving between different (i,j) differs, and that cannot change a
 * single bit of any result.  oracle_gemm_entries evaluates chosen (i,j) one at
 * a time with the page's own i-j-k running-sum loop.  Rows are split over
 * POSIX threads; each thread owns whole rows, so the result does not depend on
 * the thread count.
 *
 * dtype codes for the stored inputs: 0 = float64, 1 = float32, 2 = bf16
 * (uint16 bit patterns; the value is the fp32 whose upper 16 bits they are).
 *
 * Build: cc -O2 -std=c11 -fPIC -shared -pthread oracle.c -o liboracle.so
 * (no -ffast-math: the fp64 arithmetic must stay IEEE, no contraction either:
 * -ffp-contract=off keeps each product rounded before it is added).
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F64 = 0, ORACLE_F32 = 1, ORACLE_BF16 = 2 };

/* Exact widening of one stored element to double. */
static double oracle_load(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_F64)
        return ((const double *)base)[idx];
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    /* bf16: the 16 stored bits are the top half of an fp32 bit pattern. */
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Whole row of N widened into a double buffer (the j loop then runs over
 * plain doubles). */
static void oracle_load_row(const void *N, int dtype, int64_t row_off,
                            int64_t n, double *out)
{
    for (int64_t j = 0; j < n; ++j)
        out[j] = oracle_load(N, dtype, row_off + j);
}

typedef struct {
    int64_t m, n, k;
    const void *M; int64_t ldm; int mtype;
    const void *N; int64_t ldn; int ntype;
    double *P; double *D; int64_t ldp;
    int64_t row_begin, row_end;
    int status;
} oracle_job;

static void *oracle_rows(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int64_t n = job->n, k = job->k;
    double *nrow = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    double *accp = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    double *accd = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!nrow || !accp || !accd) {
        job->status = 1;
        free(nrow); free(accp); free(accd);
        return NULL;
    }
    for (int64_t i = job->row_begin; i < job->row_end; ++i) {
        for (int64_t j = 0; j < n; ++j) { accp[j] = 0.0; accd[j] = 0.0; }
        for (int64_t kk = 0; kk < k; ++kk) {
            const double a = oracle_load(job->M, job->mtype, i * job->ldm + kk);
            const double abs_a = fabs(a);
            oracle_load_row(job->N, job->ntype, kk * job->ldn, n, nrow);
            for (int64_t j = 0; j < n; ++j) {
                accp[j] += a * nrow[j];
                accd[j] += abs_a * fabs(nrow[j]);
            }
        }
        for (int64_t j = 0; j < n; ++j) {
            job->P[i * job->ldp + j] = accp[j];
            if (job->D) job->D[i * job->ldp + j] = accd[j];
        }
    }
    free(nrow); free(accp); free(accd);
    return NULL;
}

/* Number of host cores this process may run on. */
int oracle_available_cores(void)
{
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof set, &set) == 0) {
        int c = CPU_COUNT(&set);
        if (c > 0) return c;
    }
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

/*
 * P (m x n, leading dimension ldp) = M (m x k, ldm) * N (k x n, ldn), in fp64.
 * D, if not NULL, receives sum_k |M(i,k)|*|N(k,j)| with the same layout.
 * nthreads <= 0 means every available core.  Returns 0 on success, 1 on bad
 * arguments, 2 on allocation or thread failure.
 */
int oracle_gemm(int64_t m, int64_t n, int64_t k,
                const void *M, int64_t ldm, int mtype,
                const void *N, int64_t ldn, int ntype,
                double *P, double *D, int64_t ldp, int nthreads)
{
    if (m < 0 || n < 0 || k < 0) return 1;
    if (m == 0 || n == 0) return 0;
    if (!P || ldp < n) return 1;
    if (k > 0 && (!M || !N || ldm < k || ldn < n)) return 1;
    if (mtype < 0 || mtype > 2 || ntype < 0 || ntype > 2) return 1;

    int t = nthreads > 0 ? nthreads : oracle_available_cores();
    if (t > m) t = (int)m;
    oracle_job *jobs = (oracle_job *)calloc((size_t)t, sizeof *jobs);
    pthread_t *tids = (pthread_t *)calloc((size_t)t, sizeof *tids);
    if (!jobs || !tids) { free(jobs); free(tids); return 2; }

    int started = 0, status = 0;
    for (int w = 0; w < t; ++w) {
        oracle_job *j = &jobs[w];
        j->m = m; j->n = n; j->k = k;
        j->M = M; j->ldm = ldm; j->mtype = mtype;
        j->N = N; j->ldn = ldn; j->ntype = ntype;
        j->P = P; j->D = D; j->ldp = ldp;
        j->row_begin = m * w / t;
        j->row_end = m * (w + 1) / t;
        if (t == 1) {
            oracle_rows(j);
        } else if (pthread_create(&tids[w], NULL, oracle_rows, j) == 0) {
            ++started;
        } else {
            oracle_rows(j);   /* could not spawn: do the rows here */
        }
    }
    if (t > 1)
        for (int w = 0; w < t; ++w)
            if (tids[w]) pthread_join(tids[w], NULL);
    for (int w = 0; w < t; ++w)
        if (jobs[w].status) status = 2;
    (void)started;
    free(jobs); free(tids);
    return status;
}

/*
 * Chosen entries only: for each c < count, P[c] = sum_k M(rows[c],k) *
 * N(k,cols[c]) and D[c] = sum_k |M(rows[c],k)|*|N(k,cols[c])|, each a single
 * fp64 running sum over ascending k -- the page's per-element loop written
 * out.  Used to check outputs of problems too large for oracle_gemm.
 * Returns 0 on success, 1 on bad arguments.
 */
int oracle_gemm_entries(int64_t m, int64_t n, int64_t k,
                        const void *M, int64_t ldm, int mtype,
                        const void *N, int64_t ldn, int ntype,
                        const int64_t *rows, const int64_t *cols, int64_t count,
                        double *P, double *D)
{
    if (m < 0 || n < 0 || k < 0 || count < 0) return 1;
    if (count == 0) return 0;
    if (!rows || !cols || !P) return 1;
    if (k > 0 && (!M || !N || ldm < k || ldn < n)) return 1;
    for (int64_t c = 0; c < count; ++c) {
        const int64_t i = rows[c], j = cols[c];
        if (i < 0 || i >= m || j < 0 || j >= n) return 1;
        double sum = 0.0, sum_abs = 0.0;
        for (int64_t kk = 0; kk < k; ++kk) {
            const double a = oracle_load(M, mtype, i * ldm + kk);
            const double b = oracle_load(N, ntype, kk * ldn + j);
            sum += a * b;
            sum_abs += fabs(a) * fabs(b);
        }
        P[c] = sum;
        if (D) D[c] = sum_abs;
    }
    return 0;
}
