/*
 * gemm_oracle.c -- plain CPU reference for the pipelined tiled GEMM C = A * B.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline / reference legs load this file's library.  It shares no code
 * with the GPU library: it has its own binary16 decoder and its own loops.
 *
 * What it computes, and why that is the whole specification:
 *   "Pipeline GPU Kernel" (skill page), Step 5 "Verify correctness", item 4:
 *   software pipelining reorders loads only and never changes the arithmetic.
 *   So the pipelined kernel must reach the plain matrix product.  This file
 *   writes that product out with no tiling, blocking or reordering:
 *
 *     INT8 -> INT32 (the pages' IGEMM, IMMA with int32 accumulate):
 *         C[i][j] = sum_{k<K} (int64) A[i][k] * (int64) B[k][j]
 *       accumulated exactly in int64, then checked to fit int32.
 *     FP16 -> FP32 (the pages' HMMA GEMM):
 *         C[i][j] = (float) sum_{k<K} (double) A[i][k] * (double) B[k][j]
 *       every product of two binary16 values is exact in binary64; the sum is
 *       accumulated in binary64 in k order and rounded once to binary32
 *       (round to nearest even).
 *
 *   A is M x K row-major (lda = K), B is K x N row-major (ldb = N), C is M x N
 *   row-major (ldc = N).  K = 0 gives the empty sum, C = 0.
 *
 * Also here, from the same page, Steps 1 and 2:
 *   - the shared-memory budget of one stage, smem_a = BM*BK*sizeof(T),
 *     smem_b = BK*BN*sizeof(T), and of the doubled buffer 2*smem_a + 2*smem_b;
 *   - the per-tile compute/load ratio 2*BM*BN*BK / ((BM*BK + BK*BN)*sizeof(T)).
 *
 * Loop order is i-k-j (row of A times rows of B), threads split the rows.
 * Compile without -ffast-math and with -ffp-contract=off.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16 -> binary64, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits.  Exponent field 0 encodes
 * subnormals f * 2^-24, field 31 encodes infinities (f = 0) and NaNs. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

typedef struct {
    int64_t M, N, K;
    const void *A, *B;
    void *C;               /* output rows, packed in the order of `rows` */
    const int64_t *rows;   /* NULL: all rows 0..M-1 */
    int64_t r0, r1;        /* range of positions in the row list */
    int overflow;          /* int8 path: a sum left the int32 range */
    int status;
} oracle_job;

static void *rows_s8(void *arg)
{
    oracle_job *jb = (oracle_job *)arg;
    const int8_t *A = (const int8_t *)jb->A;
    const int8_t *B = (const int8_t *)jb->B;
    int32_t *C = (int32_t *)jb->C;
    int64_t N = jb->N, K = jb->K;
    int64_t *acc = (int64_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
    if (!acc) { jb->status = -2; return NULL; }
    for (int64_t p = jb->r0; p < jb->r1; ++p) {
        int64_t i = jb->rows ? jb->rows[p] : p;
        for (int64_t j = 0; j < N; ++j) acc[j] = 0;
        for (int64_t k = 0; k < K; ++k) {
            int64_t a = (int64_t)A[i * K + k];
            const int8_t *brow = B + k * N;
            for (int64_t j = 0; j < N; ++j) acc[j] += a * (int64_t)brow[j];
        }
        for (int64_t j = 0; j < N; ++j) {
            if (acc[j] > INT32_MAX || acc[j] < INT32_MIN) jb->overflow = 1;
            C[p * N + j] = (int32_t)acc[j];
        }
    }
    free(acc);
    return NULL;
}

static void *rows_f16(void *arg)
{
    oracle_job *jb = (oracle_job *)arg;
    const uint16_t *A = (const uint16_t *)jb->A;
    const uint16_t *B = (const uint16_t *)jb->B;
    float *C = (float *)jb->C;
    int64_t N = jb->N, K = jb->K;
    double *acc = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *brow = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!acc || !brow) { free(acc); free(brow); jb->status = -2; return NULL; }
    for (int64_t p = jb->r0; p < jb->r1; ++p) {
        int64_t i = jb->rows ? jb->rows[p] : p;
        for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = oracle_f16_to_f64(A[i * K + k]);
            const uint16_t *b = B + k * N;
            for (int64_t j = 0; j < N; ++j) brow[j] = oracle_f16_to_f64(b[j]);
            for (int64_t j = 0; j < N; ++j) acc[j] += a * brow[j];
        }
        for (int64_t j = 0; j < N; ++j) C[p * N + j] = (float)acc[j];
    }
    free(acc);
    free(brow);
    return NULL;
}

/* Runs `fn` over the row positions [0, nrows) with `threads` POSIX threads.
 * Returns 0, 1 (int32 overflow seen), -1 (bad arguments) or -2 (no memory). */
static int run_rows(void *(*fn)(void *), int64_t M, int64_t N, int64_t K,
                    const void *A, const void *B, const int64_t *rows,
                    int64_t nrows, void *C, int threads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (!C || (K > 0 && (!A || !B))) return -1;
    if (rows)
        for (int64_t p = 0; p < nrows; ++p)
            if (rows[p] < 0 || rows[p] >= M) return -1;
    if (threads < 1) threads = 1;
    if (threads > nrows) threads = (int)nrows;
    oracle_job *jobs = (oracle_job *)calloc((size_t)threads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -2; }
    int64_t per = (nrows + threads - 1) / threads;
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        oracle_job *jb = &jobs[t];
        jb->M = M; jb->N = N; jb->K = K; jb->A = A; jb->B = B; jb->C = C;
        jb->rows = rows;
        jb->r0 = (int64_t)t * per;
        jb->r1 = jb->r0 + per < nrows ? jb->r0 + per : nrows;
        if (jb->r0 >= jb->r1) continue;
        if (threads == 1 || pthread_create(&tids[t], NULL, fn, jb) != 0) {
            fn(jb);            /* run inline when single-threaded or on failure */
            tids[t] = 0;
        } else {
            ++started;
        }
    }
    int rc = 0;
    for (int t = 0; t < threads; ++t) {
        if (tids[t]) pthread_join(tids[t], NULL);
        if (jobs[t].status) rc = jobs[t].status;
        else if (jobs[t].overflow && rc == 0) rc = 1;
    }
    (void)started;
    free(jobs);
    free(tids);
    return rc;
}

/* INT8 x INT8 -> INT32.  rows == NULL computes every row into C (M x N);
 * otherwise C receives the listed rows, packed (nrows x N). */
int oracle_gemm_s8s8s32(int64_t M, int64_t N, int64_t K, const int8_t *A,
                        const int8_t *B, const int64_t *rows, int64_t nrows,
                        int32_t *C, int threads)
{
    if (!rows) nrows = M;
    return run_rows(rows_s8, M, N, K, A, B, rows, nrows, C, threads);
}

/* FP16 x FP16 -> FP32 (fp64 accumulation, one rounding).  A and B hold the
 * raw binary16 bit patterns.  Row selection as above. */
int oracle_gemm_f16f32(int64_t M, int64_t N, int64_t K, const uint16_t *A,
                       const uint16_t *B, const int64_t *rows, int64_t nrows,
                       float *C, int threads)
{
    if (!rows) nrows = M;
    return run_rows(rows_f16, M, N, K, A, B, rows, nrows, C, threads);
}

/* Step 1 of the skill page: bytes of one A tile and one B tile. */
int64_t oracle_smem_a_bytes(int64_t BM, int64_t BK, int64_t elem_bytes)
{
    return BM * BK * elem_bytes;
}

int64_t oracle_smem_b_bytes(int64_t BK, int64_t BN, int64_t elem_bytes)
{
    return BK * BN * elem_bytes;
}

/* Step 1: the doubled buffer, smem_a * 2 + smem_b * 2. */
int64_t oracle_smem_doubled_bytes(int64_t BM, int64_t BN, int64_t BK, int64_t elem_bytes)
{
    return oracle_smem_a_bytes(BM, BK, elem_bytes) * 2 +
           oracle_smem_b_bytes(BK, BN, elem_bytes) * 2;
}

/* Step 2: multiply-adds count two flops; the tile loads one A and one B tile. */
double oracle_compute_load_ratio(int64_t BM, int64_t BN, int64_t BK, int64_t elem_bytes)
{
    double flops = 2.0 * (double)BM * (double)BN * (double)BK;
    double bytes = (double)(BM * BK + BK * BN) * (double)elem_bytes;
    return flops / bytes;
}
