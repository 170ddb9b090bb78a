/*
 * CPU oracle for the dense matrix multiply C = A x B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no source, header or constant with the CUDA
 * library.
 *
 * What it computes (the definition, written out, no blocking or reordering):
 *
 *   C[i][j] = sum_{kk < k} A[i][kk] * B[kk][j]
 *
 * This is the product the TPU's 256x256 INT8 multiply-accumulate array
 * evaluates when A and B are fed through it in several passes ("文章导读:
 * Motivation for and Evaluation of the First Tensor Processing Unit",
 * sections "TPU介绍" and "TPU使用的技术"), and the operation whose tiling the
 * patent CN114238853A ("一種矩陣乘分片配置選擇方法及系統", claim 4 S2: an m*k
 * left matrix times a k*n right matrix) plans.
 *
 * Storage (the layout the GPU path uses too):
 *   A   m x k, row-major            A[i][kk]  = A[i*k + kk]
 *   Bt  n x k, row-major (B stored K-major, i.e. transposed)
 *                                   B[kk][j]  = Bt[j*k + kk]
 *   C   m x n, row-major            C[i][j]   = C[i*n + j]
 *
 * int8 x int8 -> int32: every product and partial sum is formed in int64, so
 * the sum is exact; the result is stored as int32 only after checking that it
 * fits (status ORACLE_ERR_OVERFLOW otherwise; nothing wraps).
 *
 * bf16 x bf16 -> fp32: every bf16 value is widened exactly to double, the
 * products and the sum are formed in double in increasing kk order, and the
 * sum is rounded once to the nearest float.  S[i][j] = sum |a*b| (double) is
 * returned beside it to scale the tolerance |err| <= 1e-3 * S.
 *
 * Rows of C are split over POSIX threads; each thread owns whole rows, so the
 * arithmetic of every element is the same as in a single-threaded run.
 *
 * Requantisation of the exact int32 product (oracle_requant): the usual
 * consumer of an int8 GEMM scales C per row and per column and stores a
 * narrower type.  The pages do not define it; the library states it as
 *
 *   D[i][j] = q( (float)((float)C[i][j] * row_scale[i]) * col_scale[j] )
 *
 * every step one IEEE-754 binary32 operation rounded to nearest, ties to
 * even: (1) int32 -> float, (2) times the row scale, (3) times the column
 * scale, (4) q = bfloat16 (round to nearest even; NaN stays NaN; overflow
 * gives infinity) or int8 (round to the nearest integer, ties to even, then
 * clamp to [-128, 127]; NaN gives 0).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>
#include <math.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_OVERFLOW 2
#define ORACLE_ERR_THREAD 3

/* ---- bf16 -> double, exactly: a bf16 is the top 16 bits of an IEEE float. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- one element of the int8 product, exact in int64 ------------------- */
static int64_t dot_i8(const int8_t *a_row, const int8_t *bt_row, int64_t k)
{
    int64_t sum = 0;
    for (int64_t kk = 0; kk < k; ++kk)
        sum += (int64_t)a_row[kk] * (int64_t)bt_row[kk];
    return sum;
}

/* ---- one element of the bf16 product in double ------------------------ */
static void dot_bf16(const uint16_t *a_row, const uint16_t *bt_row, int64_t k,
                     double *sum_out, double *abs_out)
{
    double sum = 0.0, abs_sum = 0.0;
    for (int64_t kk = 0; kk < k; ++kk) {
        double p = bf16_to_double(a_row[kk]) * bf16_to_double(bt_row[kk]);
        sum += p;
        abs_sum += (p < 0.0) ? -p : p;
    }
    *sum_out = sum;
    *abs_out = abs_sum;
}

/* ---- row-parallel driver ------------------------------------------------ */
typedef struct {
    int dtype; /* 0 = int8, 1 = bf16 */
    int64_t row_begin, row_end, k, n;
    const void *A, *Bt;
    void *C;
    double *S;
    int status;
} job_t;

static void *run_rows(void *arg)
{
    job_t *job = (job_t *)arg;
    const int64_t k = job->k, n = job->n;
    job->status = ORACLE_OK;
    for (int64_t i = job->row_begin; i < job->row_end; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            if (job->dtype == 0) {
                const int8_t *a = (const int8_t *)job->A + i * k;
                const int8_t *b = (const int8_t *)job->Bt + j * k;
                int64_t s = dot_i8(a, b, k);
                if (s > INT32_MAX || s < INT32_MIN) {
                    job->status = ORACLE_ERR_OVERFLOW;
                    return NULL;
                }
                ((int32_t *)job->C)[i * n + j] = (int32_t)s;
            } else {
                const uint16_t *a = (const uint16_t *)job->A + i * k;
                const uint16_t *b = (const uint16_t *)job->Bt + j * k;
                double s, sa;
                dot_bf16(a, b, k, &s, &sa);
                ((float *)job->C)[i * n + j] = (float)s;
                if (job->S)
                    job->S[i * n + j] = sa;
            }
        }
    }
    return NULL;
}

static int run_parallel(int dtype, int64_t m, int64_t k, int64_t n,
                        const void *A, const void *Bt, void *C, double *S,
                        int nthreads)
{
    if (m < 0 || k < 0 || n < 0)
        return ORACLE_ERR_ARG;
    if (m == 0 || n == 0)
        return ORACLE_OK;
    if (!C || (k > 0 && (!A || !Bt)))
        return ORACLE_ERR_ARG;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > m)
        nthreads = (int)m;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ERR_THREAD;
    }
    int status = ORACLE_OK, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].dtype = dtype;
        jobs[t].row_begin = m * t / nthreads;
        jobs[t].row_end = m * (t + 1) / nthreads;
        jobs[t].k = k;
        jobs[t].n = n;
        jobs[t].A = A;
        jobs[t].Bt = Bt;
        jobs[t].C = C;
        jobs[t].S = S;
        if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) {
            status = ORACLE_ERR_THREAD;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        pthread_join(tids[t], NULL);
        if (jobs[t].status != ORACLE_OK && status == ORACLE_OK)
            status = jobs[t].status;
    }
    free(jobs);
    free(tids);
    return status;
}

/* ---- exported entry points ------------------------------------------------ */

/* Full int8 product: C (m x n int32).  Returns ORACLE_ERR_OVERFLOW if any
 * exact sum falls outside int32. */
int oracle_gemm_i8(int64_t m, int64_t k, int64_t n, const int8_t *A,
                   const int8_t *Bt, int32_t *C, int nthreads)
{
    return run_parallel(0, m, k, n, A, Bt, C, NULL, nthreads);
}

/* Full bf16 product: C (m x n float) and, if S is not NULL, S (m x n double)
 * = sum |a*b|. */
int oracle_gemm_bf16(int64_t m, int64_t k, int64_t n, const uint16_t *A,
                     const uint16_t *Bt, float *C, double *S, int nthreads)
{
    return run_parallel(1, m, k, n, A, Bt, C, S, nthreads);
}

/* Selected int8 entries: out[t] = exact int64 C[rows[t]][cols[t]]. */
int oracle_gemm_i8_entries(int64_t m, int64_t k, int64_t n, const int8_t *A,
                           const int8_t *Bt, int64_t count, const int64_t *rows,
                           const int64_t *cols, int64_t *out)
{
    if (m < 0 || k < 0 || n < 0 || count < 0 || (count > 0 && (!rows || !cols || !out)))
        return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < count; ++t) {
        if (rows[t] < 0 || rows[t] >= m || cols[t] < 0 || cols[t] >= n)
            return ORACLE_ERR_ARG;
        out[t] = dot_i8(A + rows[t] * k, Bt + cols[t] * k, k);
    }
    return ORACLE_OK;
}

/* Selected bf16 entries: sum_out[t] = double sum, abs_out[t] = sum |a*b|. */
int oracle_gemm_bf16_entries(int64_t m, int64_t k, int64_t n, const uint16_t *A,
                             const uint16_t *Bt, int64_t count, const int64_t *rows,
                             const int64_t *cols, double *sum_out, double *abs_out)
{
    if (m < 0 || k < 0 || n < 0 || count < 0 ||
        (count > 0 && (!rows || !cols || !sum_out || !abs_out)))
        return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < count; ++t) {
        if (rows[t] < 0 || rows[t] >= m || cols[t] < 0 || cols[t] >= n)
            return ORACLE_ERR_ARG;
        dot_bf16(A + rows[t] * k, Bt + cols[t] * k, k, &sum_out[t], &abs_out[t]);
    }
    return ORACLE_OK;
}

/* ---- requantisation ------------------------------------------------------ */

/* Step 4 for bfloat16: the upper half of the float's bits, rounded to nearest
 * with ties to even by adding 0x7fff plus the lowest kept bit; NaN -> 0x7fc0. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return 0x7fc0;
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Step 4 for int8: nearest integer, ties to even, then saturation. */
static int8_t float_to_i8_rne_sat(float z)
{
    if (z != z)
        return 0;
    float r;
    if (fabsf(z) >= 8388608.0f) {          /* 2^23: already an integer (or infinite) */
        r = z;
    } else {
        const float fl = floorf(z);
        const float d = z - fl;            /* exact: z and fl are within 2^23 */
        if (d > 0.5f)
            r = fl + 1.0f;
        else if (d < 0.5f)
            r = fl;
        else
            r = (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
    }
    if (r > 127.0f)
        return 127;
    if (r < -128.0f)
        return -128;
    return (int8_t)r;
}

/* D (m x n) from C (m x n int32), row_scale (m), col_scale (n).  out_type 1:
 * D is bfloat16 (uint16 bit patterns); out_type 2: D is int8. */
int oracle_requant(int64_t m, int64_t n, const int32_t *C, const float *row_scale,
                   const float *col_scale, int out_type, void *D)
{
    if (m < 0 || n < 0 || (out_type != 1 && out_type != 2))
        return ORACLE_ERR_ARG;
    if (m == 0 || n == 0)
        return ORACLE_OK;
    if (!C || !row_scale || !col_scale || !D)
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            const float x = (float)C[i * n + j];          /* (1) */
            const float y = x * row_scale[i];            /* (2) */
            const float z = y * col_scale[j];            /* (3) */
            if (out_type == 1)
                ((uint16_t *)D)[i * n + j] = float_to_bf16_rne(z);   /* (4) */
            else
                ((int8_t *)D)[i * n + j] = float_to_i8_rne_sat(z);
        }
    }
    return ORACLE_OK;
}
