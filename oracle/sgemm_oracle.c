/*
 * CPU oracle for dense single-precision row-major matrix multiplication.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or
 * calls this file: only the test suite, the smoke check and the bench's
 * cpu-baseline leg do. It shares no code, header or constant with the CUDA
 * library, and it is compiled for the host alone (gcc, -O2,
 * -ffp-contract=off, no fast-math), so every float product and every float
 * sum below is rounded separately, exactly as the C source reads.
 *
 * What it computes is the plain definition of the product that all four
 * source pages state in the same form:
 *
 *     C[i][j] = sum over k = 0 .. K-1 of A[i][k] * B[k][j]
 *
 *   - "CUDA内存优化入门：从Naive到Tiled矩阵乘法" (From Naive to Tiled matrix
 *     multiplication), section 三 "矩阵乘法的计算原理", formula block, and
 *     section 四 "版本1：CPU基准实现" (the CPU baseline: one float
 *     accumulator per output, k ascending, row-major A = M x K, B = K x N);
 *   - "CUDA算子优化(4)：矩阵乘法", section "矩阵乘法的数学定义" (the same
 *     sum) and "版本V0矩阵乘法cpu实现" (the same loop nest);
 *   - "【infra之路】Tiled Matrix Multiplication详解", opening section (the
 *     element as a dot product along K).
 *
 * The pages index contiguous matrices (row length = K for A, N for B and C).
 * Here every matrix also takes a row stride (lda, ldb, ldc >= row length);
 * element (r, c) of a matrix with stride ld sits at offset r * ld + c.
 *
 * Routines
 *   oracle_sgemm_f32     the pages' CPU loop: i, j, then k ascending, one
 *                        float accumulator, product and sum rounded apart.
 *   oracle_sgemm_f64     the same loop in double: C64 and the absolute-value
 *                        sum S[i][j] = sum_k |A[i][k]| * |B[k][j]|. A product
 *                        of two floats is exact in double, so only the sums
 *                        round, and an FMA or not makes no difference.
 *   oracle_sgemm_f64_rows  the same double arithmetic with i, k, j loop order
 *                        over a band of rows [row_begin, row_end), split
 *                        across threads by rows; output row 0 is row_begin.
 *                        Each element still adds its terms in k-ascending
 *                        order, so it equals oracle_sgemm_f64 bit for bit.
 *   oracle_sgemm_f64_at  C64 and S at a list of (row, col) samples, for
 *                        checks at sizes where the full product is too slow.
 *
 * Pins (tests/test_oracle_pins.py, CPU only): all-ones inputs give C = K
 * exactly (the all-ones check of "CUDA 性能优化实战笔记 + C++示例代码（第七章
 * 重点）" section 二, where every output of the 1024 x 1024 product must be
 * 1024); identity and permutation products; a polynomial closed form that
 * changes under any transposition; the block identity C00 = A00 B00 + A01 B10
 * of the 8 x 8 / 4 x 4 example of the "Tiled Matrix Multiplication" page;
 * brute force in exact rational arithmetic on tiny shapes; float32 brute
 * force with numpy scalars in the same order (bit-identical); the empty sum
 * (K = 0) and a single nonzero term.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#include "sgemm_oracle.h"

static int oracle_args_ok(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                          const void *B, int64_t ldb, const void *C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return 0;
    if (lda < K || ldb < N || ldc < N) return 0;
    if (M > 0 && N > 0 && C == NULL) return 0;
    if (M > 0 && K > 0 && A == NULL) return 0;
    if (K > 0 && N > 0 && B == NULL) return 0;
    return 1;
}

int oracle_sgemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                     const float *B, int64_t ldb, float *C, int64_t ldc)
{
    if (!oracle_args_ok(M, N, K, A, lda, B, ldb, C, ldc)) return 1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            float sum = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float prod = A[i * lda + k] * B[k * ldb + j];
                sum = sum + prod;
            }
            C[i * ldc + j] = sum;
        }
    }
    return 0;
}

int oracle_sgemm_f64(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                     const float *B, int64_t ldb, double *C64, double *S, int64_t ldc)
{
    if (!oracle_args_ok(M, N, K, A, lda, B, ldb, C64, ldc)) return 1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = (double)A[i * lda + k];
                double b = (double)B[k * ldb + j];
                sum = sum + a * b;
                abs_sum = abs_sum + fabs(a) * fabs(b);
            }
            C64[i * ldc + j] = sum;
            if (S) S[i * ldc + j] = abs_sum;
        }
    }
    return 0;
}

struct rows_job {
    int64_t band0, row_begin, row_end, N, K, lda, ldb, ldc;
    const float *A, *B;
    double *C64, *S;
};

static void *rows_worker(void *arg)
{
    const struct rows_job *job = (const struct rows_job *)arg;
    for (int64_t i = job->row_begin; i < job->row_end; ++i) {
        double *c = job->C64 + (i - job->band0) * job->ldc;
        double *s = job->S ? job->S + (i - job->band0) * job->ldc : NULL;
        for (int64_t j = 0; j < job->N; ++j) {
            c[j] = 0.0;
            if (s) s[j] = 0.0;
        }
        for (int64_t k = 0; k < job->K; ++k) {
            double a = (double)job->A[i * job->lda + k];
            const float *brow = job->B + k * job->ldb;
            for (int64_t j = 0; j < job->N; ++j) {
                double b = (double)brow[j];
                c[j] = c[j] + a * b;
            }
            if (s) {
                double abs_a = fabs(a);
                for (int64_t j = 0; j < job->N; ++j)
                    s[j] = s[j] + abs_a * fabs((double)brow[j]);
            }
        }
    }
    return NULL;
}

int oracle_sgemm_f64_rows(int64_t row_begin, int64_t row_end, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          double *C64, double *S, int64_t ldc, int nthreads)
{
    if (row_begin < 0 || row_end < row_begin) return 1;
    if (!oracle_args_ok(row_end, N, K, A, lda, B, ldb, C64, ldc)) return 1;
    int64_t rows = row_end - row_begin;
    if (rows == 0 || N == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = (int)rows;
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *created = (char *)calloc((size_t)nthreads, 1);
    struct rows_job *jobs = (struct rows_job *)calloc((size_t)nthreads, sizeof(struct rows_job));
    if (!tid || !created || !jobs) {
        free(tid);
        free(created);
        free(jobs);
        return 2;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].band0 = row_begin;
        jobs[t].row_begin = row_begin + rows * t / nthreads;
        jobs[t].row_end = row_begin + rows * (t + 1) / nthreads;
        jobs[t].N = N;
        jobs[t].K = K;
        jobs[t].lda = lda;
        jobs[t].ldb = ldb;
        jobs[t].ldc = ldc;
        jobs[t].A = A;
        jobs[t].B = B;
        jobs[t].C64 = C64;
        jobs[t].S = S;
    }
    /* Bands 1.. go to new threads (run inline if a thread cannot start);
     * the calling thread takes band 0. */
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, rows_worker, &jobs[t]) == 0)
            created[t] = 1;
        else
            rows_worker(&jobs[t]);
    }
    rows_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (created[t]) pthread_join(tid[t], NULL);
    free(tid);
    free(created);
    free(jobs);
    return 0;
}

int oracle_sgemm_f64_at(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                        const float *B, int64_t ldb, int64_t n_samples, const int64_t *rows,
                        const int64_t *cols, double *c64, double *s)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || n_samples < 0) return 1;
    if (n_samples > 0 && (!rows || !cols || !c64 || (K > 0 && (!A || !B)))) return 1;
    for (int64_t t = 0; t < n_samples; ++t) {
        int64_t i = rows[t], j = cols[t];
        if (i < 0 || i >= M || j < 0 || j >= N) return 1;
        double sum = 0.0, abs_sum = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = (double)A[i * lda + k];
            double b = (double)B[k * ldb + j];
            sum = sum + a * b;
            abs_sum = abs_sum + fabs(a) * fabs(b);
        }
        c64[t] = sum;
        if (s) s[t] = abs_sum;
    }
    return 0;
}
