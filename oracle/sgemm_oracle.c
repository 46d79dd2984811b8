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
 *   oracle_sgemm_f32_rows  the pages' float arithmetic with i, k, j loop order
 *                        over a band of rows, split across threads by rows
 *                        (the timed CPU baseline): every element still adds
 *                        its rounded products in k-ascending order into one
 *                        float, so it equals oracle_sgemm_f32 bit for bit;
 *                        the inner loop runs along a row of B, which the
 *                        compiler may vectorise across j without changing
 *                        any element's order of operations.
 *   oracle_sgemm_f64_at  C64 and S at a list of (row, col) samples, for
 *                        checks at sizes where the full product is too slow.
 *   oracle_gemm_f64      the general form C = alpha * op(A) * op(B) + beta * C
 *   oracle_gemm_f64_at   (op = the matrix or its transpose), in double, with
 *                        the error scale S = |alpha| sum_k |op(A)||op(B)| +
 *                        |beta| |C_in|. The pages define only C = A * B; the
 *                        general form is the standard BLAS GEMM, taken with
 *                        its convention that beta = 0 means C_in is not read.
 *   oracle_epilogue_f64  the fused epilogue act(x + bias) applied to values
 *                        of the double product, in double, with |bias| added
 *                        to S. The pages compute the product alone and call
 *                        it the core operation of neural-network layers
 *                        ("CUDA内存优化入门：从Naive到Tiled矩阵乘法",
 *                        section 一); a layer adds a bias and applies an
 *                        activation to it. Each activation is its textbook
 *                        definition on top of libm: ReLU(x) = max(x, 0) with
 *                        NaN kept, GELU(x) = x Phi(x) with the standard
 *                        normal CDF Phi(x) = (1 + erf(x / sqrt 2)) / 2,
 *                        SiLU(x) = x sigma(x) = x / (1 + exp(-x)).
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

struct f32_rows_job {
    int64_t band0, row_begin, row_end, N, K, lda, ldb, ldc;
    const float *A, *B;
    float *C;
};

static void *f32_rows_worker(void *arg)
{
    const struct f32_rows_job *job = (const struct f32_rows_job *)arg;
    for (int64_t i = job->row_begin; i < job->row_end; ++i) {
        float *c = job->C + (i - job->band0) * job->ldc;
        for (int64_t j = 0; j < job->N; ++j) c[j] = 0.0f;
        for (int64_t k = 0; k < job->K; ++k) {
            const float a = job->A[i * job->lda + k];
            const float *brow = job->B + k * job->ldb;
            for (int64_t j = 0; j < job->N; ++j) {
                float prod = a * brow[j];
                c[j] = c[j] + prod;
            }
        }
    }
    return NULL;
}

int oracle_sgemm_f32_rows(int64_t row_begin, int64_t row_end, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          float *C, int64_t ldc, int nthreads)
{
    if (row_begin < 0 || row_end < row_begin) return 1;
    if (!oracle_args_ok(row_end, N, K, A, lda, B, ldb, C, ldc)) return 1;
    int64_t rows = row_end - row_begin;
    if (rows == 0 || N == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = (int)rows;
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *created = (char *)calloc((size_t)nthreads, 1);
    struct f32_rows_job *jobs = (struct f32_rows_job *)calloc((size_t)nthreads, sizeof(struct f32_rows_job));
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
        jobs[t].C = C;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, f32_rows_worker, &jobs[t]) == 0)
            created[t] = 1;
        else
            f32_rows_worker(&jobs[t]);
    }
    f32_rows_worker(&jobs[0]);
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

/* Element (r, c) of op(X) for a row-major X with row stride ld. */
static double op_at(const float *X, int64_t ld, int trans, int64_t r, int64_t c)
{
    return trans ? (double)X[c * ld + r] : (double)X[r * ld + c];
}

static int gemm_args_ok(int transA, int transB, int64_t M, int64_t N, int64_t K, const void *A,
                        int64_t lda, const void *B, int64_t ldb)
{
    if (M < 0 || N < 0 || K < 0) return 0;
    if ((transA && lda < M) || (!transA && lda < K)) return 0;
    if ((transB && ldb < K) || (!transB && ldb < N)) return 0;
    if (M > 0 && K > 0 && A == NULL) return 0;
    if (K > 0 && N > 0 && B == NULL) return 0;
    return 1;
}

/* One element of alpha * op(A) * op(B) + beta * C_in and its error scale. */
static void gemm_element(int transA, int transB, int64_t K, double alpha, const float *A,
                         int64_t lda, const float *B, int64_t ldb, double beta, double c_in,
                         int64_t i, int64_t j, double *c, double *s)
{
    double sum = 0.0, abs_sum = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double a = op_at(A, lda, transA, i, k);
        double b = op_at(B, ldb, transB, k, j);
        sum = sum + a * b;
        abs_sum = abs_sum + fabs(a) * fabs(b);
    }
    double out = alpha * sum, scale = fabs(alpha) * abs_sum;
    if (beta != 0.0) {
        out = out + beta * c_in;
        scale = scale + fabs(beta) * fabs(c_in);
    }
    *c = out;
    if (s) *s = scale;
}

int oracle_gemm_f64(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                    const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                    const float *C_in, int64_t ldc_in, double *C64, double *S, int64_t ldc)
{
    if (!gemm_args_ok(transA, transB, M, N, K, A, lda, B, ldb)) return 1;
    if (ldc < N || (M > 0 && N > 0 && C64 == NULL)) return 1;
    if (beta != 0.0 && M > 0 && N > 0 && (C_in == NULL || ldc_in < N)) return 1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double c_in = beta != 0.0 ? (double)C_in[i * ldc_in + j] : 0.0;
            gemm_element(transA, transB, K, alpha, A, lda, B, ldb, beta, c_in, i, j,
                         &C64[i * ldc + j], S ? &S[i * ldc + j] : NULL);
        }
    return 0;
}

int oracle_gemm_f64_at(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                       const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                       const float *C_in, int64_t ldc_in, int64_t n_samples, const int64_t *rows,
                       const int64_t *cols, double *c64, double *s)
{
    if (!gemm_args_ok(transA, transB, M, N, K, A, lda, B, ldb) || n_samples < 0) return 1;
    if (n_samples > 0 && (!rows || !cols || !c64)) return 1;
    if (beta != 0.0 && n_samples > 0 && (C_in == NULL || ldc_in < N)) return 1;
    for (int64_t t = 0; t < n_samples; ++t) {
        int64_t i = rows[t], j = cols[t];
        if (i < 0 || i >= M || j < 0 || j >= N) return 1;
        double c_in = beta != 0.0 ? (double)C_in[i * ldc_in + j] : 0.0;
        gemm_element(transA, transB, K, alpha, A, lda, B, ldb, beta, c_in, i, j, &c64[t],
                     s ? &s[t] : NULL);
    }
    return 0;
}

/* Activation codes of oracle_epilogue_f64 (this oracle's own numbering). */
enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_GELU = 2, ORACLE_ACT_SILU = 3 };
enum { ORACLE_BIAS_NONE = 0, ORACLE_BIAS_COL = 1, ORACLE_BIAS_ROW = 2 };

static double oracle_activate(int act, double x)
{
    switch (act) {
    case ORACLE_ACT_RELU:
        return x < 0.0 ? 0.0 : x;
    case ORACLE_ACT_GELU: {
        double phi = 0.5 * (1.0 + erf(x / sqrt(2.0))); /* standard normal CDF */
        return x * phi;
    }
    case ORACLE_ACT_SILU: {
        double sigma = 1.0 / (1.0 + exp(-x)); /* logistic function */
        return x * sigma;
    }
    default:
        return x;
    }
}

int oracle_epilogue_f64(int64_t n, const int64_t *rows, const int64_t *cols, int64_t M, int64_t N,
                        const float *bias, int bias_kind, int act, double *c64, double *s)
{
    if (n < 0 || M < 0 || N < 0) return 1;
    if (bias_kind < ORACLE_BIAS_NONE || bias_kind > ORACLE_BIAS_ROW) return 1;
    if (act < ORACLE_ACT_NONE || act > ORACLE_ACT_SILU) return 1;
    if (n > 0 && (!rows || !cols || !c64)) return 1;
    if (n > 0 && bias_kind != ORACLE_BIAS_NONE && !bias) return 1;
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = rows[t], j = cols[t];
        if (i < 0 || i >= M || j < 0 || j >= N) return 1;
        double b = 0.0;
        if (bias_kind == ORACLE_BIAS_COL) b = (double)bias[j];
        if (bias_kind == ORACLE_BIAS_ROW) b = (double)bias[i];
        c64[t] = oracle_activate(act, c64[t] + b);
        if (s) s[t] += fabs(b);
    }
    return 0;
}
