/*
 * CPU oracle for C = A * B over row-major fp32 matrices. Test
 * infrastructure only: the product library never includes this header.
 * All routines return 0 on success and nonzero on a bad argument.
 */
#ifndef SGEMM_ORACLE_H
#define SGEMM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CPU loop of the source pages: float accumulator, k ascending. */
int oracle_sgemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                     const float *B, int64_t ldb, float *C, int64_t ldc);

/* Same loop in double; S (may be NULL) receives sum_k |A[i][k]|*|B[k][j]|. */
int oracle_sgemm_f64(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                     const float *B, int64_t ldb, double *C64, double *S, int64_t ldc);

/* Rows [row_begin, row_end) of the double product, i-k-j order, threaded by rows.
 * Output row r of C64 / S is product row row_begin + r. Bit-identical to
 * oracle_sgemm_f64 on those rows. */
int oracle_sgemm_f64_rows(int64_t row_begin, int64_t row_end, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          double *C64, double *S, int64_t ldc, int nthreads);

/* Rows [row_begin, row_end) of the float product (the pages' loop arithmetic)
 * in i-k-j order, threaded by rows: bit-identical to oracle_sgemm_f32 on
 * those rows. Output row r of C is product row row_begin + r. */
int oracle_sgemm_f32_rows(int64_t row_begin, int64_t row_end, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          float *C, int64_t ldc, int nthreads);

/* Double product and S at n_samples (rows[t], cols[t]) positions. */
int oracle_sgemm_f64_at(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                        const float *B, int64_t ldb, int64_t n_samples, const int64_t *rows,
                        const int64_t *cols, double *c64, double *s);

/* C64 = alpha * op(A) * op(B) + beta * C_in in double (op = matrix or its
 * transpose; trans = 0 or 1; A is M x K, or K x M when transA; B is K x N, or
 * N x K when transB; all row-major). S = |alpha| sum_k |op(A)||op(B)| +
 * |beta| |C_in|. beta == 0: C_in is not read. */
int oracle_gemm_f64(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                    const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                    const float *C_in, int64_t ldc_in, double *C64, double *S, int64_t ldc);

/* The same at n_samples (rows[t], cols[t]) positions. */
int oracle_gemm_f64_at(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                       const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                       const float *C_in, int64_t ldc_in, int64_t n_samples, const int64_t *rows,
                       const int64_t *cols, double *c64, double *s);

/* Fused epilogue on n values of a double product at (rows[t], cols[t]) of
 * an M x N result, in place: x = c64[t] + b with b = bias[cols[t]]
 * (bias_kind 1), bias[rows[t]] (2) or 0 (0); c64[t] = act(x) with act
 * 0 none, 1 ReLU, 2 GELU (x Phi(x)), 3 SiLU (x / (1 + exp(-x))); s[t] += |b|
 * (s may be NULL). */
int oracle_epilogue_f64(int64_t n, const int64_t *rows, const int64_t *cols, int64_t M, int64_t N,
                        const float *bias, int bias_kind, int act, double *c64, double *s);

#ifdef __cplusplus
}
#endif

#endif
