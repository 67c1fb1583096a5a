/*
 * fp64 oracle for dense row-major single-precision matrix multiplication.
 *
 * TEST INFRASTRUCTURE. This file is the independent checker of the CUDA
 * library: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it. It shares no code, header, table or helper with the library.
 *
 * What it computes (the plain definition, written out):
 *
 *     C64[i][j] = sum_{k = 0 .. K-1} (double)A[i][k] * (double)B[k][j]
 *     S[i][j]   = sum_{k = 0 .. K-1} |A[i][k]| * |B[k][j]|
 *
 * A is M x K, B is K x N and C is M x N, all row-major with leading
 * dimensions lda, ldb, ldc (in elements). This is the product that
 * "Optimizing a WebGPU Matmul Kernel using Subgroups", section 1 "Naive",
 * defines one output cell at a time (the dot product of row i of A with
 * column j of B, k running from 0 upward), and the CPU triple loop of
 * "WebGPU 行列積の限界を測る" (the matmulCPU routine under its three
 * implementations). The problem statement C = A x B with A M x K and B K x N
 * is the one of "WebGPU WGSL Compute Shaders: Custom Matrix Multiplication
 * (GEMM) Optimization Guide", section 1.
 *
 * S = |A|.|B| is the scale the per-element error bounds are stated against.
 *
 * Precision: every product of two fp32 values is exact in fp64 (24 + 24 <= 53
 * significand bits), so the only rounding is the fp64 accumulation, whose
 * error is at most about K * 2^-53 * S -- negligible next to any fp32 bound.
 * Each output accumulates its K products in increasing k, exactly as the
 * definition is written. The loops over i and j only choose which output is
 * being accumulated; no blocking, reassociation or fusion is applied, and the
 * build disables floating-point contraction.
 *
 * Parallelism: rows of C are independent, so rows are split across OpenMP
 * threads when the file is built with -fopenmp; this does not change any
 * arithmetic.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* One row of C64 and S: i-k-j order, so B is streamed row by row. The sum for
 * each C64[i][j] still runs over k = 0, 1, ..., K-1 in that order. */
static void oracle_row(int64_t i, int64_t N, int64_t K,
                       const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       double *c_row, double *s_row)
{
    for (int64_t j = 0; j < N; ++j) {
        c_row[j] = 0.0;
        if (s_row) s_row[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
        const double a = (double)A[i * lda + k];
        const double abs_a = fabs(a);
        const float *b_row = B + k * ldb;
        for (int64_t j = 0; j < N; ++j) {
            const double b = (double)b_row[j];
            c_row[j] += a * b;
            if (s_row) s_row[j] += abs_a * fabs(b);
        }
    }
}

/* Full product: C64 (ldc64) and, if S is non-null, S (lds). */
void oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     double *C64, int64_t ldc64,
                     double *S, int64_t lds)
{
    int64_t i;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (i = 0; i < M; ++i)
        oracle_row(i, N, K, A, lda, B, ldb, C64 + i * ldc64, S ? S + i * lds : NULL);
}

/* Selected rows: output row r (packed, N wide) is row rows[r] of the product. */
void oracle_gemm_rows_f64(int64_t nrows, const int64_t *rows,
                          int64_t N, int64_t K,
                          const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          double *C64, double *S)
{
    int64_t r;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (r = 0; r < nrows; ++r)
        oracle_row(rows[r], N, K, A, lda, B, ldb, C64 + r * N, S ? S + r * N : NULL);
}

/* Selected entries (ii[t], jj[t]): one dot product each, k increasing. */
void oracle_gemm_entries_f64(int64_t n, const int64_t *ii, const int64_t *jj,
                             int64_t K,
                             const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             double *c64, double *s)
{
    int64_t t;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (t = 0; t < n; ++t) {
        const int64_t i = ii[t], j = jj[t];
        double acc = 0.0, scale = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const double b = (double)B[k * ldb + j];
            acc += a * b;
            scale += fabs(a) * fabs(b);
        }
        c64[t] = acc;
        if (s) s[t] = scale;
    }
}

/* General form: Cout[i][j] = alpha * sum_k op(A)[i][k] * op(B)[k][j] + beta * Cin[i][j]
 * (beta == 0: Cin is not read), all in fp64, row-major storage, with
 *   op(A)[i][k] = A[i * lda + k] (opa == 0) or A[k * lda + i] (opa == 1: the
 *                 caller stores A transposed, K x M),
 *   op(B)[k][j] = B[k * ldb + j] (opb == 0) or B[j * ldb + k] (opb == 1: B
 *                 stored transposed, N x K).
 * The scale S[i][j] = sum_k |op(A)[i][k]| * |op(B)[k][j]|. This is the
 * product of oracle_gemm_f64 with the transposed-B storage of "Optimizing a
 * WebGPU Matmul Kernel using Subgroups", section 7 "Vectorized Buffers", the
 * transposed (column-major) storage that "WebGPU 计算着色器矩阵乘法优化：从
 * Naive 到 Tiled 深度实战" mentions under "工程实践建议", and the usual
 * scale-and-add of an existing C. Rows of the output are selected by rows[]
 * (nrows of them; output row r is row rows[r]). */
void oracle_gemm_general_rows_f64(int opa, int opb, int64_t nrows, const int64_t *rows,
                                  int64_t N, int64_t K, double alpha,
                                  const float *A, int64_t lda,
                                  const float *B, int64_t ldb,
                                  double beta, const float *Cin, int64_t ldc,
                                  double *Cout, double *S)
{
    int64_t r;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (r = 0; r < nrows; ++r) {
        const int64_t i = rows[r];
        double *c_row = Cout + r * N;
        double *s_row = S ? S + r * N : NULL;
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, scale = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = (double)(opa ? A[k * lda + i] : A[i * lda + k]);
                const double b = (double)(opb ? B[j * ldb + k] : B[k * ldb + j]);
                acc += a * b;
                scale += fabs(a) * fabs(b);
            }
            c_row[j] = alpha * acc + (beta != 0.0 ? beta * (double)Cin[i * ldc + j] : 0.0);
            if (s_row) s_row[j] = scale;
        }
    }
}

/* Threads the parallel loops above will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
