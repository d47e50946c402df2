/*
 * CPU oracle for single-precision GEMM, C = A . B, row-major.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against. Only the tests, the
 * smoke check and the bench's CPU-baseline leg may load it. The CUDA library
 * never links, includes or calls it, and it shares no code with the library.
 *
 * What it computes (the definition, written out):
 *
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j],   0 <= i < M, 0 <= j < N
 *
 *   - "Перемножение матриц: наивное и тайловое", section 1: element
 *     C_row,col is the dot product of row `row` of A with column `col` of B;
 *     a matrix is stored row by row, element (row, col) at offset
 *     row * n + col. Here the row length is generalised to a leading
 *     dimension (lda, ldb, ldc >= the row length).
 *   - Chapter 9: Optimised Matrix Multiplication, section 9.1: N^3
 *     multiply-adds, 2N^3 FLOPs (2MNK for rectangular shapes).
 *
 * Precision. Every float is widened to double before use. A float*float
 * product has at most 48 significant bits, so it is exact in double; only the
 * K-term sum rounds, with error at most K * 2^-53 * S, where
 *
 *   S[i][j] = sum_k |A[i][k] * B[k][j]|
 *
 * is also returned (it sets the tolerance of the FP32 comparison).
 *
 * Loop order is i, k, j: row i of C is accumulated in a double row buffer,
 * adding A[i][k] * B[k][:] for k = 0, 1, ..., K-1 in order. This is still
 * the plain triple loop (no blocking, no reordering of the k sum). Rows are
 * independent and are split across OpenMP threads.
 *
 * Conventions the pages leave open (stated once here):
 *   - K == 0 gives C = 0 (the empty sum); M == 0 or N == 0 does nothing.
 *   - C is written, never read (the pages' listings all assign C = sum).
 *   - Matrix entries beyond the row length (between N and ld) are neither
 *     read nor written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of threads the oracle's parallel loops use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the OpenMP thread count for later calls (n <= 0 leaves it as is). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * One row of the product: crow[j] = sum_k A[i][k] * B[k][j] and
 * srow[j] = sum_k |A[i][k] * B[k][j]| for j in [0, N).
 */
static void oracle_row(int64_t N, int64_t K, const float *arow,
                       const float *B, int64_t ldb, double *crow, double *srow)
{
    for (int64_t j = 0; j < N; ++j) {
        crow[j] = 0.0;
        if (srow) srow[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
        const double a = (double)arow[k];
        const float *brow = B + k * ldb;
        for (int64_t j = 0; j < N; ++j) {
            const double p = a * (double)brow[j];
            crow[j] += p;
            if (srow) srow[j] += fabs(p);
        }
    }
}

/*
 * Full product. C (M x N, leading dimension ldc) receives the double result;
 * S (nullable, leading dimension lds) receives sum_k |A_ik B_kj|.
 * Returns 0, or -1 if an argument is invalid (nothing is written then).
 */
int oracle_sgemm_f64(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda, const float *B, int64_t ldb,
                     double *C, int64_t ldc, double *S, int64_t lds)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (lda < K || ldb < N || ldc < N || (S && lds < N)) return -1;
    if (!C || (K > 0 && (!A || !B))) return -1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        oracle_row(N, K, K > 0 ? A + i * lda : A, B, ldb, C + i * ldc,
                   S ? S + i * lds : NULL);
    }
    return 0;
}

/*
 * Selected rows of the product: for r in [0, nrows), row rows[r] of C goes to
 * Crows[r * N .. r * N + N) (and of S to Srows, nullable).
 */
int oracle_sgemm_rows_f64(int64_t M, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          const int64_t *rows, int64_t nrows,
                          double *Crows, double *Srows)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (lda < K || ldb < N) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        oracle_row(N, K, A + rows[r] * lda, B, ldb, Crows + r * N,
                   Srows ? Srows + r * N : NULL);
    }
    return 0;
}

/*
 * Selected columns of the product: for c in [0, ncols), column cols[c] of C
 * goes to Ccols[i * ncols + c] for i in [0, M) (an M x ncols matrix; S alike).
 * The selected columns of B are first copied into a K x ncols buffer so that
 * the same i, k, j loop (j over the selected columns) applies.
 */
int oracle_sgemm_cols_f64(int64_t M, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          const int64_t *cols, int64_t ncols,
                          double *Ccols, double *Scols)
{
    if (M < 0 || N < 0 || K < 0 || ncols < 0) return -1;
    if (lda < K || ldb < N) return -1;
    for (int64_t c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N) return -1;
    if (M == 0 || ncols == 0) return 0;

    float *Bsel = (float *)malloc((size_t)(K > 0 ? K : 1) * (size_t)ncols * sizeof(float));
    if (!Bsel) return -2;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t c = 0; c < ncols; ++c)
            Bsel[k * ncols + c] = B[k * ldb + cols[c]];

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        oracle_row(ncols, K, A + i * lda, Bsel, ncols, Ccols + i * ncols,
                   Scols ? Scols + i * ncols : NULL);
    }
    free(Bsel);
    return 0;
}

/*
 * General form (a library extension of the definition above; the pages have
 * no alpha, beta, transposes or batches):
 *
 *   C_b[i][j] = alpha * sum_k opA_b[i][k] * opB_b[k][j] + beta * C_b[i][j]
 *
 * for b in [0, batch), i < M, j < N, where opA_b[i][k] = A[b*sa + i*lda + k]
 * (op_a == 0, A stored M x K) or A[b*sa + k*lda + i] (op_a == 1, A stored
 * K x M), and opB_b[k][j] = B[b*sb + k*ldb + j] (op_b == 0) or
 * B[b*sb + j*ldb + k] (op_b == 1). C_in (float, leading dimension ldc, batch
 * stride sc) is read only when beta != 0. Results go to Cout (double, M x N
 * per batch entry, contiguous); S (nullable, same shape) receives
 * |alpha| * sum_k |opA opB| + |beta * C_in|, the scale of the tolerance.
 * Plain triple loop per entry in i, k, j order.
 */
int oracle_sgemm_general_f64(int op_a, int op_b, int64_t M, int64_t N, int64_t K, double alpha,
                             const float *A, int64_t lda, int64_t sa,
                             const float *B, int64_t ldb, int64_t sb,
                             double beta, const float *Cin, int64_t ldc, int64_t sc,
                             int64_t batch, double *Cout, double *S)
{
    if (M < 0 || N < 0 || K < 0 || batch < 0) return -1;
    if ((op_a != 0 && op_a != 1) || (op_b != 0 && op_b != 1)) return -1;
    if (batch == 0 || M == 0 || N == 0) return 0;
    if (beta != 0.0 && (!Cin || ldc < N)) return -1;
    if (K > 0 && (!A || !B)) return -1;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t i = 0; i < M; ++i) {
            double *crow = Cout + (b * M + i) * N;
            double *srow = S ? S + (b * M + i) * N : NULL;
            for (int64_t j = 0; j < N; ++j) {
                crow[j] = 0.0;
                if (srow) srow[j] = 0.0;
            }
            for (int64_t k = 0; k < K; ++k) {
                const double a = (double)(op_a == 0 ? A[b * sa + i * lda + k] : A[b * sa + k * lda + i]);
                for (int64_t j = 0; j < N; ++j) {
                    const double bv = (double)(op_b == 0 ? B[b * sb + k * ldb + j] : B[b * sb + j * ldb + k]);
                    const double p = a * bv;
                    crow[j] += p;
                    if (srow) srow[j] += fabs(p);
                }
            }
            for (int64_t j = 0; j < N; ++j) {
                const double c = beta != 0.0 ? (double)Cin[b * sc + i * ldc + j] : 0.0;
                crow[j] = alpha * crow[j] + beta * c;
                if (srow) srow[j] = fabs(alpha) * srow[j] + fabs(beta * c);
            }
        }
    }
    return 0;
}
