/*
 * CPU oracle for dense matrix multiplication C = A x B.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition of the product, as stated in
 * "Tiled Matrix Multiplication in CUDA", section 1 ("What matrix
 * multiplication actually does") and "Tiled GEMM: Matrix Multiplication in
 * CUDA", section 1: every output cell is the dot product of a row of A with a
 * column of B,
 *
 *     C[i][j] = sum over k = 0 .. K-1 of A[i][k] * B[k][j],
 *
 * with every matrix stored row-major and addressed by the flat index
 * row * leading_dimension + col ("Tiled Matrix Multiplication in CUDA",
 * section 2, "flat indexing"). The square "width" of the pages is generalised
 * to M x K times K x N with a leading dimension per matrix, as in the ragged-
 * edge code of "Tiled GEMM: Matrix Multiplication in CUDA", section 7.1.
 *
 * Arithmetic: the inputs arrive as IEEE doubles (the caller converts fp32 or
 * bf16 values, which is exact). Each product of two fp32/bf16 values is exact
 * in double (at most 48 significand bits), and the sum for each output cell
 * is accumulated in double in ascending k. The loops run i, then k, then j,
 * with C's row as the accumulator: for every single cell the products are
 * still added one at a time in ascending k, so each cell's sum is exactly the
 * one the i-j-k loop nest gives; only the order in which different cells are
 * visited changes. Build with -ffp-contract=off so that no multiply-add is
 * fused (with exact products it would not change the result, but the file
 * should mean the same thing for any double input).
 *
 * Alongside C it returns absAB[i][j] = sum_k |A[i][k]| * |B[k][j]|, the scale
 * that the parity tolerances are stated in.
 *
 * Rows of C are independent (section 1 of the first page: "every cell of C is
 * independent"), so the outer loop over rows is spread over OpenMP threads;
 * this changes no arithmetic.
 */
#include <math.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One row of the product: C[i][0..N-1] and absAB[i][0..N-1]. */
static void oracle_row(long i, int N, int K,
                       const double* A, long lda,
                       const double* B, long ldb,
                       double* c_row, double* abs_row)
{
    for (int j = 0; j < N; ++j) {
        c_row[j] = 0.0;
        abs_row[j] = 0.0;
    }
    for (int k = 0; k < K; ++k) {
        const double a = A[i * lda + k];
        const double abs_a = fabs(a);
        const double* b_row = B + (long)k * ldb;
        for (int j = 0; j < N; ++j) {
            c_row[j] += a * b_row[j];
            abs_row[j] += abs_a * fabs(b_row[j]);
        }
    }
}

/*
 * Selected rows of C = A x B.
 *   M, N, K      : A is M x K, B is K x N (K = 0 gives all-zero rows).
 *   A, lda       : row-major A, lda >= K doubles between row starts.
 *   B, ldb       : row-major B, ldb >= N.
 *   rows, n_rows : indices (0 <= rows[r] < M) of the rows of C wanted.
 *   C, ldc       : output, n_rows x N, row r holds row rows[r] of the product.
 *   absAB, ldabs : output, n_rows x N, sum_k |A[i][k]| |B[k][j]|.
 * Returns 0, or -1 if an argument is out of range (nothing is written then).
 */
int oracle_gemm_rows(int M, int N, int K,
                     const double* A, long lda,
                     const double* B, long ldb,
                     const long* rows, int n_rows,
                     double* C, long ldc,
                     double* absAB, long ldabs)
{
    if (M < 0 || N < 0 || K < 0 || n_rows < 0) return -1;
    if (lda < K || ldb < N || ldc < N || ldabs < N) return -1;
    for (int r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;

    #pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r)
        oracle_row(rows[r], N, K, A, lda, B, ldb,
                   C + (long)r * ldc, absAB + (long)r * ldabs);
    return 0;
}

/* All of C = A x B (rows 0 .. M-1), same arguments as above. */
int oracle_gemm(int M, int N, int K,
                const double* A, long lda,
                const double* B, long ldb,
                double* C, long ldc,
                double* absAB, long ldabs)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (lda < K || ldb < N || ldc < N || ldabs < N) return -1;

    #pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < M; ++i)
        oracle_row(i, N, K, A, lda, B, ldb,
                   C + i * ldc, absAB + i * ldabs);
    return 0;
}

/*
 * Extended form, for the library's gemm_ex (operands given transposed, and
 * the scaled-and-shifted output of the usual BLAS convention):
 *
 *     C[i][j] = alpha * sum_k opA[i][k] * opB[k][j] + beta * C0[i][j] + bias[j]
 *
 * opA[i][k] is A[i][k] (A stored M x K, lda >= K) or, with trans_a, A[k][i]
 * (A stored K x M, lda >= M; the column-major reading of an M x K matrix,
 * "Tiled Matrix Multiplication in CUDA", section 2). opB likewise: B[k][j]
 * (B stored K x N) or, with trans_b, B[j][k] (B stored N x K). The sum is
 * the definition above, accumulated in double in ascending k; the output
 * terms are then added in double. C0 is not read when beta == 0 (it may be
 * NULL); bias may be NULL (no shift).
 *
 * scale[i][j] = |alpha| * sum_k |opA[i][k]| |opB[k][j]| + |beta C0[i][j]| + |bias[j]|
 * is the magnitude the tolerances of this form are stated in.
 */
int oracle_gemm_ex(int M, int N, int K,
                   const double* A, long lda, int trans_a,
                   const double* B, long ldb, int trans_b,
                   double alpha, double beta,
                   const double* C0, long ldc0, const double* bias,
                   double* C, long ldc, double* scale, long ldscale)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? K : N)) return -1;
    if (ldc < N || ldscale < N) return -1;
    if (beta != 0.0 && (C0 == NULL || ldc0 < N)) return -1;

    #pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < M; ++i) {
        double* c_row = C + i * ldc;
        double* s_row = scale + i * ldscale;
        for (int j = 0; j < N; ++j) {
            c_row[j] = 0.0;
            s_row[j] = 0.0;
        }
        for (int k = 0; k < K; ++k) {
            const double a = trans_a ? A[(long)k * lda + i] : A[i * lda + k];
            for (int j = 0; j < N; ++j) {
                const double b = trans_b ? B[(long)j * ldb + k] : B[(long)k * ldb + j];
                c_row[j] += a * b;
                s_row[j] += fabs(a) * fabs(b);
            }
        }
        for (int j = 0; j < N; ++j) {
            double v = alpha * c_row[j];
            double m = fabs(alpha) * s_row[j];
            if (beta != 0.0) {
                v += beta * C0[i * ldc0 + j];
                m += fabs(beta * C0[i * ldc0 + j]);
            }
            if (bias != NULL) {
                v += bias[j];
                m += fabs(bias[j]);
            }
            c_row[j] = v;
            s_row[j] = m;
        }
    }
    return 0;
}

/* Thread control, so that callers can state how many cores a timing used. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
