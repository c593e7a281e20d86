/*
 * CPU oracle for single-precision GEMM, C = alpha * op(A) * op(B) + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no source, header, table or helper with
 * the CUDA library, and it includes nothing from it.
 *
 * What it computes (the plain definition of GEMM):
 *   "Optimising fp32 GEMM on A100", section "What is GEMM?": C = alpha*(A x B)
 *   + beta*C with A M x K, B K x N, C M x N, and the three nested loops over
 *   i, j, k;  "CuTe-ly writing an SM86 SGEMM", section "epilogue":
 *   C_out = alpha*(AB) + beta*C_in.
 *
 * Storage convention (a reading: the pages use both row- and column-major;
 * the configurations this library is measured on are row-major):
 *   op(A)(i,k) = A[i*lda + k]  when transA is 'N' (A stored M x K),
 *              = A[k*lda + i]  when transA is 'T' (A stored K x M);
 *   op(B)(k,j) = B[k*ldb + j]  when transB is 'N' (B stored K x N),
 *              = B[j*ldb + k]  when transB is 'T' (B stored N x K);
 *   C(i,j)     = C[i*ldc + j].
 *
 * Two functions:
 *   oracle_gemm_f64      - the exact-as-possible reference.  Every fp32
 *                          input widens exactly to double, every product of
 *                          two fp32 numbers is exact in double, and the sum
 *                          runs in ascending k in double.  In the same pass
 *                          it forms the error bound
 *                            bound = 4*K*2^-24 * (|alpha|*sum_k |a||b|
 *                                                  + |beta|*|c|).
 *                          beta == 0 drops the C term entirely (C is not
 *                          read), so NaN in an unused C cannot leak in.
 *   oracle_gemm_f32_seq  - the same definition evaluated in fp32 in the
 *                          naive loop's order: acc = fmaf(a, b, acc) for
 *                          k = 0, 1, ..., K-1 from acc = 0, then
 *                          alpha*acc (beta == 0) or fmaf(alpha, acc, beta*c).
 *                          "How to get a matmul kernel into the top
 *                          percentile (worklog)", section "Optimization 1":
 *                          a k-tiled loop that keeps the naive ascending
 *                          order gives an identical fp32 result.  This is
 *                          the bitwise reference for the CUDA-core path.
 *
 * Both accept an optional list of (row, col) sample points; with no list
 * they fill the whole M x N output.  Built with -ffp-contract=off so that the
 * only fused operations are the explicit fmaf calls, and without fast-math.
 * Parallel over output entries with OpenMP when available; every entry is
 * computed by one thread in a fixed order, so results do not depend on the
 * thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* status codes, negative = -(1-based position of the bad argument) */
#define ORACLE_OK 0

static int is_n(char t) { return t == 'N' || t == 'n'; }
static int is_t(char t) { return t == 'T' || t == 't' || t == 'C' || t == 'c'; }

/* op(A)(i,k) for the storage convention in the header comment */
static float op_a(const float *A, int64_t lda, int ta_n, int64_t i, int64_t k)
{
    return ta_n ? A[i * lda + k] : A[k * lda + i];
}

/* op(B)(k,j) */
static float op_b(const float *B, int64_t ldb, int tb_n, int64_t k, int64_t j)
{
    return tb_n ? B[k * ldb + j] : B[j * ldb + k];
}

static int check_args(char ta, char tb, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc)
{
    if (!is_n(ta) && !is_t(ta)) return -1;
    if (!is_n(tb) && !is_t(tb)) return -2;
    if (M < 0) return -3;
    if (N < 0) return -4;
    if (K < 0) return -5;
    /* stored row length must fit in the leading dimension */
    int64_t a_row = is_n(ta) ? K : M;
    int64_t b_row = is_n(tb) ? N : K;
    if (lda < (a_row > 1 ? a_row : 1)) return -8;
    if (ldb < (b_row > 1 ? b_row : 1)) return -10;
    if (ldc < (N > 1 ? N : 1)) return -13;
    return ORACLE_OK;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (n >= 1); the results do not depend on it. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * ref[p], bound[p] for every output point p.  With rows == NULL the points
 * are all (i, j) in row-major order and ref/bound are M*N arrays; otherwise
 * point p is (rows[p], cols[p]) and npts points are written.
 */
int oracle_gemm_f64(char ta, char tb, int64_t M, int64_t N, int64_t K,
                    float alpha, const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    float beta, const float *C, int64_t ldc,
                    const int64_t *rows, const int64_t *cols, int64_t npts,
                    double *ref, double *bound)
{
    int st = check_args(ta, tb, M, N, K, lda, ldb, ldc);
    if (st != ORACLE_OK) return st;
    const int ta_n = is_n(ta), tb_n = is_n(tb);
    const int64_t total = rows ? npts : M * N;
    const double a64 = (double)alpha, b64 = (double)beta;
    const double unit = ldexp(1.0, -24);

    int64_t p;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (p = 0; p < total; ++p) {
        const int64_t i = rows ? rows[p] : p / N;
        const int64_t j = rows ? cols[p] : p % N;
        double sum = 0.0, mag = 0.0;
        /* alpha == 0 means op(A)*op(B) is not formed at all (BLAS rule),
           so A and B are not read */
        const int64_t kend = (alpha == 0.0f) ? 0 : K;
        for (int64_t k = 0; k < kend; ++k) {
            const double a = (double)op_a(A, lda, ta_n, i, k);
            const double b = (double)op_b(B, ldb, tb_n, k, j);
            sum += a * b;
            mag += fabs(a) * fabs(b);
        }
        double r = (alpha == 0.0f) ? 0.0 : a64 * sum;
        double m = fabs(a64) * mag;
        if (beta != 0.0f) {
            const double c = (double)C[i * ldc + j];
            r += b64 * c;
            m += fabs(b64) * fabs(c);
        }
        ref[p] = r;
        bound[p] = 4.0 * (double)K * unit * m;
    }
    return ORACLE_OK;
}

/*
 * out[p] = the fp32 evaluation in ascending-k FMA order for every point.
 * Same point convention as oracle_gemm_f64.
 */
int oracle_gemm_f32_seq(char ta, char tb, int64_t M, int64_t N, int64_t K,
                        float alpha, const float *A, int64_t lda,
                        const float *B, int64_t ldb,
                        float beta, const float *C, int64_t ldc,
                        const int64_t *rows, const int64_t *cols, int64_t npts,
                        float *out)
{
    int st = check_args(ta, tb, M, N, K, lda, ldb, ldc);
    if (st != ORACLE_OK) return st;
    const int ta_n = is_n(ta), tb_n = is_n(tb);
    const int64_t total = rows ? npts : M * N;

    int64_t p;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (p = 0; p < total; ++p) {
        const int64_t i = rows ? rows[p] : p / N;
        const int64_t j = rows ? cols[p] : p % N;
        float acc = 0.0f;
        float r;
        if (alpha == 0.0f) {
            /* no product term (BLAS rule): C = beta*C, or 0 when beta == 0 */
            r = (beta == 0.0f) ? 0.0f : beta * C[i * ldc + j];
        } else {
            for (int64_t k = 0; k < K; ++k)
                acc = fmaf(op_a(A, lda, ta_n, i, k), op_b(B, ldb, tb_n, k, j), acc);
            if (beta == 0.0f) {
                r = alpha * acc;
            } else {
                const float bc = beta * C[i * ldc + j];
                r = fmaf(alpha, acc, bc);
            }
        }
        out[p] = r;
    }
    return ORACLE_OK;
}

/*
 * GEMM with a fused epilogue (the pages' "prologue and epilogue" fusion,
 * "Optimising fp32 GEMM on A100", section "Performance comparison"; the
 * axpby epilogue of "CuTe-ly writing an SM86 SGEMM", section "epilogue",
 * extended by per-row scaling, "Matmul II", section 6, and a bias and an
 * activation applied to each element):
 *
 *   D(i,j) = act( alpha * s_i * sum_k op(A)(i,k) op(B)(k,j)
 *                 + beta * C(i,j) + bias_j )
 *
 * s = row_scale (M entries; NULL means every s_i = 1), bias (N entries;
 * NULL means 0), act 0 = identity, 1 = ReLU (max(x, 0)).  Evaluated in
 * fp64 exactly as the plain reference (alpha == 0: no product term, A and
 * B not read; beta == 0: C not read), ReLU applied to the fp64 value.
 * The bound adds the epilogue's own fp32 roundings (alpha*s_i, the fused
 * multiply-add with beta*c, the bias add: at most three, each within 2^-24
 * of the magnitudes involved) to the summation bound:
 *   bound = (4*K + 3) * 2^-24 * (|alpha*s_i| * sum_k |a||b|
 *                                + |beta|*|c| + |bias_j|);
 * ReLU is 1-Lipschitz and leaves it valid.
 */
int oracle_gemm_epilogue_f64(char ta, char tb, int64_t M, int64_t N, int64_t K,
                             float alpha, const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             float beta, const float *C, int64_t ldc,
                             const float *row_scale, const float *bias, int act,
                             const int64_t *rows, const int64_t *cols, int64_t npts,
                             double *ref, double *bound)
{
    int st = check_args(ta, tb, M, N, K, lda, ldb, ldc);
    if (st != ORACLE_OK) return st;
    if (act != 0 && act != 1) return -16;
    const int ta_n = is_n(ta), tb_n = is_n(tb);
    const int64_t total = rows ? npts : M * N;
    const double unit = ldexp(1.0, -24);

    int64_t p;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (p = 0; p < total; ++p) {
        const int64_t i = rows ? rows[p] : p / N;
        const int64_t j = rows ? cols[p] : p % N;
        const double scale = (double)alpha * (row_scale ? (double)row_scale[i] : 1.0);
        double sum = 0.0, mag = 0.0;
        const int64_t kend = (alpha == 0.0f) ? 0 : K;
        for (int64_t k = 0; k < kend; ++k) {
            const double a = (double)op_a(A, lda, ta_n, i, k);
            const double b = (double)op_b(B, ldb, tb_n, k, j);
            sum += a * b;
            mag += fabs(a) * fabs(b);
        }
        double r = (alpha == 0.0f) ? 0.0 : scale * sum;
        double m = fabs(scale) * mag;
        if (beta != 0.0f) {
            const double c = (double)C[i * ldc + j];
            r += (double)beta * c;
            m += fabs((double)beta) * fabs(c);
        }
        if (bias) {
            r += (double)bias[j];
            m += fabs((double)bias[j]);
        }
        if (act == 1 && r < 0.0) r = 0.0;
        ref[p] = r;
        bound[p] = (4.0 * (double)K + 3.0) * unit * m;
    }
    return ORACLE_OK;
}
