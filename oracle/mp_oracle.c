/*
 * mp_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct fp64 CPU oracle for the dense GEMM with
 * epilogue
 *
 *     D[i][j] = alpha * sum_k A[i][k] * B[k][j] + beta * C[i][j]
 *
 * with A, B given as bf16 bit patterns (row-major, leading dimensions lda,
 * ldb), C given as fp32 (row-major, ldc; never read when beta == 0) and D
 * returned in fp64.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library; the GPU library never does, and the
 * two share no code.
 *
 * Sources (page titles and sections):
 *   - "Optimizing Dynamic-Shape Neural Networks on Accelerators via On-the-Fly
 *     Micro-Kernel Polymerization" (MikPoly summary), preliminaries part 2 "loop tiling structure":
 *     the plain i-j-k matrix-multiply nest (C[i][j] zeroed, then accumulated
 *     over k) and the loop-tiled nest with TILE_SIZE 32.
 *   - BOLT summary, "Persistent kernel (GEMM/Conv) fusion": the epilogue form
 *     D = alpha*A*W + beta*C.
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *   - M, N, K are run-time sizes (the printed nest uses undefined M and K).
 *   - The printed tiled nest neither zeroes C nor clamps the tile edges; here
 *     D starts at zero and every tile loop is clamped to the matrix edge, so
 *     the nest is defined for sizes that are not multiples of 32.
 *   - bf16 is the upper 16 bits of an IEEE binary32; widening is exact.
 *
 * Build: plain C, -O2 -ffp-contract=off (no fused multiply-add, no
 * reassociation), OpenMP only for the row-parallel variant.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64: the bf16 bits are the high half of an fp32 word. */
static double widen_bf16(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double c_term(const float* C, int64_t ldc, int64_t i, int64_t j, double beta) {
    if (beta == 0.0) return 0.0; /* BLAS convention: C is not read */
    return beta * (double)C[i * ldc + j];
}

/*
 * The plain nest of the MikPoly summary, preliminaries part 2: for each (i, j), zero
 * the accumulator and add A[i][k]*B[k][j] for k = 0..K-1 in order; then the
 * epilogue of the BOLT summary.
 */
void oracle_gemm_naive(int64_t M, int64_t N, int64_t K,
                       const uint16_t* A, int64_t lda,
                       const uint16_t* B, int64_t ldb,
                       const float* C, int64_t ldc,
                       double alpha, double beta,
                       double* D, int64_t ldd) {
    for (int64_t i = 0; i < M; i++) {
        for (int64_t j = 0; j < N; j++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++)
                acc += widen_bf16(A[i * lda + k]) * widen_bf16(B[k * ldb + j]);
            D[i * ldd + j] = alpha * acc + c_term(C, ldc, i, j, beta);
        }
    }
}

/*
 * The loop-tiled nest of the MikPoly summary, preliminaries part 2 (TILE_SIZE 32):
 * tiles of i, j, k outermost, then ii, jj, kk inside each tile, accumulating
 * straight into the output.  The output is zeroed first and every tile is
 * clamped to the matrix edge (reading noted above).  The sum for one (i, j)
 * runs over k in increasing order, tile by tile, exactly like the plain nest,
 * so on inputs whose partial sums are exact the two agree bit for bit.
 */
#define ORACLE_TILE 32
void oracle_gemm_tiled(int64_t M, int64_t N, int64_t K,
                       const uint16_t* A, int64_t lda,
                       const uint16_t* B, int64_t ldb,
                       const float* C, int64_t ldc,
                       double alpha, double beta,
                       double* D, int64_t ldd) {
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++) D[i * ldd + j] = 0.0;
    for (int64_t i = 0; i < M; i += ORACLE_TILE) {
        int64_t ie = i + ORACLE_TILE < M ? i + ORACLE_TILE : M;
        for (int64_t j = 0; j < N; j += ORACLE_TILE) {
            int64_t je = j + ORACLE_TILE < N ? j + ORACLE_TILE : N;
            for (int64_t k = 0; k < K; k += ORACLE_TILE) {
                int64_t ke = k + ORACLE_TILE < K ? k + ORACLE_TILE : K;
                for (int64_t ii = i; ii < ie; ii++)
                    for (int64_t jj = j; jj < je; jj++)
                        for (int64_t kk = k; kk < ke; kk++)
                            D[ii * ldd + jj] += widen_bf16(A[ii * lda + kk]) *
                                                widen_bf16(B[kk * ldb + jj]);
            }
        }
    }
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++)
            D[i * ldd + j] = alpha * D[i * ldd + j] + c_term(C, ldc, i, j, beta);
}

/*
 * Same definition, loops reordered i-k-j so that one output row accumulates
 * with unit stride; rows are independent and shared out over OpenMP threads.
 * For each (i, j) the products are still added in increasing k.  Used for
 * large parity cases and as the timed CPU baseline.  Returns the number of
 * threads used.
 */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K,
                     const uint16_t* A, int64_t lda,
                     const uint16_t* B, int64_t ldb,
                     const float* C, int64_t ldc,
                     double alpha, double beta,
                     double* D, int64_t ldd, int threads) {
    int used = 1;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
    used = threads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t i = 0; i < M; i++) {
        double* d = D + i * ldd;
        for (int64_t j = 0; j < N; j++) d[j] = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double a = widen_bf16(A[i * lda + k]);
            const uint16_t* b = B + k * ldb;
            for (int64_t j = 0; j < N; j++) d[j] += a * widen_bf16(b[j]);
        }
        for (int64_t j = 0; j < N; j++) d[j] = alpha * d[j] + c_term(C, ldc, i, j, beta);
    }
    return used;
}

/*
 * Selected entries (rows[t], cols[t]) of the same definition, with the
 * element-wise magnitude  sum_k |A[i][k]||B[k][j]| + |beta*C[i][j]|  that the
 * parity tolerance scales with.  Used where the full product is too large.
 */
void oracle_gemm_entries(int64_t M, int64_t N, int64_t K,
                         const uint16_t* A, int64_t lda,
                         const uint16_t* B, int64_t ldb,
                         const float* C, int64_t ldc,
                         double alpha, double beta,
                         int64_t n, const int64_t* rows, const int64_t* cols,
                         double* out, double* mag) {
    (void)M; (void)N;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t t = 0; t < n; t++) {
        int64_t i = rows[t], j = cols[t];
        double acc = 0.0, abs_acc = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double p = widen_bf16(A[i * lda + k]) * widen_bf16(B[k * ldb + j]);
            acc += p;
            abs_acc += fabs(p);
        }
        double ct = c_term(C, ldc, i, j, beta);
        out[t] = alpha * acc + ct;
        if (mag) mag[t] = abs_acc + fabs(ct);
    }
}

/*
 * Full magnitude matrix  sum_k |A[i][k]||B[k][j]| + |beta*C[i][j]|  (fp64),
 * the scale of the parity bound for every entry.
 */
void oracle_gemm_magnitude(int64_t M, int64_t N, int64_t K,
                           const uint16_t* A, int64_t lda,
                           const uint16_t* B, int64_t ldb,
                           const float* C, int64_t ldc, double beta,
                           double* G, int64_t ldg) {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < M; i++) {
        double* g = G + i * ldg;
        for (int64_t j = 0; j < N; j++) g[j] = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double a = fabs(widen_bf16(A[i * lda + k]));
            const uint16_t* b = B + k * ldb;
            for (int64_t j = 0; j < N; j++) g[j] += a * fabs(widen_bf16(b[j]));
        }
        for (int64_t j = 0; j < N; j++) g[j] += fabs(c_term(C, ldc, i, j, beta));
    }
}

/*
 * Freivalds-style probe for outputs too large to recompute: given a candidate
 * D (fp32) and a probe vector x, return  y = D x - (alpha A (B x) + beta C x)
 * in fp64, and the matching magnitude  |alpha| |A| (|B| |x|) + |beta| |C| |x|
 * per row.  A correct D gives |y_i| within the accumulated rounding of the
 * entries of row i.  Right-multiplying keeps the cost at O(MK + KN + MN).
 */
void oracle_freivalds(int64_t M, int64_t N, int64_t K,
                      const uint16_t* A, int64_t lda,
                      const uint16_t* B, int64_t ldb,
                      const float* C, int64_t ldc,
                      double alpha, double beta,
                      const float* Dgpu, int64_t ldd,
                      const double* x, double* bx, double* abx,
                      double* y, double* ymag) {
    /* bx = B x, abx = |B| |x| */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t k = 0; k < K; k++) {
        double s = 0.0, sa = 0.0;
        for (int64_t j = 0; j < N; j++) {
            double b = widen_bf16(B[k * ldb + j]);
            s += b * x[j];
            sa += fabs(b) * fabs(x[j]);
        }
        bx[k] = s;
        abx[k] = sa;
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < M; i++) {
        double dx = 0.0, ab = 0.0, aab = 0.0, cx = 0.0, acx = 0.0;
        for (int64_t j = 0; j < N; j++) dx += (double)Dgpu[i * ldd + j] * x[j];
        for (int64_t k = 0; k < K; k++) {
            double a = widen_bf16(A[i * lda + k]);
            ab += a * bx[k];
            aab += fabs(a) * abx[k];
        }
        if (beta != 0.0) {
            for (int64_t j = 0; j < N; j++) {
                cx += (double)C[i * ldc + j] * x[j];
                acx += fabs((double)C[i * ldc + j]) * fabs(x[j]);
            }
        }
        y[i] = dx - (alpha * ab + beta * cx);
        ymag[i] = fabs(alpha) * aab + fabs(beta) * acx;
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
