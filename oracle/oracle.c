/*
 * oracle.c -- plain CPU reference for the BF16 GEMM and the implicit-GEMM
 * convolution. TEST INFRASTRUCTURE ONLY: tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library never does.
 *
 * What it computes is the textbook definition, in fp64, with nothing blocked,
 * fused or reordered:
 *
 *   GEMM (the "BF16 GEMM C = A.B" the pipelined tensor-core mainloop serves,
 *   "two-free-pipeline-stages" note, 256x128x64 tile discussion):
 *       ref[i][j] = sum_{k<K} a(i,k) * b(k,j)
 *       abs[i][j] = sum_{k<K} |a(i,k) * b(k,j)|
 *   with A row-major (a(i,k) = A[i*lda + k]) and B column-major, i.e. stored
 *   as N rows of K (b(k,j) = B[j*ldb + k]).
 *
 *   Convolution (forward, implicit-GEMM form of the same mainloop, same note,
 *   "SM100_TMA_2SM_LOAD_IM2COL"): cross-correlation, zero padding, no
 *   dilation, no groups,
 *       ref[n][p][q][k] = sum_{r,s,c} x[n][p*st-pad+r][q*st-pad+s][c] * w[k][r][s][c]
 *   where taps that fall outside the input contribute zero; abs likewise
 *   over |.|. x is NHWC, w is KRSC, y is NPQK with
 *   P = (H + 2 pad - R) / st + 1 and Q = (W + 2 pad - S) / st + 1.
 *
 * bf16 operands are decoded exactly (bits << 16 is the fp32 value) and every
 * product of two bf16 values is exact in fp64, so the only rounding is the
 * fp64 summation. OpenMP (when available) splits the outermost loop only.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Sub-block of the GEMM: rows[0..nrows) x cols[0..ncols) of C (NULL index
 * list = every row / every column). ref and absb are nrows x ncols,
 * row-major.
 */
void oracle_gemm(const uint16_t *A, const uint16_t *B,
                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                 const int64_t *rows, int64_t nrows,
                 const int64_t *cols, int64_t ncols,
                 double *ref, double *absb)
{
    if (rows == NULL) nrows = M;
    if (cols == NULL) ncols = N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ii = 0; ii < nrows; ++ii) {
        const int64_t i = rows ? rows[ii] : ii;
        for (int64_t jj = 0; jj < ncols; ++jj) {
            const int64_t j = cols ? cols[jj] : jj;
            double sum = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double prod = bf16_value(A[i * lda + k]) * bf16_value(B[j * ldb + k]);
                sum += prod;
                sabs += fabs(prod);
            }
            ref[ii * ncols + jj] = sum;
            absb[ii * ncols + jj] = sabs;
        }
    }
}

/*
 * Output pixels pix[0..npix) (linear index n*P*Q + p*Q + q; NULL = all) times
 * every output channel k. ref and absb are npix x K, row-major.
 */
void oracle_conv(const uint16_t *x, const uint16_t *w,
                 int64_t N, int64_t H, int64_t W, int64_t C,
                 int64_t K, int64_t R, int64_t S, int64_t st, int64_t pad,
                 const int64_t *pix, int64_t npix,
                 double *ref, double *absb)
{
    const int64_t P = (H + 2 * pad - R) / st + 1;
    const int64_t Q = (W + 2 * pad - S) / st + 1;
    if (pix == NULL) npix = N * P * Q;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < npix; ++t) {
        const int64_t m = pix ? pix[t] : t;
        const int64_t n = m / (P * Q);
        const int64_t p = (m / Q) % P;
        const int64_t q = m % Q;
        for (int64_t k = 0; k < K; ++k) {
            double sum = 0.0, sabs = 0.0;
            for (int64_t r = 0; r < R; ++r) {
                const int64_t h = p * st - pad + r;
                if (h < 0 || h >= H) continue;
                for (int64_t s = 0; s < S; ++s) {
                    const int64_t ww = q * st - pad + s;
                    if (ww < 0 || ww >= W) continue;
                    const uint16_t *xp = x + ((n * H + h) * W + ww) * C;
                    const uint16_t *wp = w + ((k * R + r) * S + s) * C;
                    for (int64_t c = 0; c < C; ++c) {
                        const double prod = bf16_value(xp[c]) * bf16_value(wp[c]);
                        sum += prod;
                        sabs += fabs(prod);
                    }
                }
            }
            ref[t * K + k] = sum;
            absb[t * K + k] = sabs;
        }
    }
}
