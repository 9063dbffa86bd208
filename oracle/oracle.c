/*
 * fp64 reference oracle for dense MTTKRP.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this library; the GPU
 * library never does, and this file shares no code with it.
 *
 * What it computes (the definition, written out):
 *
 *   M_k(i, r) = sum over all (i_n)_{n != k} of  Y(i_0, .., i_{d-1}) * prod_{n != k} A_n(i_n, r)
 *
 * with i_k = i.  This is the "matricized tensor times Khatri-Rao product"
 * that "A Performance Portable Matrix Free Dense MTTKRP in GenTen" (abstract)
 * names as the workhorse kernel of CP decomposition: M_k = Y_(k) * KRP, where
 * Y_(k) is the mode-k unfolding (rows i_k, columns the other indices in a fixed,
 * consistent order; "An HPC Approach to Accelerate Tensor Decompositions",
 * section 2) and row kappa of the Khatri-Rao product is the elementwise product
 * of the factor rows A_n(i_n(kappa), :) over n != k.
 *
 * Layouts: Y is C-order (last index fastest), A_n is I_n x R row-major, the
 * output is rows x R row-major.  All arithmetic is fp64; fp32 inputs are
 * converted exactly.  Compiled with -ffp-contract=off so that the result does
 * not depend on whether the host compiler fuses multiply-adds.
 *
 * Two entry points:
 *   oracle_mttkrp_naive  one multi-index at a time, product recomputed per
 *                        element; single thread; tiny inputs only.
 *   oracle_mttkrp        the unfolding times the Khatri-Rao product, one KRP
 *                        row formed per column kappa of the unfolding and
 *                        reused for every requested output row.  The column
 *                        range is cut into a fixed number of chunks that
 *                        depends only on the problem size; chunk partial sums
 *                        are added in chunk order, so the result is bitwise
 *                        independent of the OpenMP thread count.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_D 16

static int check_args(int d, const int64_t* dims, int64_t R, int k) {
    if (d < 2 || d > ORACLE_MAX_D || R < 1 || k < 0 || k >= d || dims == NULL) return -1;
    for (int n = 0; n < d; ++n)
        if (dims[n] < 1) return -1;
    return 0;
}

int oracle_mttkrp_naive(int d, const int64_t* dims, int64_t R, const double* Y,
                        const double* const* A, int k, double* M) {
    if (check_args(d, dims, R, k) || !Y || !A || !M) return -1;
    int64_t total = 1;
    for (int n = 0; n < d; ++n) total *= dims[n];
    memset(M, 0, sizeof(double) * (size_t)(dims[k] * R));
    int64_t idx[ORACLE_MAX_D];
    for (int64_t lin = 0; lin < total; ++lin) {
        /* multi-index of element lin in C order */
        int64_t rem = lin;
        for (int n = d - 1; n >= 0; --n) {
            idx[n] = rem % dims[n];
            rem /= dims[n];
        }
        double y = Y[lin];
        for (int64_t r = 0; r < R; ++r) {
            double prod = 1.0;
            for (int n = 0; n < d; ++n)
                if (n != k) prod *= A[n][idx[n] * R + r];
            M[idx[k] * R + r] += y * prod;
        }
    }
    return 0;
}

/* Number of column chunks: fixed by the problem (never by the thread count),
 * at most 64, and small enough that the chunk buffers stay below 2^24 doubles. */
static int64_t chunk_count(int64_t ncols, int64_t nrows, int64_t R) {
    int64_t per = nrows * R;
    int64_t c = (int64_t)1 << 24;
    c = per > 0 ? c / per : 64;
    if (c > 64) c = 64;
    if (c < 1) c = 1;
    if (c > ncols) c = ncols;
    return c;
}

int oracle_mttkrp(int d, const int64_t* dims, int64_t R, const void* Y, int y_is_f64,
                  const double* const* A, int k, const int64_t* rows, int64_t nrows,
                  double* M) {
    if (check_args(d, dims, R, k) || !Y || !A || !M) return -1;
    const int64_t Ik = dims[k];
    if (rows == NULL) nrows = Ik;
    if (nrows < 0) return -1;
    for (int64_t t = 0; rows && t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= Ik) return -1;
    memset(M, 0, sizeof(double) * (size_t)(nrows * R));
    if (nrows == 0) return 0;

    /* C-order strides of Y, and the list of modes other than k (first = slowest) */
    int64_t stride[ORACLE_MAX_D];
    stride[d - 1] = 1;
    for (int n = d - 2; n >= 0; --n) stride[n] = stride[n + 1] * dims[n + 1];
    int other[ORACLE_MAX_D];
    int m = 0;
    int64_t ncols = 1;
    for (int n = 0; n < d; ++n)
        if (n != k) {
            other[m++] = n;
            ncols *= dims[n];
        }

    const int64_t nchunk = chunk_count(ncols, nrows, R);
    double* part = (double*)calloc((size_t)(nchunk * nrows * R), sizeof(double));
    if (!part) return -2;
    const float* Yf = (const float*)Y;
    const double* Yd = (const double*)Y;

#pragma omp parallel
    {
        double* w = (double*)malloc(sizeof(double) * (size_t)R);
#pragma omp for schedule(dynamic, 1)
        for (int64_t c = 0; c < nchunk; ++c) {
            int64_t lo = ncols * c / nchunk, hi = ncols * (c + 1) / nchunk;
            double* acc = part + c * nrows * R;
            int64_t jdx[ORACLE_MAX_D]; /* indices of the other modes for column kappa */
            int64_t rem = lo;
            for (int t = m - 1; t >= 0; --t) {
                jdx[t] = rem % dims[other[t]];
                rem /= dims[other[t]];
            }
            for (int64_t kappa = lo; kappa < hi; ++kappa) {
                /* Khatri-Rao row kappa and the offset of column kappa of Y_(k) */
                int64_t base = 0;
                for (int64_t r = 0; r < R; ++r) w[r] = 1.0;
                for (int t = 0; t < m; ++t) {
                    const double* arow = A[other[t]] + jdx[t] * R;
                    for (int64_t r = 0; r < R; ++r) w[r] *= arow[r];
                    base += jdx[t] * stride[other[t]];
                }
                for (int64_t t = 0; t < nrows; ++t) {
                    int64_t i = rows ? rows[t] : t;
                    int64_t off = base + i * stride[k];
                    double y = y_is_f64 ? Yd[off] : (double)Yf[off];
                    double* a = acc + t * R;
                    for (int64_t r = 0; r < R; ++r) a[r] += y * w[r];
                }
                /* next column: odometer increment, last other-mode fastest */
                for (int t = m - 1; t >= 0; --t) {
                    if (++jdx[t] < dims[other[t]]) break;
                    jdx[t] = 0;
                }
            }
        }
        free(w);
    }
    /* fixed-order sum of the chunk partials */
    for (int64_t c = 0; c < nchunk; ++c) {
        const double* src = part + c * nrows * R;
        for (int64_t e = 0; e < nrows * R; ++e) M[e] += src[e];
    }
    free(part);
    return 0;
}

/* Thread count the OpenMP runtime will use (reported by the CPU baseline). */
int oracle_threads(void) {
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
