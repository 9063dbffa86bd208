// The CP-ALS sweep around the MTTKRP ("A Performance Portable Matrix Free Dense
// MTTKRP in GenTen", Fig. 5: one MTTKRP per mode plus the other CP-ALS
// operations, an inner product and a Cholesky solve among them).  Per mode n:
// V = Hadamard product of the other modes' Gram matrices, M = MTTKRP(Y, A, n),
// A_n = M V^{-1} through the Cholesky factor of V, column 2-norms into lambda;
// after the sweep the fit from ||X||^2 = lambda^T (Hadamard of all Grams)
// lambda and <Y, X> = sum_r lambda_r sum_i M(i, r) A_{d-1}(i, r).
//
// The R x R algebra runs in fp64 (Gram sums, Cholesky, the two triangular
// solves, the fit); factors stay fp32.  Every reduction has a fixed order, so
// a sweep is bitwise reproducible.  The single-block Cholesky suits the ranks
// CP-ALS is run at (R up to a few hundred); it is correct, if slow, beyond.
#include "internal.h"

namespace mk {
namespace {

// G = A^T A (R x R, fp64) for A (I x R, fp32 row-major): 16 x 16 output tiles,
// 32-row slabs of the two column blocks staged in shared memory.
__global__ void __launch_bounds__(256) gram_kernel(const float* __restrict__ A, int64_t I, int R,
                                                   double* __restrict__ G) {
    __shared__ double sa[32][17], sb[32][17];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int r0 = blockIdx.y * 16, c0 = blockIdx.x * 16;
    double acc = 0.0;
    for (int64_t i0 = 0; i0 < I; i0 += 32) {
        for (int t = threadIdx.x; t < 32 * 16; t += 256) {
            const int ii = t / 16, cc = t % 16;
            const int64_t i = i0 + ii;
            sa[ii][cc] = (i < I && r0 + cc < R) ? (double)A[i * R + r0 + cc] : 0.0;
            sb[ii][cc] = (i < I && c0 + cc < R) ? (double)A[i * R + c0 + cc] : 0.0;
        }
        __syncthreads();
#pragma unroll 8
        for (int ii = 0; ii < 32; ++ii) acc = fma(sa[ii][ty], sb[ii][tx], acc);
        __syncthreads();
    }
    if (r0 + ty < R && c0 + tx < R) G[(int64_t)(r0 + ty) * R + c0 + tx] = acc;
}

// V = Hadamard product of G[m] over m != skip (skip < 0: all d)
__global__ void hadamard_kernel(const double* __restrict__ G, int d, int skip, int R, double* __restrict__ V) {
    const int64_t n = (int64_t)R * R;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        double v = 1.0;
        for (int m = 0; m < d; ++m)
            if (m != skip) v *= G[m * n + e];
        V[e] = v;
    }
}

// In-place lower Cholesky factor of the symmetric matrix V (row-major; the
// strict upper triangle is left as it was).  *info = j + 1 if the j-th pivot is
// not positive (then the factor holds NaN from there on).  One block.
__global__ void __launch_bounds__(1024) cholesky_kernel(double* __restrict__ V, int R, int* __restrict__ info) {
    __shared__ double piv;
    for (int j = 0; j < R; ++j) {
        if (threadIdx.x == 0) {
            const double p = V[(int64_t)j * R + j];
            if (!(p > 0.0) && *info == 0) *info = j + 1;
            piv = sqrt(p);
            V[(int64_t)j * R + j] = piv;
        }
        __syncthreads();
        const double l = piv;
        for (int i = j + 1 + threadIdx.x; i < R; i += blockDim.x) V[(int64_t)i * R + j] /= l;
        __syncthreads();
        // trailing lower triangle: V[i][k] -= V[i][j] V[k][j], j < k <= i
        const int n = R - j - 1;
        for (int64_t t = threadIdx.x; t < (int64_t)n * n; t += blockDim.x) {
            const int i = j + 1 + (int)(t / n), k = j + 1 + (int)(t % n);
            if (k <= i) V[(int64_t)i * R + k] -= V[(int64_t)i * R + j] * V[(int64_t)k * R + j];
        }
        __syncthreads();
    }
}

// X(i, :) = M(i, :) (L L^T)^{-1}: one warp per row, forward then back
// substitution, dot products split over the lanes and reduced by shuffles.
__global__ void __launch_bounds__(256) solve_kernel(const double* __restrict__ L, int R, const float* __restrict__ M,
                                                    int64_t I, double* __restrict__ X) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= I) return;
    double* x = X + row * R;
    const float* b = M + row * R;
    for (int k = 0; k < R; ++k) {          // L y = b
        double s = 0.0;
        for (int j = lane; j < k; j += 32) s = fma(L[(int64_t)k * R + j], x[j], s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) x[k] = ((double)b[k] - s) / L[(int64_t)k * R + k];
        __syncwarp();
    }
    for (int k = R - 1; k >= 0; --k) {     // L^T x = y
        double s = 0.0;
        for (int j = k + 1 + lane; j < R; j += 32) s = fma(L[(int64_t)j * R + k], x[j], s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) x[k] = (x[k] - s) / L[(int64_t)k * R + k];
        __syncwarp();
    }
}

// lambda_r = ||X(:, r)||_2 and A(:, r) = X(:, r) / lambda_r (0 for a zero
// column); one block per 32 columns, rows split over 8 warps in a fixed order.
__global__ void __launch_bounds__(256) normalize_kernel(const double* __restrict__ X, int64_t I, int R,
                                                        float* __restrict__ A, float* __restrict__ lam) {
    __shared__ double part[8][32];
    __shared__ double norm[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * 32 + lane;
    double s = 0.0;
    if (r < R)
        for (int64_t i = warp; i < I; i += 8) {
            const double v = X[i * R + r];
            s = fma(v, v, s);
        }
    part[warp][lane] = s;
    __syncthreads();
    if (warp == 0) {
        double t = 0.0;
        for (int w = 0; w < 8; ++w) t += part[w][lane];
        norm[lane] = sqrt(t);
        if (r < R) lam[r] = (float)norm[lane];
    }
    __syncthreads();
    const double nr = norm[lane];
    if (r < R)
        for (int64_t i = warp; i < I; i += 8) A[i * R + r] = nr > 0.0 ? (float)(X[i * R + r] / nr) : 0.f;
}

__device__ double block_sum(double v, double* sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += sh[w];
    __syncthreads();
    return t;   // valid in thread 0
}

// fit = 1 - sqrt(max(||Y||^2 + lambda^T H lambda - 2 <Y, X>, 0)) / ||Y||, with
// <Y, X> = sum_r lambda_r sum_i M(i, r) A(i, r); NaN if the Cholesky failed.
__global__ void __launch_bounds__(256) fit_kernel(const double* __restrict__ H, const float* __restrict__ lam,
                                                  const float* __restrict__ M, const float* __restrict__ A,
                                                  int64_t I, int R, const double* __restrict__ norm_y2,
                                                  const int* __restrict__ info, double* __restrict__ fit) {
    __shared__ double sh[8];
    double x2 = 0.0, in = 0.0;
    for (int64_t e = threadIdx.x; e < (int64_t)R * R; e += blockDim.x)
        x2 += (double)lam[e / R] * H[e] * (double)lam[e % R];
    for (int64_t e = threadIdx.x; e < I * R; e += blockDim.x)
        in += (double)lam[e % R] * (double)M[e] * (double)A[e];
    x2 = block_sum(x2, sh);
    in = block_sum(in, sh);
    if (threadIdx.x == 0) {
        const double y2 = *norm_y2;
        const double res2 = y2 + x2 - 2.0 * in;
        *fit = (*info != 0) ? __longlong_as_double(0x7ff8000000000000ll)
                            : 1.0 - sqrt(res2 > 0.0 ? res2 : 0.0) / sqrt(y2);
    }
}

// ||Y||^2 in fp64: fixed-order block partials, then one block adds them
constexpr int kSqBlocks = 1024;
__global__ void __launch_bounds__(256) sumsq_partial_kernel(const float* __restrict__ y, int64_t n,
                                                            double* __restrict__ part) {
    __shared__ double sh[8];
    double s = 0.0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const double v = (double)y[i];
        s = fma(v, v, s);
    }
    s = block_sum(s, sh);
    if (threadIdx.x == 0) part[blockIdx.x] = s;
}

__global__ void __launch_bounds__(256) sumsq_final_kernel(const double* __restrict__ part, int n,
                                                          double* __restrict__ out) {
    __shared__ double sh[8];
    double s = 0.0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s += part[i];
    s = block_sum(s, sh);
    if (threadIdx.x == 0) *out = s;
}

}  // namespace

cudaError_t cpals_gram(const float* A, int64_t I, int R, double* G, cudaStream_t s) {
    dim3 grid((unsigned)((R + 15) / 16), (unsigned)((R + 15) / 16));
    gram_kernel<<<grid, 256, 0, s>>>(A, I, R, G);
    return cudaGetLastError();
}

cudaError_t cpals_hadamard(const double* G, int d, int skip, int R, double* V, cudaStream_t s) {
    const int64_t n = (int64_t)R * R;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    hadamard_kernel<<<(unsigned)blocks, 256, 0, s>>>(G, d, skip, R, V);
    return cudaGetLastError();
}

cudaError_t cpals_cholesky(double* V, int R, int* info, cudaStream_t s) {
    cholesky_kernel<<<1, 1024, 0, s>>>(V, R, info);
    return cudaGetLastError();
}

cudaError_t cpals_solve(const double* L, int R, const float* M, int64_t I, double* X, cudaStream_t s) {
    solve_kernel<<<(unsigned)((I + 7) / 8), 256, 0, s>>>(L, R, M, I, X);
    return cudaGetLastError();
}

cudaError_t cpals_normalize(const double* X, int64_t I, int R, float* A, float* lam, cudaStream_t s) {
    normalize_kernel<<<(unsigned)((R + 31) / 32), 256, 0, s>>>(X, I, R, A, lam);
    return cudaGetLastError();
}

cudaError_t cpals_fit(const double* H, const float* lam, const float* M, const float* A, int64_t I, int R,
                      const double* norm_y2, const int* info, double* fit, cudaStream_t s) {
    fit_kernel<<<1, 256, 0, s>>>(H, lam, M, A, I, R, norm_y2, info, fit);
    return cudaGetLastError();
}

size_t cpals_sumsq_scratch_bytes() { return kSqBlocks * sizeof(double); }

cudaError_t cpals_sum_squares(const float* Y, int64_t n, double* part, double* out, cudaStream_t s) {
    sumsq_partial_kernel<<<kSqBlocks, 256, 0, s>>>(Y, n, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sumsq_final_kernel<<<1, 256, 0, s>>>(part, kSqBlocks, out);
    return cudaGetLastError();
}

}  // namespace mk
