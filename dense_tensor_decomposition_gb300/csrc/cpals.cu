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
// a sweep is bitwise reproducible.
#include "internal.h"

namespace mk {
namespace {

// G = A^T A (R x R, fp64) for A (I x R, fp32 row-major): 16 x 16 output tiles,
// 32-row slabs of the two column blocks staged in shared memory.  blockIdx.z
// takes every gridDim.z-th slab and writes its partial Gram to part[z]; the
// partials are then added in z order (gram_sum_kernel).
__global__ void __launch_bounds__(256) gram_kernel(const float* __restrict__ A, int64_t I, int R,
                                                   double* __restrict__ part) {
    __shared__ double sa[32][17], sb[32][17];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int r0 = blockIdx.y * 16, c0 = blockIdx.x * 16;
    double* G = part + (int64_t)blockIdx.z * R * R;
    double acc = 0.0;
    for (int64_t i0 = 32 * (int64_t)blockIdx.z; i0 < I; i0 += 32 * (int64_t)gridDim.z) {
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

__global__ void gram_sum_kernel(const double* __restrict__ part, int S, int R, double* __restrict__ G) {
    const int64_t n = (int64_t)R * R;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        double v = 0.0;
        for (int z = 0; z < S; ++z) v += part[z * n + e];
        G[e] = v;
    }
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
// strict upper triangle is left as it was), right-looking in 32-column panels:
// factor the diagonal block (one CTA, in shared memory), solve the panel below
// it, update the trailing lower triangle (32 x 32 tiles).  *info = j + 1 if the
// j-th pivot is not positive (the factor then holds NaN from there on).
constexpr int kChNB = 32;

__global__ void __launch_bounds__(256) chol_diag_kernel(double* __restrict__ V, int R, int k0, int nb,
                                                        int* __restrict__ info, double* __restrict__ dinv) {
    __shared__ double a[kChNB][kChNB + 1];
    for (int t = threadIdx.x; t < nb * nb; t += blockDim.x) {
        const int i = t / nb, j = t % nb;
        a[i][j] = j <= i ? V[(int64_t)(k0 + i) * R + k0 + j] : 0.0;
    }
    __syncthreads();
    for (int j = 0; j < nb; ++j) {
        if (threadIdx.x == 0) {
            const double p = a[j][j];
            if (!(p > 0.0) && *info == 0) *info = k0 + j + 1;
            a[j][j] = sqrt(p);
        }
        __syncthreads();
        const double inv = 1.0 / a[j][j];
        if (threadIdx.x == 0) dinv[k0 + j] = inv;
        for (int i = j + 1 + threadIdx.x; i < nb; i += blockDim.x) a[i][j] *= inv;
        __syncthreads();
        const int n = nb - j - 1;
        for (int t = threadIdx.x; t < n * n; t += blockDim.x) {
            const int i = j + 1 + t / n, k = j + 1 + t % n;
            if (k <= i) a[i][k] -= a[i][j] * a[k][j];
        }
        __syncthreads();
    }
    for (int t = threadIdx.x; t < nb * nb; t += blockDim.x) {
        const int i = t / nb, j = t % nb;
        if (j <= i) V[(int64_t)(k0 + i) * R + k0 + j] = a[i][j];
    }
}

// rows i >= k0 + nb of the panel: x = v L11^{-T} (forward substitution)
__global__ void __launch_bounds__(256) chol_panel_kernel(double* __restrict__ V, int R, int k0, int nb,
                                                         const double* __restrict__ dinv) {
    __shared__ double l[kChNB][kChNB + 1];
    for (int t = threadIdx.x; t < nb * nb; t += blockDim.x) {
        const int i = t / nb, j = t % nb;
        l[i][j] = j <= i ? V[(int64_t)(k0 + i) * R + k0 + j] : 0.0;
    }
    __syncthreads();
    for (int i = k0 + nb + blockIdx.x * blockDim.x + threadIdx.x; i < R; i += gridDim.x * blockDim.x) {
        double x[kChNB];
        double* v = V + (int64_t)i * R + k0;
#pragma unroll
        for (int j = 0; j < kChNB; ++j) {
            if (j < nb) {
                double s = v[j];
#pragma unroll
                for (int t = 0; t < j; ++t) s -= x[t] * l[j][t];
                x[j] = s * dinv[k0 + j];
                v[j] = x[j];
            }
        }
    }
}

// trailing lower triangle: V[i][j] -= sum_t P[i][t] P[j][t], k0 + nb <= j <= i
__global__ void __launch_bounds__(256) chol_update_kernel(double* __restrict__ V, int R, int k0, int nb) {
    if (blockIdx.x > blockIdx.y) return;   // upper tiles
    __shared__ double pi[kChNB][kChNB + 1], pj[kChNB][kChNB + 1];
    const int i0 = k0 + nb + blockIdx.y * kChNB, j0 = k0 + nb + blockIdx.x * kChNB;
    for (int t = threadIdx.x; t < kChNB * kChNB; t += blockDim.x) {
        const int r = t / kChNB, c = t % kChNB;
        pi[r][c] = (i0 + r < R && c < nb) ? V[(int64_t)(i0 + r) * R + k0 + c] : 0.0;
        pj[r][c] = (j0 + r < R && c < nb) ? V[(int64_t)(j0 + r) * R + k0 + c] : 0.0;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < kChNB * kChNB; t += blockDim.x) {
        const int r = t / kChNB, c = t % kChNB;
        const int i = i0 + r, j = j0 + c;
        if (i < R && j <= i) {
            double s = 0.0;
#pragma unroll 8
            for (int u = 0; u < kChNB; ++u) s = fma(pi[r][u], pj[c][u], s);
            V[(int64_t)i * R + j] -= s;
        }
    }
}

// Mirror the lower Cholesky factor into the strict upper triangle (V[j][k] =
// L[k][j], j < k), so that both substitutions read L with consecutive lanes on
// consecutive addresses.
__global__ void mirror_lower_kernel(double* __restrict__ V, int R) {
    const int64_t n = (int64_t)R * R;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(e / R), k = (int)(e % R);
        if (j < k) V[e] = V[(int64_t)k * R + j];
    }
}

// X(i, :) = M(i, :) (L L^T)^{-1}, one warp per row i, the row's unknowns in
// shared memory.  Both substitutions go in blocks of 32 unknowns, lane l owning
// unknown k0 + l: the contributions of the finished blocks are one dot product
// per lane (all lanes at once), and within the block the unknowns are finished
// one by one, each broadcast by a shuffle to the lanes that still need it.
__global__ void __launch_bounds__(256) solve_kernel(const double* __restrict__ L, const double* __restrict__ dinv,
                                                    int R, const float* __restrict__ M, int64_t I,
                                                    double* __restrict__ X) {
    extern __shared__ double xs[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
    if (row >= I) return;
    double* x = xs + (int64_t)warp * R;
    for (int k = lane; k < R; k += 32) x[k] = (double)M[row * R + k];
    __syncwarp();
    // L y = b: y_k = (b_k - sum_{j<k} L[k][j] y_j) / L[k][k]
    for (int k0 = 0; k0 < R; k0 += 32) {
        const int k = k0 + lane;
        const bool live = k < R;
        double acc = live ? x[k] : 0.0;
        if (live)
            for (int j = 0; j < k0; ++j) acc -= L[(int64_t)j * R + k] * x[j];   // upper mirror: L[k][j]
        const int nb = R - k0 < 32 ? R - k0 : 32;
        for (int t = 0; t < nb; ++t) {
            const double yt = __shfl_sync(0xffffffffu, acc, t) * dinv[k0 + t];
            if (lane == t)
                acc = yt;
            else if (lane > t && live)
                acc -= L[(int64_t)k * R + k0 + t] * yt;
        }
        if (live) x[k] = acc;
        __syncwarp();
    }
    // L^T x = y: x_k = (y_k - sum_{j>k} L[j][k] x_j) / L[k][k]
    for (int k0 = ((R - 1) / 32) * 32; k0 >= 0; k0 -= 32) {
        const int k = k0 + lane;
        const bool live = k < R;
        double acc = live ? x[k] : 0.0;
        if (live)
            for (int j = k0 + 32; j < R; ++j) acc -= L[(int64_t)j * R + k] * x[j];
        const int nb = R - k0 < 32 ? R - k0 : 32;
        for (int t = nb - 1; t >= 0; --t) {
            const double xt = __shfl_sync(0xffffffffu, acc, t) * dinv[k0 + t];
            if (lane == t)
                acc = xt;
            else if (lane < t && live)
                acc -= L[(int64_t)(k0 + t) * R + k] * xt;
        }
        if (live) x[k] = acc;
        __syncwarp();
    }
    for (int k = lane; k < R; k += 32) X[row * R + k] = x[k];
}

// lambda_r = ||X(:, r)||_2 and A(:, r) = X(:, r) / lambda_r (0 for a zero
// column); one block per 32 columns, rows split over 32 warps in a fixed order.
__global__ void __launch_bounds__(1024) normalize_kernel(const double* __restrict__ X, int64_t I, int R,
                                                         float* __restrict__ A, float* __restrict__ lam) {
    __shared__ double part[32][32];
    __shared__ double norm[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * 32 + lane;
    double s = 0.0;
    if (r < R)
        for (int64_t i = warp; i < I; i += 32) {
            const double v = X[i * R + r];
            s = fma(v, v, s);
        }
    part[warp][lane] = s;
    __syncthreads();
    if (warp == 0) {
        double t = 0.0;
        for (int w = 0; w < 32; ++w) t += part[w][lane];
        norm[lane] = sqrt(t);
        if (r < R) lam[r] = (float)norm[lane];
    }
    __syncthreads();
    const double nr = norm[lane];
    const double inv = nr > 0.0 ? 1.0 / nr : 0.0;
    if (r < R)
        for (int64_t i = warp; i < I; i += 32) A[i * R + r] = (float)(X[i * R + r] * inv);
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
__global__ void __launch_bounds__(1024) fit_kernel(const double* __restrict__ H, const float* __restrict__ lam,
                                                   const float* __restrict__ M, const float* __restrict__ A,
                                                   int64_t I, int R, const double* __restrict__ norm_y2,
                                                   const int* __restrict__ info, double* __restrict__ fit) {
    __shared__ double sh[32];
    double x2 = 0.0, in = 0.0;
    // thread t takes columns c = t mod 32 + 32 q and rows r = t / 32 + 32 p
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int c = lane; c < R; c += 32) {
        const double lc = (double)lam[c];
        for (int r = warp; r < R; r += 32) x2 += (double)lam[r] * H[(int64_t)r * R + c] * lc;
        double t = 0.0;
        for (int64_t i = warp; i < I; i += 32) t += (double)M[i * R + c] * (double)A[i * R + c];
        in += lc * t;
    }
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
    const int64_t n4 = n / 4;   // y is 16-byte aligned
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = t0; i < n4; i += stride) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(y) + i);
        // four squares in fp32 (each within one rounding), accumulated in fp64
        s += (double)fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, v.w * v.w)));
    }
    for (int64_t i = 4 * n4 + t0; i < n; i += stride) s += (double)y[i] * (double)y[i];
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

int cpals_gram_slabs(int64_t I, int R) {
    // enough CTAs to fill the GPU, at least one 32-row slab each
    const int64_t tiles = (int64_t)((R + 15) / 16) * ((R + 15) / 16);
    int64_t S = (152 * 4 + tiles - 1) / tiles;
    const int64_t slabs = (I + 31) / 32;
    if (S > slabs) S = slabs;
    if (S > 64) S = 64;
    return S < 1 ? 1 : (int)S;
}

cudaError_t cpals_gram(const float* A, int64_t I, int R, double* G, double* part, cudaStream_t s) {
    const int S = cpals_gram_slabs(I, R);
    dim3 grid((unsigned)((R + 15) / 16), (unsigned)((R + 15) / 16), (unsigned)S);
    gram_kernel<<<grid, 256, 0, s>>>(A, I, R, S == 1 ? G : part);
    if (S > 1) {
        const int64_t n = (int64_t)R * R;
        int64_t blocks = (n + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        gram_sum_kernel<<<(unsigned)blocks, 256, 0, s>>>(part, S, R, G);
    }
    return cudaGetLastError();
}

cudaError_t cpals_hadamard(const double* G, int d, int skip, int R, double* V, cudaStream_t s) {
    const int64_t n = (int64_t)R * R;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    hadamard_kernel<<<(unsigned)blocks, 256, 0, s>>>(G, d, skip, R, V);
    return cudaGetLastError();
}

cudaError_t cpals_cholesky(double* V, int R, int* info, double* dinv, cudaStream_t s) {
    for (int k0 = 0; k0 < R; k0 += kChNB) {
        const int nb = R - k0 < kChNB ? R - k0 : kChNB;
        chol_diag_kernel<<<1, 256, 0, s>>>(V, R, k0, nb, info, dinv);
        const int rest = R - k0 - nb;
        if (rest > 0) {
            chol_panel_kernel<<<(unsigned)((rest + 255) / 256), 256, 0, s>>>(V, R, k0, nb, dinv);
            const unsigned nt = (unsigned)((rest + kChNB - 1) / kChNB);
            chol_update_kernel<<<dim3(nt, nt), 256, 0, s>>>(V, R, k0, nb);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int cpals_cholesky_launches(int R) {
    int n = 0;
    for (int k0 = 0; k0 < R; k0 += kChNB) n += (R - k0 > kChNB) ? 3 : 1;
    return n;
}

cudaError_t cpals_solve(double* L, const double* dinv, int R, const float* M, int64_t I, double* X,
                        cudaStream_t s) {
    // one warp per row, its R unknowns in shared memory (at most 96 KB a block)
    int warps = (int)((96 * 1024) / ((size_t)R * sizeof(double)));
    if (warps > 8) warps = 8;
    if (warps < 1) return cudaErrorInvalidValue;   // R > 12288
    const size_t smem = (size_t)warps * R * sizeof(double);
    cudaError_t e = cudaFuncSetAttribute(solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    {
        const int64_t n = (int64_t)R * R;
        int64_t blocks = (n + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        mirror_lower_kernel<<<(unsigned)blocks, 256, 0, s>>>(L, R);
    }
    solve_kernel<<<(unsigned)((I + warps - 1) / warps), warps * 32, smem, s>>>(L, dinv, R, M, I, X);
    return cudaGetLastError();
}

cudaError_t cpals_normalize(const double* X, int64_t I, int R, float* A, float* lam, cudaStream_t s) {
    normalize_kernel<<<(unsigned)((R + 31) / 32), 1024, 0, s>>>(X, I, R, A, lam);
    return cudaGetLastError();
}

cudaError_t cpals_fit(const double* H, const float* lam, const float* M, const float* A, int64_t I, int R,
                      const double* norm_y2, const int* info, double* fit, cudaStream_t s) {
    fit_kernel<<<1, 1024, 0, s>>>(H, lam, M, A, I, R, norm_y2, info, fit);
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
