// The CP-ALS sweep around the MTTKRP ("A Performance Portable Matrix Free Dense
// MTTKRP in GenTen", Fig. 5: one MTTKRP per mode plus the other CP-ALS
// operations, an inner product and a Cholesky solve among them).  Per mode n:
// V = Hadamard product of the other modes' Gram matrices, M = MTTKRP(Y, A, n),
// A_n = M V^{-1} through the Cholesky factor of V, column 2-norms into lambda;
// after the sweep the fit from ||X||^2 = lambda^T (Hadamard of all Grams)
// lambda and <Y, X> = sum_r lambda_r sum_i M(i, r) A_{d-1}(i, r).
//
// Precision.  GB300 runs fp64 at about 1/64 of its fp32 rate (two fused
// multiply-adds a clock an SM), so the O(I R^2) steps use fp32 arithmetic
// that keeps fp64-level accuracy, and fp64 is kept for the small O(R^2)
// steps:
//   * Gram matrices: exact fp32 products (p = a b and its rounding error
//     fma(a, b, -p)) summed with compensation, stored in fp64;
//   * A_n = M V^{-1}: V is factored in fp32 (blocked, 32-column panels), the
//     rows are solved in fp32, and one refinement step solves for the residual
//     M - X V, computed with V split into two fp32 words and compensated sums,
//     so the result carries the accuracy of V (fp64) rather than of the fp32
//     factor; it needs cond(V) well below 1 / 2^-24 (a failing fp32 pivot gives
//     a NaN fit).  Above R = 1024 the factor and solves run in fp64.
//   * Hadamard products, column norms and the fit in fp64.
// Factors stay fp32.  Every reduction has a fixed order, so a sweep is bitwise
// reproducible.
#include "internal.h"

namespace mk {
namespace {

// Compensated fp32 addition (Neumaier): sum + c carries the exact running total
// to about one fp32 rounding.
__device__ __forceinline__ void neumaier(float& sum, float& c, float x) {
    const float t = sum + x;
    c += fabsf(sum) >= fabsf(x) ? (sum - t) + x : (x - t) + sum;
    sum = t;
}

// G = A^T A (R x R, fp64) for A (I x R, fp32 row-major): 16 x 16 output tiles of
// the lower triangle (mirrored), 32-row slabs of the two column blocks staged in
// shared memory.  Each product a b is split exactly into p = fl(a b) and
// fma(a, b, -p); the p are summed with compensation and the small parts plainly,
// which gives the Gram to about fp64 accuracy on the fp32 pipe.  blockIdx.z
// takes every gridDim.z-th slab and writes its partial Gram to part[z]; the
// partials are then added in z order (gram_sum_kernel).
__global__ void __launch_bounds__(256) gram_kernel(const float* __restrict__ A, int64_t I, int R,
                                                   double* __restrict__ part) {
    if (blockIdx.x > blockIdx.y) return;   // upper tiles: mirrored from the lower ones
    __shared__ float sa[32][17], sb[32][17];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int r0 = blockIdx.y * 16, c0 = blockIdx.x * 16;
    double* G = part + (int64_t)blockIdx.z * R * R;
    float s = 0.f, c = 0.f, small = 0.f;
    for (int64_t i0 = 32 * (int64_t)blockIdx.z; i0 < I; i0 += 32 * (int64_t)gridDim.z) {
        for (int t = threadIdx.x; t < 32 * 16; t += 256) {
            const int ii = t / 16, cc = t % 16;
            const int64_t i = i0 + ii;
            sa[ii][cc] = (i < I && r0 + cc < R) ? A[i * R + r0 + cc] : 0.f;
            sb[ii][cc] = (i < I && c0 + cc < R) ? A[i * R + c0 + cc] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int ii = 0; ii < 32; ++ii) {
            const float a = sa[ii][ty], b = sb[ii][tx];
            const float p = a * b;
            small += fmaf(a, b, -p);
            neumaier(s, c, p);
        }
        __syncthreads();
    }
    const int r = r0 + ty, col = c0 + tx;
    if (r < R && col < R) {
        const double v = (double)s + ((double)c + (double)small);
        G[(int64_t)r * R + col] = v;
        G[(int64_t)col * R + r] = v;
    }
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

template <typename T>
__global__ void __launch_bounds__(256) chol_diag_kernel(T* __restrict__ V, int R, int k0, int nb,
                                                        int* __restrict__ info, T* __restrict__ dinv) {
    __shared__ T a[kChNB][kChNB + 1];
    for (int t = threadIdx.x; t < nb * nb; t += blockDim.x) {
        const int i = t / nb, j = t % nb;
        a[i][j] = j <= i ? V[(int64_t)(k0 + i) * R + k0 + j] : 0.0;
    }
    __syncthreads();
    for (int j = 0; j < nb; ++j) {
        if (threadIdx.x == 0) {
            const T p = a[j][j];
            if (!(p > T(0)) && *info == 0) *info = k0 + j + 1;
            a[j][j] = sqrt(p);
        }
        __syncthreads();
        const T inv = T(1) / a[j][j];
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
template <typename T>
__global__ void __launch_bounds__(256) chol_panel_kernel(T* __restrict__ V, int R, int k0, int nb,
                                                         const T* __restrict__ dinv) {
    __shared__ T l[kChNB][kChNB + 1];
    for (int t = threadIdx.x; t < nb * nb; t += blockDim.x) {
        const int i = t / nb, j = t % nb;
        l[i][j] = j <= i ? V[(int64_t)(k0 + i) * R + k0 + j] : 0.0;
    }
    __syncthreads();
    for (int i = k0 + nb + blockIdx.x * blockDim.x + threadIdx.x; i < R; i += gridDim.x * blockDim.x) {
        T x[kChNB];
        T* v = V + (int64_t)i * R + k0;
#pragma unroll
        for (int j = 0; j < kChNB; ++j) {
            if (j < nb) {
                T s = v[j];
#pragma unroll
                for (int t = 0; t < j; ++t) s -= x[t] * l[j][t];
                x[j] = s * dinv[k0 + j];
                v[j] = x[j];
            }
        }
    }
}

// trailing lower triangle: V[i][j] -= sum_t P[i][t] P[j][t], k0 + nb <= j <= i
template <typename T>
__global__ void __launch_bounds__(256) chol_update_kernel(T* __restrict__ V, int R, int k0, int nb) {
    if (blockIdx.x > blockIdx.y) return;   // upper tiles
    __shared__ T pi[kChNB][kChNB + 1], pj[kChNB][kChNB + 1];
    const int i0 = k0 + nb + blockIdx.y * kChNB, j0 = k0 + nb + blockIdx.x * kChNB;
    for (int t = threadIdx.x; t < kChNB * kChNB; t += blockDim.x) {
        const int r = t / kChNB, c = t % kChNB;
        pi[r][c] = (i0 + r < R && c < nb) ? V[(int64_t)(i0 + r) * R + k0 + c] : T(0);
        pj[r][c] = (j0 + r < R && c < nb) ? V[(int64_t)(j0 + r) * R + k0 + c] : T(0);
    }
    __syncthreads();
    for (int t = threadIdx.x; t < kChNB * kChNB; t += blockDim.x) {
        const int r = t / kChNB, c = t % kChNB;
        const int i = i0 + r, j = j0 + c;
        if (i < R && j <= i) {
            T s = T(0);
#pragma unroll 8
            for (int u = 0; u < kChNB; ++u) s = fma(pi[r][u], pj[c][u], s);
            V[(int64_t)i * R + j] -= s;
        }
    }
}

// Mirror the lower Cholesky factor into the strict upper triangle (V[j][k] =
// L[k][j], j < k), so that both substitutions read L with consecutive lanes on
// consecutive addresses.
template <typename T>
__global__ void mirror_lower_kernel(T* __restrict__ V, int R) {
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

constexpr int kChol32MaxR = 1024;

// Small ranks (R <= kSmemMaxR): the factorisation and the solves keep the lower
// triangle of the fp32 factor packed in shared memory (row i at i (i + 1) / 2).
constexpr int kSmemMaxR = 288;

__host__ __device__ __forceinline__ int tri(int i) { return i * (i + 1) / 2; }

// One CTA factors V (fp32, only the lower triangle read) in shared memory in
// 32-column panels: warp 0 factors the diagonal block in registers (lane i holds
// row i), every thread forward-substitutes one row of the panel below it, and the
// trailing lower triangle is updated in 4 x 4 register blocks from the panel.
// Writes L (dense row-major: lower triangle and its mirror above) and
// dinv[j] = 1 / L[j][j]; *info = j + 1 for the first pivot that is not positive.
constexpr int kCholSmemThreads = 256;   // no register cap: the row arrays stay in registers
__global__ void __launch_bounds__(kCholSmemThreads, 1) chol_smem_kernel(const float* __restrict__ V, int R,
                                                            float* __restrict__ L, float* __restrict__ dinv,
                                                            int* __restrict__ info) {
    extern __shared__ float sm[];
    float* a = sm;                         // packed lower triangle, tri(R) floats
    float* panel = sm + tri(R);            // [R][33]
    __shared__ float l11[32][33];
    __shared__ float dv[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = warp; i < R; i += nw)
        for (int j = lane; j <= i; j += 32) a[tri(i) + j] = V[(int64_t)i * R + j];
    __syncthreads();
    for (int k0 = 0; k0 < R; k0 += 32) {
        const int nb = R - k0 < 32 ? R - k0 : 32;
        if (warp == 0) {
            float r[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) r[t] = (lane < nb && t <= lane) ? a[tri(k0 + lane) + k0 + t] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < nb) {
                    const float piv = __shfl_sync(0xffffffffu, r[j], j);
                    if (lane == 0 && !(piv > 0.f) && *info == 0) *info = k0 + j + 1;
                    const float d = sqrtf(piv), inv = 1.f / d;
                    if (lane == j) r[j] = d;
                    if (lane > j) r[j] *= inv;
                    if (lane == 0) dv[j] = inv;
#pragma unroll
                    for (int t = j + 1; t < 32; ++t) {
                        const float ltj = __shfl_sync(0xffffffffu, r[j], t);
                        if (t < nb && lane >= t) r[t] = fmaf(-r[j], ltj, r[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                l11[lane][t] = (t <= lane) ? r[t] : 0.f;
                if (lane < nb && t <= lane) a[tri(k0 + lane) + k0 + t] = r[t];
            }
            __syncwarp();
            if (lane < nb) dinv[k0 + lane] = dv[lane];
        }
        __syncthreads();
        const int rest = R - k0 - nb;
        for (int ii = tid; ii < rest; ii += blockDim.x) {
            const int i = k0 + nb + ii;
            float x[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) x[t] = t < nb ? a[tri(i) + k0 + t] : 0.f;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                if (t < nb) {
                    float v = x[t];
#pragma unroll
                    for (int u = 0; u < t; ++u) v = fmaf(-x[u], l11[t][u], v);
                    x[t] = v * dv[t];
                }
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                if (t < nb) a[tri(i) + k0 + t] = x[t];
                panel[ii * 33 + t] = x[t];
            }
        }
        __syncthreads();
        const int nblk = (rest + 3) / 4;
        const int pairs = nblk * (nblk + 1) / 2;
        for (int pq = tid; pq < pairs; pq += blockDim.x) {
            int bi = (int)((sqrtf(8.f * (float)pq + 1.f) - 1.f) * 0.5f);
            while (bi * (bi + 1) / 2 > pq) --bi;
            while ((bi + 1) * (bi + 2) / 2 <= pq) ++bi;
            const int bk = pq - bi * (bi + 1) / 2;
            float acc[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
            for (int t = 0; t < nb; ++t) {
                float pi[4], pk[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int ri = 4 * bi + u, rk = 4 * bk + u;
                    pi[u] = ri < rest ? panel[ri * 33 + t] : 0.f;
                    pk[u] = rk < rest ? panel[rk * 33 + t] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(pi[u], pk[v], acc[u][v]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int ri = 4 * bi + u, rk = 4 * bk + v;
                    if (ri < rest && rk <= ri) a[tri(k0 + nb + ri) + k0 + nb + rk] -= acc[u][v];
                }
        }
        __syncthreads();
    }
    for (int i = warp; i < R; i += nw)
        for (int j = lane; j < R; j += 32) L[(int64_t)i * R + j] = j <= i ? a[tri(i) + j] : a[tri(j) + i];
}

// Y(i, :) = B(i, :) (L L^T)^{-1} in fp32, one warp per row, 32 rows a CTA, the
// packed lower triangle of L staged in shared memory (L dense, lower part read).
// Blocks of 32 unknowns as in solve_kernel.  out32 / (add, out64) as in
// solve32_kernel.
__global__ void __launch_bounds__(1024, 1) solve_smem_kernel(const float* __restrict__ L,
                                                             const float* __restrict__ dinv, int R,
                                                             const float* __restrict__ B, int64_t I,
                                                             float* __restrict__ out32,
                                                             const float* __restrict__ add,
                                                             double* __restrict__ out64) {
    extern __shared__ float sm[];
    float* lp = sm;                        // packed lower triangle
    float* ds = sm + tri(R);               // the pivots' reciprocals (R)
    float* xs = ds + R;                    // [32 warps][R]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = warp; i < R; i += nw)
        for (int j = lane; j <= i; j += 32) lp[tri(i) + j] = L[(int64_t)i * R + j];
    for (int j = tid; j < R; j += blockDim.x) ds[j] = dinv[j];
    const int64_t row = (int64_t)blockIdx.x * nw + warp;
    float* x = xs + (int64_t)warp * R;
    if (row < I)
        for (int k = lane; k < R; k += 32) x[k] = B[row * R + k];
    __syncthreads();
    if (row >= I) return;
    for (int k0 = 0; k0 < R; k0 += 32) {
        const int k = k0 + lane;
        const bool live = k < R;
        float acc = live ? x[k] : 0.f;
        if (live) {
            const float* lk = lp + tri(k);
            for (int j = 0; j < k0; ++j) acc = fmaf(-lk[j], x[j], acc);
        }
        const int nb = R - k0 < 32 ? R - k0 : 32;
        for (int t = 0; t < nb; ++t) {
            const float yt = __shfl_sync(0xffffffffu, acc, t) * ds[k0 + t];
            if (lane == t)
                acc = yt;
            else if (lane > t && live)
                acc = fmaf(-lp[tri(k) + k0 + t], yt, acc);
        }
        if (live) x[k] = acc;
        __syncwarp();
    }
    for (int k0 = ((R - 1) / 32) * 32; k0 >= 0; k0 -= 32) {
        const int k = k0 + lane;
        const bool live = k < R;
        float acc = live ? x[k] : 0.f;
        if (live)
            for (int j = k0 + 32; j < R; ++j) acc = fmaf(-lp[tri(j) + k], x[j], acc);
        const int nb = R - k0 < 32 ? R - k0 : 32;
        for (int t = nb - 1; t >= 0; --t) {
            const float xt = __shfl_sync(0xffffffffu, acc, t) * ds[k0 + t];
            if (lane == t)
                acc = xt;
            else if (lane < t && live)
                acc = fmaf(-lp[tri(k0 + t) + k], xt, acc);
        }
        if (live) x[k] = acc;
        __syncwarp();
    }
    for (int k = lane; k < R; k += 32) {
        const int64_t e = row * R + k;
        if (out32 != nullptr) out32[e] = x[k];
        if (out64 != nullptr) out64[e] = (double)add[e] + (double)x[k];
    }
}

// Y(i, :) = B(i, :) (L L^T)^{-1} in fp32 with the fp32 Cholesky factor (its
// upper triangle mirrored).  One warp solves kSolveRows rows together, so every
// load of L serves kSolveRows independent chains; lane l owns unknown k0 + l of
// each row in blocks of 32 unknowns: the finished blocks' contributions are dot
// products (loads of L issued eight at a time ahead of the arithmetic), and
// within the block the unknowns are finished one by one and broadcast by
// shuffles.  out32 (if non-null) receives the fp32 result; out64 (if non-null)
// receives add + result in fp64.
constexpr int kSolveRows = 1;
__global__ void __launch_bounds__(32) solve32_kernel(const float* __restrict__ L, const float* __restrict__ dinv,
                                                     int R, const float* __restrict__ B, int64_t I,
                                                     float* __restrict__ out32, const float* __restrict__ add,
                                                     double* __restrict__ out64) {
    extern __shared__ float xs32[];   // [kSolveRows][R], then the staged block of L [R][33]
    constexpr int NR = kSolveRows;
    const int lane = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * NR;
    float* x = xs32;
    float* lst = xs32 + NR * R;
    // lst[j][l] = L[j][k0 + l] for the rows j the block's dot products need (all
    // loads issued before any use)
    auto stage = [&](int j0, int j1, int k0) {
        const bool in = k0 + lane < R;
        int j = j0;
        for (; j + 8 <= j1; j += 8) {   // eight loads in flight before their stores
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = in ? L[(int64_t)(j + q) * R + k0 + lane] : 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) lst[(j + q) * 33 + lane] = v[q];
        }
        for (; j < j1; ++j) lst[j * 33 + lane] = in ? L[(int64_t)j * R + k0 + lane] : 0.f;
        __syncwarp();
    };
    for (int u = 0; u < NR; ++u)
        for (int k = lane; k < R; k += 32) x[u * R + k] = row0 + u < I ? B[(row0 + u) * R + k] : 0.f;
    __syncwarp();
    // L y = b
    for (int k0 = 0; k0 < R; k0 += 32) {
        const int k = k0 + lane;
        const bool live = k < R;
        float acc[NR];
#pragma unroll
        for (int u = 0; u < NR; ++u) acc[u] = live ? x[u * R + k] : 0.f;
        stage(0, k0, k0);   // upper mirror: L[j][k] = L[k][j]
        if (live)
            for (int j = 0; j < k0; ++j) {
                const float l = lst[j * 33 + lane];
#pragma unroll
                for (int u = 0; u < NR; ++u) acc[u] = fmaf(-l, x[u * R + j], acc[u]);
            }
        __syncwarp();
        const int nb = R - k0 < 32 ? R - k0 : 32;
        float lb[32], db[32];   // this lane's row of the diagonal block, and the pivots' reciprocals
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            lb[t] = (live && t < nb && lane > t) ? L[(int64_t)k * R + k0 + t] : 0.f;
            db[t] = t < nb ? dinv[k0 + t] : 0.f;
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            if (t < nb) {
#pragma unroll
                for (int u = 0; u < NR; ++u) {
                    const float yt = __shfl_sync(0xffffffffu, acc[u], t) * db[t];
                    if (lane == t)
                        acc[u] = yt;
                    else if (lane > t)
                        acc[u] = fmaf(-lb[t], yt, acc[u]);
                }
            }
        }
        if (live)
#pragma unroll
            for (int u = 0; u < NR; ++u) x[u * R + k] = acc[u];
        __syncwarp();
    }
    // L^T x = y
    for (int k0 = ((R - 1) / 32) * 32; k0 >= 0; k0 -= 32) {
        const int k = k0 + lane;
        const bool live = k < R;
        float acc[NR];
#pragma unroll
        for (int u = 0; u < NR; ++u) acc[u] = live ? x[u * R + k] : 0.f;
        stage(k0 + 32 < R ? k0 + 32 : R, R, k0);
        if (live)
            for (int j = k0 + 32; j < R; ++j) {
                const float l = lst[j * 33 + lane];
#pragma unroll
                for (int u = 0; u < NR; ++u) acc[u] = fmaf(-l, x[u * R + j], acc[u]);
            }
        __syncwarp();
        const int nb = R - k0 < 32 ? R - k0 : 32;
        float lb[32], db[32];   // column k of the diagonal block (L[k0 + t][k]), and the reciprocals
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            lb[t] = (live && t < nb && lane < t) ? L[(int64_t)(k0 + t) * R + k] : 0.f;
            db[t] = t < nb ? dinv[k0 + t] : 0.f;
        }
#pragma unroll
        for (int t = 31; t >= 0; --t) {
            if (t < nb) {
#pragma unroll
                for (int u = 0; u < NR; ++u) {
                    const float xt = __shfl_sync(0xffffffffu, acc[u], t) * db[t];
                    if (lane == t)
                        acc[u] = xt;
                    else if (lane < t)
                        acc[u] = fmaf(-lb[t], xt, acc[u]);
                }
            }
        }
        if (live)
#pragma unroll
            for (int u = 0; u < NR; ++u) x[u * R + k] = acc[u];
        __syncwarp();
    }
    for (int u = 0; u < NR; ++u) {
        if (row0 + u >= I) break;
        for (int k = lane; k < R; k += 32) {
            const int64_t e = (row0 + u) * R + k;
            if (out32 != nullptr) out32[e] = x[u * R + k];
            if (out64 != nullptr) out64[e] = (double)add[e] + (double)x[u * R + k];
        }
    }
}

// V (fp64) as two fp32 words, vhi = fl32(V) and vlo = fl32(V - vhi), which hold
// it to about 2^-48 relative
// (L receives a copy of vhi: the working matrix of the fp32 factorisation)
__global__ void split_v_kernel(const double* __restrict__ V, int64_t n, float* __restrict__ vhi,
                               float* __restrict__ vlo, float* __restrict__ L) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        const double v = V[e];
        const float h = (float)v;
        vhi[e] = h;
        vlo[e] = (float)(v - (double)h);
        L[e] = h;
    }
}

// Res = M - X V (I x R) with V = vhi + vlo: each product x vhi split exactly
// (fma), summed with compensation; x vlo and the product errors summed plainly.
// kResRows rows and kResCols columns a block (one column a thread).
constexpr int kResRows = 2, kResCols = 128;
__global__ void __launch_bounds__(kResCols) residual_kernel(const float* __restrict__ M, const float* __restrict__ X,
                                                       const float* __restrict__ vhi_m, const float* __restrict__ vlo_m,
                                                       int64_t I, int R, float* __restrict__ Res) {
    extern __shared__ float xr[];   // [kResRows][R]
    const int64_t i0 = (int64_t)blockIdx.y * kResRows;
    for (int t = threadIdx.x; t < kResRows * R; t += blockDim.x) {
        const int u = t / R;
        xr[t] = i0 + u < I ? X[(i0 + u) * R + (t - u * R)] : 0.f;
    }
    __syncthreads();
    {
        const int j = blockIdx.x * kResCols + threadIdx.x;
        if (j >= R) return;
        float s[kResRows], c[kResRows], sm[kResRows];
#pragma unroll
        for (int u = 0; u < kResRows; ++u) s[u] = c[u] = sm[u] = 0.f;
        int k = 0;
        for (; k + 8 <= R; k += 8) {   // eight rows of V in flight
            float vh[8], vl[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                vh[q] = vhi_m[(int64_t)(k + q) * R + j];
                vl[q] = vlo_m[(int64_t)(k + q) * R + j];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
#pragma unroll
                for (int u = 0; u < kResRows; ++u) {
                    const float x = xr[u * R + k + q];
                    const float p = x * vh[q];
                    sm[u] += fmaf(x, vh[q], -p) + x * vl[q];
                    neumaier(s[u], c[u], p);
                }
        }
        for (; k < R; ++k) {
            const float vhi = vhi_m[(int64_t)k * R + j], vlo = vlo_m[(int64_t)k * R + j];
#pragma unroll
            for (int u = 0; u < kResRows; ++u) {
                const float x = xr[u * R + k];
                const float p = x * vhi;
                sm[u] += fmaf(x, vhi, -p) + x * vlo;
                neumaier(s[u], c[u], p);
            }
        }
#pragma unroll
        for (int u = 0; u < kResRows; ++u)
            if (i0 + u < I) {
                const int64_t e = (i0 + u) * R + j;
                Res[e] = (M[e] - s[u]) - (c[u] + sm[u]);
            }
    }
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

// The fit over many blocks: block b takes rows r = b, b + B, ... of H for
// lambda^T H lambda and rows i = b, b + B, ... of M and A for <Y, X>, and writes
// its two partial sums; fit_final_kernel adds them in block order.
constexpr int kFitBlocks = 128;
__global__ void __launch_bounds__(256) fit_partial_kernel(const double* __restrict__ H, const float* __restrict__ lam,
                                                          const float* __restrict__ M, const float* __restrict__ A,
                                                          int64_t I, int R, double* __restrict__ part) {
    __shared__ double sh[8];
    double x2 = 0.0, in = 0.0;
    for (int r = blockIdx.x; r < R; r += gridDim.x) {
        double t = 0.0;
        for (int c = threadIdx.x; c < R; c += blockDim.x) t += H[(int64_t)r * R + c] * (double)lam[c];
        x2 += (double)lam[r] * t;
    }
    for (int64_t i = blockIdx.x; i < I; i += gridDim.x)
        for (int c = threadIdx.x; c < R; c += blockDim.x)
            in += (double)lam[c] * ((double)M[i * R + c] * (double)A[i * R + c]);
    x2 = block_sum(x2, sh);
    in = block_sum(in, sh);
    if (threadIdx.x == 0) {
        part[2 * blockIdx.x] = x2;
        part[2 * blockIdx.x + 1] = in;
    }
}

__global__ void fit_final_kernel(const double* __restrict__ part, int nb, const double* __restrict__ norm_y2,
                                 const int* __restrict__ info, double* __restrict__ fit) {
    if (threadIdx.x != 0) return;
    double x2 = 0.0, in = 0.0;
    for (int b = 0; b < nb; ++b) {
        x2 += part[2 * b];
        in += part[2 * b + 1];
    }
    const double y2 = *norm_y2;
    const double res2 = y2 + x2 - 2.0 * in;
    *fit = (*info != 0) ? __longlong_as_double(0x7ff8000000000000ll) : 1.0 - sqrt(res2 > 0.0 ? res2 : 0.0) / sqrt(y2);
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

template <typename T>
cudaError_t blocked_cholesky(T* V, int R, int* info, T* dinv, cudaStream_t s) {
    for (int k0 = 0; k0 < R; k0 += kChNB) {
        const int nb = R - k0 < kChNB ? R - k0 : kChNB;
        chol_diag_kernel<T><<<1, 256, 0, s>>>(V, R, k0, nb, info, dinv);
        const int rest = R - k0 - nb;
        if (rest > 0) {
            // panel rows spread over CTAs of 32 threads, so that short panels still
            // use several SMs
            chol_panel_kernel<T><<<(unsigned)((rest + 31) / 32), 32, 0, s>>>(V, R, k0, nb, dinv);
            const unsigned nt = (unsigned)((rest + kChNB - 1) / kChNB);
            chol_update_kernel<T><<<dim3(nt, nt), 256, 0, s>>>(V, R, k0, nb);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t cpals_cholesky(double* V, int R, int* info, double* dinv, cudaStream_t s) {
    return blocked_cholesky<double>(V, R, info, dinv, s);
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
        mirror_lower_kernel<double><<<(unsigned)blocks, 256, 0, s>>>(L, R);
    }
    solve_kernel<<<(unsigned)((I + warps - 1) / warps), warps * 32, smem, s>>>(L, dinv, R, M, I, X);
    return cudaGetLastError();
}

int cpals_mixed_max_rank() { return kChol32MaxR; }

int cpals_mixed_launches(int R) { return R <= kSmemMaxR ? 5 : 5 + cpals_cholesky_launches(R); }

cudaError_t cpals_solve_mixed(const double* V, int R, const float* M, int64_t I, double* X, float* vhi, float* vlo,
                              float* L, float* dinv, float* x0, float* res, int* info, cudaStream_t s) {
    if (R > kChol32MaxR) return cudaErrorInvalidValue;
    const int64_t n = (int64_t)R * R;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    split_v_kernel<<<(unsigned)blocks, 256, 0, s>>>(V, n, vhi, vlo, L);
    cudaError_t e;
    if (R <= kSmemMaxR) {
        // the factor and the solves with the triangle in shared memory
        const size_t csm = ((size_t)tri(R) + (size_t)R * 33) * sizeof(float);
        e = cudaFuncSetAttribute(chol_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm);
        if (e != cudaSuccess) return e;
        chol_smem_kernel<<<1, kCholSmemThreads, csm, s>>>(vhi, R, L, dinv, info);
        const size_t ssm = ((size_t)tri(R) + (size_t)33 * R) * sizeof(float);
        e = cudaFuncSetAttribute(solve_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
        if (e != cudaSuccess) return e;
        const unsigned sb = (unsigned)((I + 31) / 32);
        solve_smem_kernel<<<sb, 1024, ssm, s>>>(L, dinv, R, M, I, x0, nullptr, nullptr);
        const size_t rsm = (size_t)kResRows * R * sizeof(float);
        e = cudaFuncSetAttribute(residual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm);
        if (e != cudaSuccess) return e;
        residual_kernel<<<dim3((unsigned)((R + kResCols - 1) / kResCols), (unsigned)((I + kResRows - 1) / kResRows)),
                          kResCols, rsm, s>>>(M, x0, vhi, vlo, I, R, res);
        solve_smem_kernel<<<sb, 1024, ssm, s>>>(L, dinv, R, res, I, nullptr, x0, X);
        return cudaGetLastError();
    }
    e = blocked_cholesky<float>(L, R, info, dinv, s);
    if (e != cudaSuccess) return e;
    mirror_lower_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(L, R);
    const size_t ssm = ((size_t)kSolveRows * R + (size_t)R * 33) * sizeof(float);
    e = cudaFuncSetAttribute(solve32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return e;
    const unsigned sblocks = (unsigned)((I + kSolveRows - 1) / kSolveRows);
    solve32_kernel<<<sblocks, 32, ssm, s>>>(L, dinv, R, M, I, x0, nullptr, nullptr);
    const size_t rsm = (size_t)kResRows * R * sizeof(float);
    e = cudaFuncSetAttribute(residual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm);
    if (e != cudaSuccess) return e;
    residual_kernel<<<dim3((unsigned)((R + kResCols - 1) / kResCols), (unsigned)((I + kResRows - 1) / kResRows)),
                      kResCols, rsm, s>>>(M, x0, vhi, vlo, I, R, res);
    solve32_kernel<<<sblocks, 32, ssm, s>>>(L, dinv, R, res, I, nullptr, x0, X);
    return cudaGetLastError();
}

cudaError_t cpals_normalize(const double* X, int64_t I, int R, float* A, float* lam, cudaStream_t s) {
    normalize_kernel<<<(unsigned)((R + 31) / 32), 1024, 0, s>>>(X, I, R, A, lam);
    return cudaGetLastError();
}

cudaError_t cpals_fit(const double* H, const float* lam, const float* M, const float* A, int64_t I, int R,
                      const double* norm_y2, const int* info, double* fit, double* part, cudaStream_t s) {
    fit_partial_kernel<<<kFitBlocks, 256, 0, s>>>(H, lam, M, A, I, R, part);
    fit_final_kernel<<<1, 32, 0, s>>>(part, kFitBlocks, norm_y2, info, fit);
    return cudaGetLastError();
}

size_t cpals_sumsq_scratch_bytes() {
    return (kSqBlocks > 2 * kFitBlocks ? kSqBlocks : 2 * kFitBlocks) * sizeof(double);
}

cudaError_t cpals_sum_squares(const float* Y, int64_t n, double* part, double* out, cudaStream_t s) {
    sumsq_partial_kernel<<<kSqBlocks, 256, 0, s>>>(Y, n, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sumsq_final_kernel<<<1, 256, 0, s>>>(part, kSqBlocks, out);
    return cudaGetLastError();
}

}  // namespace mk
