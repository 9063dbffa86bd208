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

// V = Hadamard product of G[m] over m != skip (skip < 0: all d); with vhi
// non-null also V as two fp32 words, vhi = fl32(V) and vlo = fl32(V - vhi),
// which hold it to about 2^-48 relative
__global__ void hadamard_kernel(const double* __restrict__ G, int d, int skip, int R, double* __restrict__ V,
                                float* __restrict__ vhi, float* __restrict__ vlo) {
    const int64_t n = (int64_t)R * R;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        double v = 1.0;
        for (int m = 0; m < d; ++m)
            if (m != skip) v *= G[m * n + e];
        V[e] = v;
        if (vhi != nullptr) {
            const float h = (float)v;
            vhi[e] = h;
            vlo[e] = (float)(v - (double)h);
        }
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

// Small ranks (R <= kSmemMaxR) take the single-launch factorisation and the
// multi-CTA row solves below; larger ranks the blocked multi-launch factor.
constexpr int kSmemMaxR = 288;
constexpr int kChB = 32;   // panel width = diagonal block size

__host__ __device__ __forceinline__ int tri(int i) { return i * (i + 1) / 2; }
__host__ __device__ __forceinline__ int round4(int x) { return (x + 3) & ~3; }

// The fp32 factor L L^T of vhi = fl32(V) by one CTA, right-looking in 32-column
// panels with the packed lower triangle in shared memory:
//   A. warp 0 factors the diagonal block in registers (lane i holds row i; the
//      pivot's 1 / sqrt from rsqrtf refined by one Newton-Raphson step, no
//      division) and inverts it (lane c computes column c of the inverse);
//   B. four threads a row of the panel below (one warp, eight rows): L21 =
//      A21 L11^{-T} as a product with the inverse (no substitution chain),
//      kept transposed in shared memory beside the triangle;
//   C. the trailing lower triangle is updated in 4 x 4 register blocks from
//      the transposed panel (16-byte loads).
// Outputs: Lm (R x R: L in the lower triangle, its mirror above), Dm (the
// inverse of every diagonal block, 32 x 32 row-major, zero above the diagonal
// and outside the block), dinv[j] = 1 / L[j][j]; *info = j + 1 for the first
// pivot that is not positive (the factor then holds NaN from there on).
constexpr int kChol2Threads = 512;   // 128 registers a thread: no spills

size_t chol2_smem_bytes(int R) { return ((size_t)round4(tri(R)) + (size_t)kChB * round4(R)) * sizeof(float); }

__device__ __forceinline__ void cp_async4(float* smem, const float* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async16(float* smem, const float* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__global__ void __launch_bounds__(kChol2Threads, 1)
    chol2_kernel(const float* __restrict__ vhi, int R, float* __restrict__ Lm, float* __restrict__ Dm,
                 float* __restrict__ dinv, int* __restrict__ info) {
    extern __shared__ __align__(16) float sm[];
    const int Rp = round4(R);
    float* a = sm;                       // packed lower triangle (row i at tri(i))
    float* P = sm + round4(tri(R));      // transposed panel [32][Rp]
    __shared__ __align__(16) float l11[kChB][kChB + 4];    // rows 16-byte aligned
    __shared__ __align__(16) float linv[kChB][kChB + 4];
    __shared__ float dvs[kChB];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = warp; i < R; i += kChol2Threads / 32)
        for (int j = lane; j <= i; j += 32) cp_async4(a + tri(i) + j, vhi + (int64_t)i * R + j);
    cp_async_wait_all();
    __syncthreads();
    int first_bad = -1;   // warp 0: first pivot that is not positive
    for (int k0 = 0; k0 < R; k0 += kChB) {
        const int nb = R - k0 < kChB ? R - k0 : kChB;
        const int r0 = k0 + nb, rest = R - r0;
        if (warp == 0) {
            // A. the diagonal block
            float r[kChB];
#pragma unroll
            for (int t = 0; t < kChB; ++t) r[t] = (lane < nb && t <= lane) ? a[tri(k0 + lane) + k0 + t] : 0.f;
            float dl = 0.f;   // 1 / L[k0 + lane][k0 + lane]
            // Every lane updates all of its row unconditionally: what lands above
            // the diagonal (t > lane) is never read by the lower part (pivots come
            // from the diagonal, shuffled column entries from lanes below) and is
            // masked when the block is stored; no per-lane selects in the loop,
            // which measured several times faster.
#pragma unroll
            for (int j = 0; j < kChB; ++j) {
                if (j < nb) {
                    const float piv = __shfl_sync(0xffffffffu, r[j], j);
                    first_bad = (first_bad < 0 && !(piv > 0.f)) ? k0 + j : first_bad;
                    float inv = rsqrtf(piv);
                    inv = inv * fmaf(-0.5f * piv * inv, inv, 1.5f);   // Newton-Raphson step for 1 / sqrt
                    dl = lane == j ? inv : dl;
                    r[j] = lane == j ? piv * inv : r[j] * inv;
#pragma unroll
                    for (int t = j + 1; t < kChB; ++t) r[t] = fmaf(-r[j], __shfl_sync(0xffffffffu, r[j], t), r[t]);
                }
            }
#pragma unroll
            for (int t = 0; t < kChB; ++t) {
                l11[lane][t] = t <= lane ? r[t] : 0.f;
                if (lane < nb && t <= lane) a[tri(k0 + lane) + k0 + t] = r[t];
            }
            if (lane < nb) dinv[k0 + lane] = dl;
            dvs[lane] = dl;
            __syncwarp();
            // inverse of the block, lane c = column c: L z = e_c by substitution,
            // z[i] = (delta_ic - sum_{k<i} L[i][k] z[k]) / L[i][i] (zero for i < c)
            float z[kChB];
#pragma unroll
            for (int i = 0; i < kChB; ++i) {
                float s0 = i == lane ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
                for (int k = 0; k + 4 <= i; k += 4) {
                    const float4 l = *reinterpret_cast<const float4*>(&l11[i][k]);
                    s0 = fmaf(-l.x, z[k], s0);
                    s1 = fmaf(-l.y, z[k + 1], s1);
                    s0 = fmaf(-l.z, z[k + 2], s0);
                    s1 = fmaf(-l.w, z[k + 3], s1);
                }
#pragma unroll
                for (int k = i & ~3; k < i; ++k) s0 = fmaf(-l11[i][k], z[k], s0);
                z[i] = (s0 + s1) * dvs[i];
            }
            float* dblk = Dm + (int64_t)(k0 / kChB) * kChB * kChB;
#pragma unroll
            for (int i = 0; i < kChB; ++i) {
                linv[i][lane] = z[i];   // z[i] = 0 above the diagonal
                dblk[i * kChB + lane] = z[i];
            }
        }
        __syncthreads();   // linv ready
        // B. the panel below the block: item (row ii, tq) forms L21[ii][t] for
        // t = tq, tq + 4, ..., tq + 28; a row's four items are in one warp, so a
        // warp barrier orders its reads before its in-place writes
        const int items = (4 * round4(rest) + 31) & ~31;   // whole warps: the loop is warp-uniform
        for (int it = tid; it < items; it += kChol2Threads) {
            const int ii = it >> 2, tq = it & 3;
            const bool act = ii < rest;
            float x[kChB];
            if (act) {
                const float* arow = a + tri(r0 + ii) + k0;
#pragma unroll
                for (int u = 0; u < kChB; ++u) x[u] = u < nb ? arow[u] : 0.f;
            }
            __syncwarp();
            if (act) {
                float* arow = a + tri(r0 + ii) + k0;
#pragma unroll
                for (int c = 0; c < kChB / 4; ++c) {
                    const int t = tq + 4 * c;
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int u = 0; u < kChB; u += 4) {
                        if (u <= 4 * c + 3) {   // linv[t][u..u+3] is zero beyond t
                            const float4 l = *reinterpret_cast<const float4*>(&linv[t][u]);
                            s0 = fmaf(x[u], l.x, s0);
                            s1 = fmaf(x[u + 1], l.y, s1);
                            s0 = fmaf(x[u + 2], l.z, s0);
                            s1 = fmaf(x[u + 3], l.w, s1);
                        }
                    }
                    const float v = s0 + s1;
                    P[t * Rp + ii] = v;
                    if (t < nb) arow[t] = v;
                }
            } else if (ii < round4(rest)) {
#pragma unroll
                for (int c = 0; c < kChB / 4; ++c) P[(tq + 4 * c) * Rp + ii] = 0.f;
            }
        }
        __syncthreads();
        // C. trailing update: a[r0 + i][r0 + k] -= sum_t L21[i][t] L21[k][t], k <= i
        const int nblk = (rest + 3) / 4;
        const int pairs = nblk * (nblk + 1) / 2;
        for (int pq = tid; pq < pairs; pq += blockDim.x) {
            int bi = (int)((sqrtf(8.f * (float)pq + 1.f) - 1.f) * 0.5f);
            while (tri(bi) > pq) --bi;
            while (tri(bi + 1) <= pq) ++bi;
            const int bk = pq - tri(bi);
            float acc[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
            for (int t = 0; t < nb; ++t) {
                const float4 pi = *reinterpret_cast<const float4*>(P + t * Rp + 4 * bi);
                const float4 pk = *reinterpret_cast<const float4*>(P + t * Rp + 4 * bk);
                const float vi[4] = {pi.x, pi.y, pi.z, pi.w}, vk[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(vi[u], vk[v], acc[u][v]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int ri = 4 * bi + u, rk = 4 * bk + v;
                    if (ri < rest && rk <= ri) a[tri(r0 + ri) + r0 + rk] -= acc[u][v];
                }
        }
        __syncthreads();
    }
    if (warp == 0 && lane == 0 && first_bad >= 0 && *info == 0) *info = first_bad + 1;
    for (int i = warp; i < R; i += kChol2Threads / 32)
        for (int j = lane; j < R; j += 32) Lm[(int64_t)i * R + j] = j <= i ? a[tri(i) + j] : a[tri(j) + i];
}

// X(i, :) = B(i, :) (L L^T)^{-1} in fp32 for R <= kSmemMaxR: y L^T = b, then
// x L = y, row by row in blocks of 32 unknowns (lane l owns unknown k0 + l).
// The finished blocks enter as dot products with columns of the factor, the
// block itself as the product with the inverse of its diagonal block, so no
// step waits on a substitution chain.  Each CTA stages the parts of the
// mirrored factor Lm that a pass reads (the strip above every diagonal block
// for the forward pass, below it for the backward pass) and Dm (rows padded to
// 33 floats: read along rows and along columns without bank conflicts) in
// shared memory with asynchronous copies; kSv2Warps warps of kSv2Rows rows
// each.
// out32 (if non-null) receives the result; out64 (if non-null) add + result in
// fp64.
constexpr int kSv2Warps = 4, kSv2Rows = 1;

__host__ __device__ __forceinline__ int64_t sv2_strip_floats(int R) {
    const int nb = (R + kChB - 1) / kChB;
    int64_t f = 0, b = 0;
    for (int kb = 0; kb < nb; ++kb) {
        f += (int64_t)kChB * kb * kChB;
        const int rows = R - kChB * (kb + 1);
        b += rows > 0 ? (int64_t)rows * kChB : 0;
    }
    return f > b ? f : b;
}
size_t sv2_smem_bytes(int R) {
    const int nb = (R + kChB - 1) / kChB;
    return ((size_t)sv2_strip_floats(R) + (size_t)nb * kChB * (kChB + 1) + (size_t)kSv2Warps * kSv2Rows * nb * kChB) *
           sizeof(float);
}

template <bool VEC>   // VEC: R % 4 == 0 and Lm 16-byte aligned (16-byte copies)
__global__ void __launch_bounds__(kSv2Warps * 32)
    solve2_kernel(const float* __restrict__ Lm, const float* __restrict__ Dm, int R, const float* __restrict__ B,
                  int64_t I, float* __restrict__ out32, const float* __restrict__ add, double* __restrict__ out64) {
    extern __shared__ __align__(16) float sm[];
    constexpr int NR = kSv2Rows;
    const int nblk = (R + kChB - 1) / kChB, Rb = nblk * kChB;
    float* strip = sm;
    float* dsm = sm + sv2_strip_floats(R);                 // [nblk][32][33]
    float* ys = dsm + (int64_t)nblk * kChB * (kChB + 1);    // [warps][NR][Rb]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float* y = ys + (int64_t)warp * NR * Rb;
    const int64_t row0 = ((int64_t)blockIdx.x * kSv2Warps + warp) * NR;

    // stage rows [j0, j1) of columns [k0, k0 + 32) of Lm at dst (32 floats a
    // row; columns at or beyond R read as 0)
    auto stage = [&](float* dst, int j0, int j1, int k0) {
        const int n = (j1 - j0) * (VEC ? kChB / 4 : kChB);
        for (int e = tid; e < n; e += blockDim.x) {
            if (VEC) {
                const int j = j0 + e / (kChB / 4), c = 4 * (e % (kChB / 4));
                float* d = dst + (int64_t)(j - j0) * kChB + c;
                if (k0 + c < R)
                    cp_async16(d, Lm + (int64_t)j * R + k0 + c);
                else
                    *reinterpret_cast<float4*>(d) = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                const int j = j0 + e / kChB, c = e % kChB;
                float* d = dst + (int64_t)(j - j0) * kChB + c;
                if (k0 + c < R)
                    cp_async4(d, Lm + (int64_t)j * R + k0 + c);
                else
                    *d = 0.f;
            }
        }
    };
    // forward strips: block kb at 1024 * kb (kb - 1) / 2 floats, rows j < 32 kb
    for (int kb = 1; kb < nblk; ++kb) stage(strip + (int64_t)kChB * kChB * kb * (kb - 1) / 2, 0, kChB * kb, kChB * kb);
    for (int e = tid; e < nblk * kChB * kChB; e += blockDim.x) cp_async4(dsm + e + e / kChB, Dm + e);
    for (int u = 0; u < NR; ++u)
        for (int k = lane; k < Rb; k += 32) y[u * Rb + k] = (row0 + u < I && k < R) ? B[(row0 + u) * R + k] : 0.f;
    cp_async_wait_all();
    __syncthreads();

    // y L^T = b
    for (int kb = 0; kb < nblk; ++kb) {
        const int k0 = kb * kChB, k = k0 + lane;
        const float* s = strip + (int64_t)kChB * kChB * kb * (kb - 1) / 2 + lane;   // s[j * 32] = L[k][j]
        float acc[NR], acc2[NR];
#pragma unroll
        for (int u = 0; u < NR; ++u) {
            acc[u] = y[u * Rb + k];
            acc2[u] = 0.f;
        }
#pragma unroll 4
        for (int j = 0; j < k0; j += 4) {
            const float l0 = s[(j + 0) * kChB], l1 = s[(j + 1) * kChB], l2 = s[(j + 2) * kChB],
                        l3 = s[(j + 3) * kChB];
#pragma unroll
            for (int u = 0; u < NR; ++u) {
                const float4 yv = *reinterpret_cast<const float4*>(y + u * Rb + j);
                acc[u] = fmaf(-l0, yv.x, acc[u]);
                acc2[u] = fmaf(-l1, yv.y, acc2[u]);
                acc[u] = fmaf(-l2, yv.z, acc[u]);
                acc2[u] = fmaf(-l3, yv.w, acc2[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < NR; ++u) acc[u] += acc2[u];
        const float* drow = dsm + kb * kChB * (kChB + 1) + lane * (kChB + 1);   // drow[t] = Linv[lane][t]
        float out[NR];
#pragma unroll
        for (int u = 0; u < NR; ++u) out[u] = 0.f;
#pragma unroll
        for (int t = 0; t < kChB; ++t) {
            const float dv = drow[t];   // zero for t > lane
#pragma unroll
            for (int u = 0; u < NR; ++u) out[u] = fmaf(dv, __shfl_sync(0xffffffffu, acc[u], t), out[u]);
        }
#pragma unroll
        for (int u = 0; u < NR; ++u) y[u * Rb + k] = out[u];   // 0 beyond R: Dm is zero there
        __syncwarp();
    }
    __syncthreads();   // every warp done with the forward strips
    // backward strips: block kb holds rows j >= 32 (kb + 1)
    {
        int64_t off = 0;
        for (int kb = 0; kb < nblk; ++kb) {
            const int j0 = kChB * (kb + 1);
            if (j0 < R) {
                stage(strip + off, j0, R, kChB * kb);
                off += (int64_t)(R - j0) * kChB;
            }
        }
    }
    cp_async_wait_all();
    __syncthreads();
    // x L = y
    int64_t off_end = 0;
    for (int kb = 0; kb < nblk; ++kb) {
        const int j0 = kChB * (kb + 1);
        if (j0 < R) off_end += (int64_t)(R - j0) * kChB;
    }
    for (int kb = nblk - 1; kb >= 0; --kb) {
        const int k0 = kb * kChB, k = k0 + lane, j0 = k0 + kChB;
        const int rows = j0 < R ? R - j0 : 0;
        off_end -= (int64_t)rows * kChB;
        const float* s = strip + off_end + lane;   // s[(j - j0) * 32] = L[j][k]
        float acc[NR], acc2[NR];
#pragma unroll
        for (int u = 0; u < NR; ++u) {
            acc[u] = y[u * Rb + k];
            acc2[u] = 0.f;
        }
        int j = 0;
#pragma unroll 4
        for (; j + 4 <= rows; j += 4) {
            const float l0 = s[(j + 0) * kChB], l1 = s[(j + 1) * kChB], l2 = s[(j + 2) * kChB],
                        l3 = s[(j + 3) * kChB];
#pragma unroll
            for (int u = 0; u < NR; ++u) {
                const float4 yv = *reinterpret_cast<const float4*>(y + u * Rb + j0 + j);
                acc[u] = fmaf(-l0, yv.x, acc[u]);
                acc2[u] = fmaf(-l1, yv.y, acc2[u]);
                acc[u] = fmaf(-l2, yv.z, acc[u]);
                acc2[u] = fmaf(-l3, yv.w, acc2[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < NR; ++u) acc[u] += acc2[u];
        for (; j < rows; ++j) {
            const float l = s[j * kChB];
#pragma unroll
            for (int u = 0; u < NR; ++u) acc[u] = fmaf(-l, y[u * Rb + j0 + j], acc[u]);
        }
        const float* dcol = dsm + kb * kChB * (kChB + 1) + lane;   // dcol[t * 33] = Linv[t][lane]
        float out[NR];
#pragma unroll
        for (int u = 0; u < NR; ++u) out[u] = 0.f;
#pragma unroll
        for (int t = 0; t < kChB; ++t) {
            const float dv = dcol[t * (kChB + 1)];   // zero for t < lane
#pragma unroll
            for (int u = 0; u < NR; ++u) out[u] = fmaf(dv, __shfl_sync(0xffffffffu, acc[u], t), out[u]);
        }
#pragma unroll
        for (int u = 0; u < NR; ++u) y[u * Rb + k] = out[u];
        __syncwarp();
    }
    for (int u = 0; u < NR; ++u) {
        if (row0 + u >= I) break;
        for (int k = lane; k < R; k += 32) {
            const int64_t e = (row0 + u) * R + k;
            if (out32 != nullptr) out32[e] = y[u * Rb + k];
            if (out64 != nullptr) out64[e] = (double)add[e] + (double)y[u * Rb + k];
        }
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
// A CTA takes a tile of kRes2Rows rows x kRes2Cols columns: the rows of X staged
// in shared memory once, V's column block streamed through shared memory in
// chunks of kResKC rows with asynchronous copies (double-buffered); a thread
// takes one row and four adjacent columns.
constexpr int kRes2Rows = 8, kRes2Cols = 64, kResKC = 32;

size_t res2_smem_bytes(int R) {
    return ((size_t)kRes2Rows * (R + 1) + (size_t)2 * 2 * kResKC * kRes2Cols) * sizeof(float);
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

template <bool VEC>   // VEC: R % 4 == 0 and vhi, vlo 16-byte aligned
__global__ void __launch_bounds__(kRes2Rows * kRes2Cols / 4)
    residual2_kernel(const float* __restrict__ M, const float* __restrict__ X, const float* __restrict__ vhi_m,
                     const float* __restrict__ vlo_m, int64_t I, int R, float* __restrict__ Res) {
    extern __shared__ __align__(16) float rs[];
    float* vb = rs;                                          // [2 buffers][hi|lo][kResKC][kRes2Cols]
    float* xr = rs + 2 * 2 * kResKC * kRes2Cols;             // [kRes2Rows][R + 1]
    constexpr int kThreads = kRes2Rows * kRes2Cols / 4;
    const int stride = R + 1;
    const int tid = threadIdx.x;
    const int64_t i0 = (int64_t)blockIdx.y * kRes2Rows;
    const int jb = blockIdx.x * kRes2Cols;
    // chunk c of V's column block into buffer b (columns at or beyond R, rows at
    // or beyond R read as 0)
    auto stage = [&](int c, int b) {
        float* dh = vb + (size_t)b * 2 * kResKC * kRes2Cols;
        float* dl = dh + kResKC * kRes2Cols;
        const int k0 = c * kResKC;
        if (VEC) {
            for (int e = tid; e < kResKC * kRes2Cols / 4; e += kThreads) {
                const int kk = e / (kRes2Cols / 4), cc = 4 * (e % (kRes2Cols / 4));
                const int k = k0 + kk, j = jb + cc;
                float* h = dh + kk * kRes2Cols + cc;
                float* l = dl + kk * kRes2Cols + cc;
                if (k < R && j < R) {
                    cp_async16(h, vhi_m + (int64_t)k * R + j);
                    cp_async16(l, vlo_m + (int64_t)k * R + j);
                } else {
                    *reinterpret_cast<float4*>(h) = make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4*>(l) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        } else {
            for (int e = tid; e < kResKC * kRes2Cols; e += kThreads) {
                const int kk = e / kRes2Cols, cc = e % kRes2Cols;
                const int k = k0 + kk, j = jb + cc;
                if (k < R && j < R) {
                    cp_async4(dh + e, vhi_m + (int64_t)k * R + j);
                    cp_async4(dl + e, vlo_m + (int64_t)k * R + j);
                } else {
                    dh[e] = 0.f;
                    dl[e] = 0.f;
                }
            }
        }
        cp_async_commit();
    };
    const int nch = (R + kResKC - 1) / kResKC;
    stage(0, 0);
    for (int t = tid; t < kRes2Rows * R; t += kThreads) {
        const int u = t / R, k = t - u * R;
        xr[u * stride + k] = i0 + u < I ? X[(i0 + u) * R + k] : 0.f;
    }
    const int r = tid / (kRes2Cols / 4), cq = 4 * (tid % (kRes2Cols / 4));
    const float* xrow = xr + r * stride;
    float s[4], c[4], sm[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) s[q] = c[q] = sm[q] = 0.f;
    for (int ch = 0; ch < nch; ++ch) {
        if (ch + 1 < nch)
            stage(ch + 1, (ch + 1) & 1);
        else
            cp_async_commit();   // an empty group keeps the wait count uniform
        cp_async_wait_prev();
        __syncthreads();
        const float* hh = vb + (size_t)(ch & 1) * 2 * kResKC * kRes2Cols + cq;
        const float* ll = hh + kResKC * kRes2Cols;
        const int k0 = ch * kResKC;
#pragma unroll 8
        for (int kk = 0; kk < kResKC; ++kk) {
            const float x = k0 + kk < R ? xrow[k0 + kk] : 0.f;
            const float4 h4 = *reinterpret_cast<const float4*>(hh + kk * kRes2Cols);
            const float4 l4 = *reinterpret_cast<const float4*>(ll + kk * kRes2Cols);
            const float vh[4] = {h4.x, h4.y, h4.z, h4.w}, vl[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float p = x * vh[q];
                sm[q] += fmaf(x, vh[q], -p);
                sm[q] = fmaf(x, vl[q], sm[q]);
                neumaier(s[q], c[q], p);
            }
        }
        __syncthreads();   // the buffer is refilled two chunks later
    }
    if (i0 + r < I) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = jb + cq + q;
            if (j < R) {
                const int64_t e = (i0 + r) * R + j;
                Res[e] = (M[e] - s[q]) - (c[q] + sm[q]);
            }
        }
    }
}

// lambda_r = ||X(:, r)||_2 and A(:, r) = X(:, r) / lambda_r (0 for a zero
// column), in fp64.  colsq_partial_kernel: block (cb, s) sums the squares of
// rows [I s / S, I (s + 1) / S) of 32 columns (eight warps, then the warps in
// order); normalize_apply_kernel: block (cb, rc) forms the 32 norms from the S
// partials (in s order) once and scales its rows.
constexpr int kNormSplits = 16, kNormRowsPerBlock = 64;

__global__ void __launch_bounds__(256) colsq_partial_kernel(const double* __restrict__ X, int64_t I, int R,
                                                            double* __restrict__ part) {
    __shared__ double ws[8][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * 32 + lane;
    const int64_t i0 = I * blockIdx.y / kNormSplits, i1 = I * (blockIdx.y + 1) / kNormSplits;
    double t = 0.0;
    if (r < R)
        for (int64_t i = i0 + warp; i < i1; i += 8) {
            const double v = X[i * R + r];
            t = fma(v, v, t);
        }
    ws[warp][lane] = t;
    __syncthreads();
    if (warp == 0 && r < R) {
        double u = 0.0;
        for (int w = 0; w < 8; ++w) u += ws[w][lane];
        part[(int64_t)blockIdx.y * R + r] = u;
    }
}

__global__ void __launch_bounds__(256) normalize_apply_kernel(const double* __restrict__ X, int64_t I, int R,
                                                              const double* __restrict__ part,
                                                              float* __restrict__ A, float* __restrict__ lam) {
    __shared__ double inv[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * 32 + lane;
    if (warp == 0) {
        double n2 = 0.0;
        if (r < R)
            for (int sp = 0; sp < kNormSplits; ++sp) n2 += part[(int64_t)sp * R + r];
        const double nr = sqrt(n2);
        inv[lane] = nr > 0.0 ? 1.0 / nr : 0.0;
        if (r < R && blockIdx.y == 0) lam[r] = (float)nr;
    }
    __syncthreads();
    if (r >= R) return;
    const double v = inv[lane];
    const int64_t i0 = (int64_t)blockIdx.y * kNormRowsPerBlock;
    const int64_t i1 = i0 + kNormRowsPerBlock < I ? i0 + kNormRowsPerBlock : I;
    for (int64_t i = i0 + warp; i < i1; i += 8) A[i * R + r] = (float)(X[i * R + r] * v);
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

__global__ void __launch_bounds__(kFitBlocks) fit_final_kernel(const double* __restrict__ part, int nb,
                                                            const double* __restrict__ norm_y2,
                                                            const int* __restrict__ info, double* __restrict__ fit) {
    // pairwise tree over the block partials (fixed order); nb <= kFitBlocks
    __shared__ double x2s[kFitBlocks], ins[kFitBlocks];
    const int t = threadIdx.x;
    x2s[t] = t < nb ? part[2 * t] : 0.0;
    ins[t] = t < nb ? part[2 * t + 1] : 0.0;
    __syncthreads();
    for (int h = kFitBlocks / 2; h > 0; h >>= 1) {
        if (t < h) {
            x2s[t] += x2s[t + h];
            ins[t] += ins[t + h];
        }
        __syncthreads();
    }
    if (t != 0) return;
    const double y2 = *norm_y2;
    const double res2 = y2 + x2s[0] - 2.0 * ins[0];
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
    // about eight working CTAs an SM (the lower-triangle tiles; the others exit
    // at once), at least one 32-row slab each: the slab loop is latency-bound
    const int64_t nt = (R + 15) / 16;
    const int64_t tiles = nt * (nt + 1) / 2;
    int64_t S = (152 * 8 + tiles - 1) / tiles;
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

cudaError_t cpals_hadamard(const double* G, int d, int skip, int R, double* V, float* vhi, float* vlo,
                           cudaStream_t s) {
    const int64_t n = (int64_t)R * R;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    hadamard_kernel<<<(unsigned)blocks, 256, 0, s>>>(G, d, skip, R, V, vhi, vlo);
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

int cpals_mixed_launches(int R) { return R <= kSmemMaxR ? 4 : 5 + cpals_cholesky_launches(R); }

size_t cpals_mixed_block_bytes(int R) { return (size_t)((R + kChB - 1) / kChB) * kChB * kChB * sizeof(float); }

namespace {
cudaError_t launch_residual(const float* M, const float* x0, const float* vhi, const float* vlo, int64_t I, int R,
                            float* res, cudaStream_t s) {
    const size_t rsm = res2_smem_bytes(R);
    const dim3 grid((unsigned)((R + kRes2Cols - 1) / kRes2Cols), (unsigned)((I + kRes2Rows - 1) / kRes2Rows));
    constexpr int threads = kRes2Rows * kRes2Cols / 4;
    cudaError_t e;
    if (R % 4 == 0 && ((reinterpret_cast<uintptr_t>(vhi) | reinterpret_cast<uintptr_t>(vlo)) & 15) == 0) {
        e = cudaFuncSetAttribute(residual2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm);
        if (e != cudaSuccess) return e;
        residual2_kernel<true><<<grid, threads, rsm, s>>>(M, x0, vhi, vlo, I, R, res);
    } else {
        e = cudaFuncSetAttribute(residual2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm);
        if (e != cudaSuccess) return e;
        residual2_kernel<false><<<grid, threads, rsm, s>>>(M, x0, vhi, vlo, I, R, res);
    }
    return cudaGetLastError();
}
}  // namespace

cudaError_t cpals_solve_mixed(const double* V, int R, const float* M, int64_t I, double* X, float* vhi, float* vlo,
                              float* L, float* dinv, float* dblk, float* x0, float* res, int* info, cudaStream_t s) {
    if (R > kChol32MaxR) return cudaErrorInvalidValue;
    cudaError_t e;
    if (R <= kSmemMaxR) {
        // one launch for the split and the factor, the row solves with the
        // inverted diagonal blocks
        const size_t csm = chol2_smem_bytes(R);
        e = cudaFuncSetAttribute(chol2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm);
        if (e != cudaSuccess) return e;
        chol2_kernel<<<1, kChol2Threads, csm, s>>>(vhi, R, L, dblk, dinv, info);
        const size_t ssm = sv2_smem_bytes(R);
        const unsigned sb = (unsigned)((I + kSv2Warps * kSv2Rows - 1) / (kSv2Warps * kSv2Rows));
        const bool vec = R % 4 == 0 && (reinterpret_cast<uintptr_t>(L) & 15) == 0;
        if (vec) {
            e = cudaFuncSetAttribute(solve2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
            if (e != cudaSuccess) return e;
            solve2_kernel<true><<<sb, kSv2Warps * 32, ssm, s>>>(L, dblk, R, M, I, x0, nullptr, nullptr);
        } else {
            e = cudaFuncSetAttribute(solve2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
            if (e != cudaSuccess) return e;
            solve2_kernel<false><<<sb, kSv2Warps * 32, ssm, s>>>(L, dblk, R, M, I, x0, nullptr, nullptr);
        }
        if ((e = launch_residual(M, x0, vhi, vlo, I, R, res, s)) != cudaSuccess) return e;
        if (vec)
            solve2_kernel<true><<<sb, kSv2Warps * 32, ssm, s>>>(L, dblk, R, res, I, nullptr, x0, X);
        else
            solve2_kernel<false><<<sb, kSv2Warps * 32, ssm, s>>>(L, dblk, R, res, I, nullptr, x0, X);
        return cudaGetLastError();
    }
    const int64_t n = (int64_t)R * R;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    split_v_kernel<<<(unsigned)blocks, 256, 0, s>>>(V, n, vhi, vlo, L);
    e = blocked_cholesky<float>(L, R, info, dinv, s);
    if (e != cudaSuccess) return e;
    mirror_lower_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(L, R);
    const size_t ssm = ((size_t)kSolveRows * R + (size_t)R * 33) * sizeof(float);
    e = cudaFuncSetAttribute(solve32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return e;
    const unsigned sblocks = (unsigned)((I + kSolveRows - 1) / kSolveRows);
    solve32_kernel<<<sblocks, 32, ssm, s>>>(L, dinv, R, M, I, x0, nullptr, nullptr);
    if ((e = launch_residual(M, x0, vhi, vlo, I, R, res, s)) != cudaSuccess) return e;
    solve32_kernel<<<sblocks, 32, ssm, s>>>(L, dinv, R, res, I, nullptr, x0, X);
    return cudaGetLastError();
}

size_t cpals_normalize_scratch_bytes(int R) { return (size_t)kNormSplits * R * sizeof(double); }

int cpals_normalize_launches() { return 2; }

cudaError_t cpals_normalize(const double* X, int64_t I, int R, float* A, float* lam, double* part, cudaStream_t s) {
    const unsigned cb = (unsigned)((R + 31) / 32);
    colsq_partial_kernel<<<dim3(cb, kNormSplits), 256, 0, s>>>(X, I, R, part);
    const int64_t rb = (I + kNormRowsPerBlock - 1) / kNormRowsPerBlock;
    normalize_apply_kernel<<<dim3(cb, (unsigned)(rb > 0 ? rb : 1)), 256, 0, s>>>(X, I, R, part, A, lam);
    return cudaGetLastError();
}

cudaError_t cpals_fit(const double* H, const float* lam, const float* M, const float* A, int64_t I, int R,
                      const double* norm_y2, const int* info, double* fit, double* part, cudaStream_t s) {
    fit_partial_kernel<<<kFitBlocks, 256, 0, s>>>(H, lam, M, A, I, R, part);
    fit_final_kernel<<<1, kFitBlocks, 0, s>>>(part, kFitBlocks, norm_y2, info, fit);
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
