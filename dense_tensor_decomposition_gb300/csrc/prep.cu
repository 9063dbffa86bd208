// Small helper kernels of the MTTKRP path:
//  * prod_table_kernel builds the factor-product tables G (pre modes) and
//    Binner (inner group) that the main kernels combine into Khatri-Rao rows
//    on the fly, plus the Y base offset of every pre index;
//  * the split reductions add the per-split partial results in a fixed order
//    with compensated (Neumaier) fp32 additions and write the fp32 output; no
//    atomics anywhere, so results are bitwise reproducible for a given plan.
#include "internal.h"
#include "scale.cuh"

namespace mk {

// One warp per (table row, run of 128 columns): the row's multi-index, Y offset
// and scale, then its columns by the lanes (coalesced; 16-byte loads and stores
// when R is a multiple of 4 and every factor is 16-byte aligned: a run is then
// 128 float4).  Splitting rows into runs keeps tables of few long rows (a single
// pre mode at a large rank) spread over the GPU.  NM = the number of factors in
// the product (a template argument, so that the per-column loop holds only its
// loads and multiplies).
template <int NM, bool V4>
__global__ void __launch_bounds__(256) prod_table_kernel(ProdTableArgs a) {
    if (a.enable != nullptr && *a.enable == 0) return;
    const int lane = threadIdx.x & 31;
    constexpr int64_t kRun = 128;   // float4 groups (V4) or columns a run
    const int64_t units = V4 ? a.R / 4 : a.R;
    const int64_t runs = (units + kRun - 1) / kRun;
    const int64_t tasks = a.rows * runs;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t task = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < tasks;
         task += nwarps) {
        const int64_t row = task / runs, run = task - row * runs;
        const float* frow[NM > 0 ? NM : 1];
        int64_t rem = row, base = 0;
#pragma unroll
        for (int m = NM - 1; m >= 0; --m) {
            const int64_t idx = rem % a.dim[m];
            rem /= a.dim[m];
            frow[m] = a.fac[m] + idx * a.R;
            base += idx * a.ystride[m];
        }
        float f = 1.f;
        if (a.slab_bits != nullptr)
            f = pow2_scale(*a.gmax_bits) * pow2_recip(slab_scale(a.slab_bits, row / a.slab_div, *a.gmax_bits));
        float* out = a.tab + row * a.R;
        const int64_t u1 = (run + 1) * kRun < units ? (run + 1) * kRun : units;
        if (V4) {
            for (int64_t c = run * kRun + lane; c < u1; c += 32) {
                float4 p = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
                for (int m = NM - 1; m >= 0; --m) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(frow[m]) + c);
                    p.x *= v.x;
                    p.y *= v.y;
                    p.z *= v.z;
                    p.w *= v.w;
                }
                reinterpret_cast<float4*>(out)[c] = make_float4(p.x * f, p.y * f, p.z * f, p.w * f);
            }
        } else {
            for (int64_t r = run * kRun + lane; r < u1; r += 32) {
                float p = 1.f;
#pragma unroll
                for (int m = NM - 1; m >= 0; --m) p *= __ldg(frow[m] + r);
                out[r] = p * f;
            }
        }
        if (a.base != nullptr && run == 0 && lane == 0) a.base[row] = base;
    }
}

template <int NM>
cudaError_t launch_prod_table_nm(const ProdTableArgs& a, bool v4, unsigned blocks, cudaStream_t s) {
    if (v4)
        prod_table_kernel<NM, true><<<blocks, 256, 0, s>>>(a);
    else
        prod_table_kernel<NM, false><<<blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prod_table(const ProdTableArgs& a, cudaStream_t s) {
    if (a.rows * a.R == 0) return cudaSuccess;
    bool v4 = a.R % 4 == 0 && (reinterpret_cast<uintptr_t>(a.tab) & 15) == 0;
    for (int m = 0; m < a.nm; ++m) v4 = v4 && (reinterpret_cast<uintptr_t>(a.fac[m]) & 15) == 0;
    const int64_t units = v4 ? a.R / 4 : a.R;
    int64_t blocks = (a.rows * ((units + 127) / 128) + 7) / 8;   // eight warps, one (row, run) each
    if (blocks > 152 * 16) blocks = 152 * 16;
    const unsigned b = (unsigned)blocks;
    static_assert(kMaxD == 8, "one instantiation per factor count");
    switch (a.nm) {
        case 0: return launch_prod_table_nm<0>(a, v4, b, s);
        case 1: return launch_prod_table_nm<1>(a, v4, b, s);
        case 2: return launch_prod_table_nm<2>(a, v4, b, s);
        case 3: return launch_prod_table_nm<3>(a, v4, b, s);
        case 4: return launch_prod_table_nm<4>(a, v4, b, s);
        case 5: return launch_prod_table_nm<5>(a, v4, b, s);
        case 6: return launch_prod_table_nm<6>(a, v4, b, s);
        case 7: return launch_prod_table_nm<7>(a, v4, b, s);
        case 8: return launch_prod_table_nm<8>(a, v4, b, s);
        default: return cudaErrorInvalidValue;
    }
}

// Compensated fp32 addition (Neumaier): sum + c carries the exact running total
// to about one fp32 rounding, independent of the number of terms; GB300's fp64
// rate is too low for a bandwidth-bound sum of this size.
__device__ __forceinline__ void kahan_add(float& sum, float& c, float x) {
    const float t = sum + x;
    c += fabsf(sum) >= fabsf(x) ? (sum - t) + x : (x - t) + sum;
    sum = t;
}

// out[e] = sum over s of part[s * n + e].  A block of 256 threads owns G
// groups of V consecutive outputs (one 16-byte group per thread when V = 4)
// and cuts the splits into Q = 256 / G contiguous slices: thread (slice q,
// group g) adds the partials of splits [q S / Q, (q + 1) S / Q) in increasing s
// with several loads in flight (compensated fp32), and the Q slice sums are
// added in slice order (compensated fp32 again).  The order depends only on
// (S, n, G), so results are bitwise reproducible; many slices keep enough
// loads in flight when there are few outputs and many splits.
constexpr int kRedThreads = 256;

template <int V, int G>   // V = 4: float4 groups; V = 1: scalars
__global__ void __launch_bounds__(kRedThreads)
    reduce_splits_kernel(const float* __restrict__ part, int64_t splits, int64_t n, float* __restrict__ out) {
    constexpr int Q = kRedThreads / G;
    __shared__ float sums[Q][G][V];
    const int gl = threadIdx.x % G, q = threadIdx.x / G;
    const int64_t s0 = splits * q / Q;
    const int64_t s1 = splits * (q + 1) / Q;
    const int64_t ng = n / V;   // groups
    for (int64_t base = (int64_t)blockIdx.x * G; base < ng; base += (int64_t)gridDim.x * G) {
        const int64_t g = base + gl;
        float acc[V], cmp[V];
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] = cmp[c] = 0.f;
        if (g < ng) {
            int64_t sp = s0;
            for (; sp + 4 <= s1; sp += 4) {
                float v[4][V];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float* p = part + (sp + u) * n + g * V;
                    if constexpr (V == 4) {
                        const float4 x = __ldcs(reinterpret_cast<const float4*>(p));
                        v[u][0] = x.x;
                        v[u][1] = x.y;
                        v[u][2] = x.z;
                        v[u][3] = x.w;
                    } else {
                        v[u][0] = __ldcs(p);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int c = 0; c < V; ++c) kahan_add(acc[c], cmp[c], v[u][c]);
            }
            for (; sp < s1; ++sp) {
                const float* p = part + sp * n + g * V;
                if constexpr (V == 4) {
                    const float4 x = __ldcs(reinterpret_cast<const float4*>(p));
                    kahan_add(acc[0], cmp[0], x.x);
                    kahan_add(acc[1], cmp[1], x.y);
                    kahan_add(acc[2], cmp[2], x.z);
                    kahan_add(acc[3], cmp[3], x.w);
                } else {
                    kahan_add(acc[0], cmp[0], __ldcs(p));
                }
            }
        }
#pragma unroll
        for (int c = 0; c < V; ++c) sums[q][gl][c] = acc[c] + cmp[c];
        __syncthreads();
        if (q == 0 && g < ng) {
            float t[V], tc[V];
#pragma unroll
            for (int c = 0; c < V; ++c) t[c] = tc[c] = 0.f;
            for (int w = 0; w < Q; ++w)
#pragma unroll
                for (int c = 0; c < V; ++c) kahan_add(t[c], tc[c], sums[w][gl][c]);
            if constexpr (V == 4)
                reinterpret_cast<float4*>(out)[g] = make_float4(t[0] + tc[0], t[1] + tc[1], t[2] + tc[2], t[3] + tc[3]);
            else
                out[g] = t[0] + tc[0];
        }
        __syncthreads();
    }
}

// One thread per 4 consecutive outputs, all splits in increasing s with eight
// 16-byte loads in flight (used when there are enough outputs to fill the GPU
// this way; no shared memory, no block barriers).
__global__ void __launch_bounds__(256)
    reduce_splits_flat_kernel(const float4* __restrict__ part, int64_t splits, int64_t n4,
                              float4* __restrict__ out) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
         e += (int64_t)gridDim.x * blockDim.x) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
        const float4* p = part + e;
        // up to eight 16-byte loads in flight (the last batch predicated), then
        // the compensated sums in split order
        for (int64_t sp = 0; sp < splits; sp += 8) {
            const int nb = splits - sp < 8 ? (int)(splits - sp) : 8;
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (u < nb) v[u] = __ldcs(p + (sp + u) * n4);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (u >= nb) break;
                kahan_add(s0, c0, v[u].x);
                kahan_add(s1, c1, v[u].y);
                kahan_add(s2, c2, v[u].z);
                kahan_add(s3, c3, v[u].w);
            }
        }
        out[e] = make_float4(s0 + c0, s1 + c1, s2 + c2, s3 + c3);
    }
}

cudaError_t launch_reduce_splits(const float* part, int64_t splits, int64_t n, float* out,
                                 cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const bool vec = n % 4 == 0 && (reinterpret_cast<uintptr_t>(part) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    const int64_t groups = vec ? n / 4 : n;
    if (vec && groups >= 152 * 256) {
        int64_t blocks = (groups + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        reduce_splits_flat_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(part), splits,
                                                                   groups, reinterpret_cast<float4*>(out));
        return cudaGetLastError();
    }
    // many splits: 32 slices of eight groups a block; few: 8 slices of 32 groups
    const bool wide = splits >= 64;
    const int G = wide ? 8 : 32;
    int64_t blocks = (groups + G - 1) / G;
    if (blocks > 152 * 16) blocks = 152 * 16;
    const unsigned b = (unsigned)blocks;
    if (vec && wide)
        reduce_splits_kernel<4, 8><<<b, kRedThreads, 0, s>>>(part, splits, n, out);
    else if (vec)
        reduce_splits_kernel<4, 32><<<b, kRedThreads, 0, s>>>(part, splits, n, out);
    else if (wide)
        reduce_splits_kernel<1, 8><<<b, kRedThreads, 0, s>>>(part, splits, n, out);
    else
        reduce_splits_kernel<1, 32><<<b, kRedThreads, 0, s>>>(part, splits, n, out);
    return cudaGetLastError();
}

}  // namespace mk
