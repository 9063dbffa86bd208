// fp32 SIMT MTTKRP kernel (CUDA cores, FMA pipe).
//
// One CTA owns a BM x BN tile of M_k (rows i, columns r) and a contiguous range
// of pre indices pi.  It walks the contraction index kappa = (pi, j) in tiles
// of BK values of j:
//   * a BM x BK tile of the unfolding Y_(k) is read from HBM with 128-bit loads
//     (vectorised along j when the inner group is contiguous after mode k, along
//     i for the innermost mode) and stored k-major in shared memory;
//   * the matching BK x BN tile of the Khatri-Rao product is built on the fly
//     as G(pi, r) * Binner(j, r) from the two small factor-product tables;
//   * every thread accumulates an 8 x 8 register tile with fp32 FMAs
//     (outer products, as in a register-blocked SGEMM).
// Global loads of tile t+1 are issued before the FMAs of tile t (register
// prefetch into a second shared-memory buffer), one barrier per tile.
// The result (or, with split ranges, the partial of this range) is written
// without atomics.
#include "internal.h"

namespace mk {

namespace {

constexpr int kBK = 16;

__device__ __forceinline__ float4 ldg4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

// 128 x 128 tiles with vector loads of Y are held to 128 registers a thread, so
// two CTAs (16 warps) share an SM: the extra warps hide the latency of the
// shared-memory and global loads behind other warps' FMAs (no spills at that
// bound; the scalar-load variants would spill and keep one CTA per SM).
template <int BM, int BN, int BK, int AMODE, bool BVEC>
__global__ void __launch_bounds__((BM / 8) * (BN / 8), (BM == 128 && BN == 128 && AMODE != kLoadScalar) ? 2 : 1)
    simt_kernel(const SimtArgs a) {
    constexpr int NT = (BM / 8) * (BN / 8);
    constexpr int APAD = 4;
    constexpr int A_ELEMS = BM * BK / NT;
    constexpr int B_ELEMS = BK * BN / NT;
    static_assert(A_ELEMS % 4 == 0 && B_ELEMS % 4 == 0, "tile/thread mismatch");
    static_assert(NT % (BN / 4) == 0, "B columns must be fixed per thread");

    __shared__ __align__(16) float As[2][BK][BM + APAD];
    __shared__ __align__(16) float Bs[2][BK][BN];

    const int tid = threadIdx.x;
    const int tx = tid % (BN / 8);
    const int ty = tid / (BN / 8);
    const int64_t m0 = (int64_t)blockIdx.y * BM;
    const int64_t r0 = (int64_t)blockIdx.x * BN;
    const int64_t pre_lo = (int64_t)blockIdx.z * a.pre_per_split;
    int64_t pre_hi = pre_lo + a.pre_per_split;
    if (pre_hi > a.npre) pre_hi = a.npre;
    const int64_t nJ = (a.J + BK - 1) / BK;
    const int64_t T = pre_hi > pre_lo ? (pre_hi - pre_lo) * nJ : 0;

    float ra[A_ELEMS];
    float rb[B_ELEMS];

    auto load_tile = [&](int64_t t) {
        const int64_t tp = t / nJ;
        const int64_t pi = pre_lo + tp;
        const int64_t j0 = (t - tp * nJ) * BK;
        const int64_t base = a.base[pi];
        // ---- Y tile: rows m0.., columns j0.. ----
        if constexpr (AMODE == kLoadVecJ) {
#pragma unroll
            for (int v = 0; v < A_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int m = f / (BK / 4);
                const int kq = f % (BK / 4);
                const int64_t i = m0 + m;
                const int64_t j = j0 + kq * 4;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < a.I && j < a.J) {
                    const int64_t jp = j / a.Jq;
                    x = ldg4(a.Y + base + i * a.s_k + jp * a.IQ + (j - jp * a.Jq));
                }
                ra[4 * v + 0] = x.x;
                ra[4 * v + 1] = x.y;
                ra[4 * v + 2] = x.z;
                ra[4 * v + 3] = x.w;
            }
        } else if constexpr (AMODE == kLoadVecI) {
#pragma unroll
            for (int v = 0; v < A_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kk = f / (BM / 4);
                const int mq = f % (BM / 4);
                const int64_t i = m0 + mq * 4;
                const int64_t j = j0 + kk;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < a.I && j < a.J) {
                    const int64_t jp = j / a.Jq;
                    x = ldg4(a.Y + base + i + jp * a.IQ + (j - jp * a.Jq));
                }
                ra[4 * v + 0] = x.x;
                ra[4 * v + 1] = x.y;
                ra[4 * v + 2] = x.z;
                ra[4 * v + 3] = x.w;
            }
        } else {
            const bool icontig = (a.s_k == 1);
#pragma unroll
            for (int e = 0; e < A_ELEMS; ++e) {
                const int f = tid + NT * e;
                const int m = icontig ? (f % BM) : (f / BK);
                const int kk = icontig ? (f / BM) : (f % BK);
                const int64_t i = m0 + m;
                const int64_t j = j0 + kk;
                float x = 0.f;
                if (i < a.I && j < a.J) {
                    const int64_t jp = j / a.Jq;
                    x = __ldg(a.Y + base + i * a.s_k + jp * a.IQ + (j - jp * a.Jq));
                }
                ra[e] = x;
            }
        }
        // ---- Khatri-Rao tile: G(pi, r) * Binner(j, r) ----
        const float* grow = a.gtab + pi * a.R;
        if constexpr (BVEC) {
#pragma unroll
            for (int v = 0; v < B_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kk = f / (BN / 4);
                const int nq = f % (BN / 4);
                const int64_t r = r0 + nq * 4;
                const int64_t j = j0 + kk;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < a.J && r < a.R) {
                    const float4 b = ldg4(a.binner + j * a.R + r);
                    const float4 g = ldg4(grow + r);
                    x = make_float4(g.x * b.x, g.y * b.y, g.z * b.z, g.w * b.w);
                }
                rb[4 * v + 0] = x.x;
                rb[4 * v + 1] = x.y;
                rb[4 * v + 2] = x.z;
                rb[4 * v + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < B_ELEMS; ++e) {
                const int f = tid + NT * e;
                const int kk = f / BN;
                const int n = f % BN;
                const int64_t r = r0 + n;
                const int64_t j = j0 + kk;
                float x = 0.f;
                if (j < a.J && r < a.R) x = __ldg(grow + r) * __ldg(a.binner + j * a.R + r);
                rb[e] = x;
            }
        }
    };

    auto store_tile = [&](int buf) {
        if constexpr (AMODE == kLoadVecJ) {
#pragma unroll
            for (int v = 0; v < A_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int m = f / (BK / 4);
                const int kq = f % (BK / 4);
#pragma unroll
                for (int c = 0; c < 4; ++c) As[buf][kq * 4 + c][m] = ra[4 * v + c];
            }
        } else if constexpr (AMODE == kLoadVecI) {
#pragma unroll
            for (int v = 0; v < A_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kk = f / (BM / 4);
                const int mq = f % (BM / 4);
                *reinterpret_cast<float4*>(&As[buf][kk][mq * 4]) =
                    make_float4(ra[4 * v], ra[4 * v + 1], ra[4 * v + 2], ra[4 * v + 3]);
            }
        } else {
            const bool icontig = (a.s_k == 1);
#pragma unroll
            for (int e = 0; e < A_ELEMS; ++e) {
                const int f = tid + NT * e;
                const int m = icontig ? (f % BM) : (f / BK);
                const int kk = icontig ? (f / BM) : (f % BK);
                As[buf][kk][m] = ra[e];
            }
        }
        if constexpr (BVEC) {
#pragma unroll
            for (int v = 0; v < B_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kk = f / (BN / 4);
                const int nq = f % (BN / 4);
                *reinterpret_cast<float4*>(&Bs[buf][kk][nq * 4]) =
                    make_float4(rb[4 * v], rb[4 * v + 1], rb[4 * v + 2], rb[4 * v + 3]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < B_ELEMS; ++e) {
                const int f = tid + NT * e;
                Bs[buf][f / BN][f % BN] = rb[e];
            }
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    if (T > 0) {
        load_tile(0);
        store_tile(0);
    }
    __syncthreads();

    for (int64_t t = 0; t < T; ++t) {
        const int buf = (int)(t & 1);
        if (t + 1 < T) load_tile(t + 1);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][BM / 2 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][BN / 2 + tx * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (t + 1 < T) store_tile(buf ^ 1);
        __syncthreads();
    }

    // ---- write the tile (or this range's partial) ----
    float* dst = a.dst + (int64_t)blockIdx.z * a.dst_split_stride;
    const bool vst = (a.R % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.dst) & 15) == 0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
        if (row >= a.I) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t col = r0 + h * (BN / 2) + tx * 4;
            float* p = dst + row * a.R + col;
            if (vst && col + 3 < a.R) {
                *reinterpret_cast<float4*>(p) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (col + c < a.R) p[c] = acc[i][4 * h + c];
            }
        }
    }
}

template <int BM, int BN>
cudaError_t launch_tile(int amode, bool bvec, const SimtArgs& a, int64_t splits, cudaStream_t s) {
    dim3 grid((unsigned)((a.R + BN - 1) / BN), (unsigned)((a.I + BM - 1) / BM), (unsigned)splits);
    dim3 block((BM / 8) * (BN / 8));
    if (amode == kLoadVecJ) {
        if (bvec) simt_kernel<BM, BN, kBK, kLoadVecJ, true><<<grid, block, 0, s>>>(a);
        else      simt_kernel<BM, BN, kBK, kLoadVecJ, false><<<grid, block, 0, s>>>(a);
    } else if (amode == kLoadVecI) {
        if (bvec) simt_kernel<BM, BN, kBK, kLoadVecI, true><<<grid, block, 0, s>>>(a);
        else      simt_kernel<BM, BN, kBK, kLoadVecI, false><<<grid, block, 0, s>>>(a);
    } else {
        if (bvec) simt_kernel<BM, BN, kBK, kLoadScalar, true><<<grid, block, 0, s>>>(a);
        else      simt_kernel<BM, BN, kBK, kLoadScalar, false><<<grid, block, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

bool simt_tile_supported(int bm, int bn) {
    return (bn == 128 && (bm == 128 || bm == 64 || bm == 32)) ||
           (bn == 64 && (bm == 128 || bm == 64 || bm == 32));
}

// Peak probe of the fp32 FMA pipe: eight independent chains of fused
// multiply-adds a thread (enough independent work to hide the pipe's latency
// at 8 warps per scheduler); each thread stores its sum so nothing is dropped.
// flops = 16 x iters x threads.
__global__ void __launch_bounds__(256) fma_probe_kernel(int iters, float* __restrict__ out) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    float x[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = 1.0f + 1e-3f * (float)(c + (t & 7));
    const float m = 0.999999f, b = 1e-7f;
#pragma unroll 4
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = fmaf(x[c], m, b);
    }
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) sum += x[c];
    out[t] = sum;
}

cudaError_t launch_fma_probe(int blocks, int iters, float* out, cudaStream_t s) {
    fma_probe_kernel<<<blocks, 256, 0, s>>>(iters, out);
    return cudaGetLastError();
}

cudaError_t launch_simt(int bm, int bn, int amode, bool bvec, const SimtArgs& a, int64_t splits,
                        cudaStream_t s) {
    if (bn == 128) {
        if (bm == 128) return launch_tile<128, 128>(amode, bvec, a, splits, s);
        if (bm == 64) return launch_tile<64, 128>(amode, bvec, a, splits, s);
        if (bm == 32) return launch_tile<32, 128>(amode, bvec, a, splits, s);
    } else if (bn == 64) {
        if (bm == 128) return launch_tile<128, 64>(amode, bvec, a, splits, s);
        if (bm == 64) return launch_tile<64, 64>(amode, bvec, a, splits, s);
        if (bm == 32) return launch_tile<32, 64>(amode, bvec, a, splits, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mk
