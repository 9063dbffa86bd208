// Dense mode-n product, TTM ("An HPC Approach to Accelerate Tensor
// Decompositions", §2, eq. (1)): T = X x_n M for M of size J x N (N = I_n),
//     T[p, j, q] = sum_i M[j, i] X[p, i, q],
// with X viewed as [P, N, Q] (P: modes before n, Q: modes after) and T as
// [P, J, Q].  All slabs form one fp32 SGEMM: rows j, columns c = p * Q + q,
// contraction over i.  Column c of the right operand starts at
// X + p*N*Q + q with stride Q, column c of the result at T + p*J*Q + q; each
// CTA puts the offsets of its columns in a shared table once.  Register-tiled
// like the SIMT MTTKRP kernel: 8 x 8 outputs per thread, 16-index K tiles,
// register prefetch of tile t+1 during the FMAs of tile t.  How X is read
// depends on where its contiguous run is:
//   kColVecQ     Q % 4 == 0: float4 along the columns (4 q of one slab);
//   kColScalarQ  Q >= 32, not a multiple of 4: scalars along the columns;
//   kColVecK     Q == 1 (innermost mode), N % 4 == 0: float4 along i;
//   kColScalarK  otherwise (short Q): scalars along i.
#include "internal.h"

namespace mk {
namespace {

constexpr int kTBK = 16;
constexpr int kTBN = 128;
enum { kColVecQ = 0, kColScalarQ = 1, kColVecK = 2, kColScalarK = 3 };

// 128-row tiles: two CTAs (16 warps) per SM, at most 128 registers a thread;
// the narrower tiles hold more prefetch registers per thread and keep theirs
template <int BM, int XMODE, bool AVEC>
__global__ void __launch_bounds__((BM / 8) * (kTBN / 8), BM == 128 ? 2 : 1)
    ttm_kernel(const float* __restrict__ X, const float* __restrict__ M, float* __restrict__ T, int64_t P, int64_t N,
               int64_t Q, int64_t J) {
    constexpr int BN = kTBN;
    constexpr int BK = kTBK;
    constexpr int NT = (BM / 8) * (BN / 8);
    constexpr int APAD = 4;
    constexpr int A_ELEMS = BM * BK / NT;
    constexpr int B_ELEMS = BK * BN / NT;
    static_assert(A_ELEMS % 4 == 0 && B_ELEMS % 4 == 0, "tile/thread mismatch");

    __shared__ __align__(16) float As[2][BK][BM + APAD];
    __shared__ __align__(16) float Bs[2][BK][BN];
    __shared__ int64_t xoff[BN];
    __shared__ int64_t toff[BN];

    const int tid = threadIdx.x;
    const int tx = tid % (BN / 8);
    const int ty = tid / (BN / 8);
    // the row tiles of one column tile are consecutive CTAs, so they run
    // together and read that slice of X from HBM once (then from L2)
    const int64_t nrt = (J + BM - 1) / BM;
    const int64_t j0 = ((int64_t)blockIdx.x % nrt) * BM;
    const int64_t c0 = ((int64_t)blockIdx.x / nrt) * BN;
    const int64_t ncol = P * Q;
    for (int n = tid; n < BN; n += NT) {
        const int64_t c = c0 + n;
        const int64_t p = c / Q, q = c - (c / Q) * Q;
        xoff[n] = c < ncol ? p * N * Q + q : -1;
        toff[n] = c < ncol ? p * J * Q + q : -1;
    }
    __syncthreads();
    const int64_t nK = (N + BK - 1) / BK;

    float ra[A_ELEMS];
    float rb[B_ELEMS];

    auto load_tile = [&](int64_t t) {
        const int64_t k0 = t * BK;
        // ---- M tile: rows j0.., indices k0.. (M is J x N row-major) ----
        if constexpr (AVEC) {
#pragma unroll
            for (int v = 0; v < A_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int m = f / (BK / 4);
                const int kq = f % (BK / 4);
                const int64_t j = j0 + m, i = k0 + kq * 4;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < J && i < N) x = __ldg(reinterpret_cast<const float4*>(M + j * N + i));
                ra[4 * v + 0] = x.x;
                ra[4 * v + 1] = x.y;
                ra[4 * v + 2] = x.z;
                ra[4 * v + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < A_ELEMS; ++e) {
                const int f = tid + NT * e;
                const int m = f / BK, kk = f % BK;
                const int64_t j = j0 + m, i = k0 + kk;
                ra[e] = (j < J && i < N) ? __ldg(M + j * N + i) : 0.f;
            }
        }
        // ---- X tile: indices k0.., columns c0.. ----
        if constexpr (XMODE == kColVecQ) {
#pragma unroll
            for (int v = 0; v < B_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kk = f / (BN / 4);
                const int nq = f % (BN / 4);
                const int64_t i = k0 + kk;
                const int64_t o = xoff[nq * 4];
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (o >= 0 && i < N) x = __ldg(reinterpret_cast<const float4*>(X + o + i * Q));
                rb[4 * v + 0] = x.x;
                rb[4 * v + 1] = x.y;
                rb[4 * v + 2] = x.z;
                rb[4 * v + 3] = x.w;
            }
        } else if constexpr (XMODE == kColScalarQ) {
#pragma unroll
            for (int e = 0; e < B_ELEMS; ++e) {
                const int f = tid + NT * e;
                const int kk = f / BN, n = f % BN;
                const int64_t i = k0 + kk;
                const int64_t o = xoff[n];
                rb[e] = (o >= 0 && i < N) ? __ldg(X + o + i * Q) : 0.f;
            }
        } else if constexpr (XMODE == kColVecK) {
#pragma unroll
            for (int v = 0; v < B_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kq = f % (BK / 4);
                const int n = f / (BK / 4);
                const int64_t i = k0 + kq * 4;
                const int64_t o = xoff[n];
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (o >= 0 && i < N) x = __ldg(reinterpret_cast<const float4*>(X + o + i));
                rb[4 * v + 0] = x.x;
                rb[4 * v + 1] = x.y;
                rb[4 * v + 2] = x.z;
                rb[4 * v + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < B_ELEMS; ++e) {
                const int f = tid + NT * e;
                const int kk = f % BK, n = f / BK;
                const int64_t i = k0 + kk;
                const int64_t o = xoff[n];
                rb[e] = (o >= 0 && i < N) ? __ldg(X + o + i * Q) : 0.f;
            }
        }
    };

    auto store_tile = [&](int buf) {
        if constexpr (AVEC) {
#pragma unroll
            for (int v = 0; v < A_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int m = f / (BK / 4);
                const int kq = f % (BK / 4);
#pragma unroll
                for (int c = 0; c < 4; ++c) As[buf][kq * 4 + c][m] = ra[4 * v + c];
            }
        } else {
#pragma unroll
            for (int e = 0; e < A_ELEMS; ++e) {
                const int f = tid + NT * e;
                As[buf][f % BK][f / BK] = ra[e];
            }
        }
        if constexpr (XMODE == kColVecQ) {
#pragma unroll
            for (int v = 0; v < B_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kk = f / (BN / 4);
                const int nq = f % (BN / 4);
                *reinterpret_cast<float4*>(&Bs[buf][kk][nq * 4]) =
                    make_float4(rb[4 * v], rb[4 * v + 1], rb[4 * v + 2], rb[4 * v + 3]);
            }
        } else if constexpr (XMODE == kColScalarQ) {
#pragma unroll
            for (int e = 0; e < B_ELEMS; ++e) {
                const int f = tid + NT * e;
                Bs[buf][f / BN][f % BN] = rb[e];
            }
        } else if constexpr (XMODE == kColVecK) {
#pragma unroll
            for (int v = 0; v < B_ELEMS / 4; ++v) {
                const int f = tid + NT * v;
                const int kq = f % (BK / 4);
                const int n = f / (BK / 4);
#pragma unroll
                for (int c = 0; c < 4; ++c) Bs[buf][kq * 4 + c][n] = rb[4 * v + c];
            }
        } else {
#pragma unroll
            for (int e = 0; e < B_ELEMS; ++e) {
                const int f = tid + NT * e;
                Bs[buf][f % BK][f / BK] = rb[e];
            }
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    load_tile(0);
    store_tile(0);
    __syncthreads();
    for (int64_t t = 0; t < nK; ++t) {
        const int buf = (int)(t & 1);
        if (t + 1 < nK) load_tile(t + 1);
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
        if (t + 1 < nK) store_tile(buf ^ 1);
        __syncthreads();
    }

    // ---- write the tile: row j of column c goes to T[toff[c] + j * Q] ----
    const bool tal = (reinterpret_cast<uintptr_t>(T) & 15) == 0;
    if (Q % 4 == 0 && tal) {                     // float4 along 4 columns of one slab
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t j = j0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
            if (j >= J) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t o = toff[h * (BN / 2) + tx * 4];
                if (o < 0) continue;
                __stcs(reinterpret_cast<float4*>(T + o + j * Q),
                       make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]));
            }
        }
    } else if (Q == 1 && J % 4 == 0 && tal) {    // innermost mode: float4 along 4 rows j
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int64_t o = toff[h * (BN / 2) + tx * 4 + c];
                if (o < 0) continue;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int64_t j = j0 + r * (BM / 2) + ty * 4;
                    if (j >= J) continue;        // J % 4 == 0: j .. j + 3 all valid
                    __stcs(reinterpret_cast<float4*>(T + o + j),
                           make_float4(acc[4 * r][4 * h + c], acc[4 * r + 1][4 * h + c], acc[4 * r + 2][4 * h + c],
                                       acc[4 * r + 3][4 * h + c]));
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t j = j0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
            if (j >= J) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int64_t o = toff[h * (BN / 2) + tx * 4 + c];
                    if (o >= 0) T[o + j * Q] = acc[i][4 * h + c];
                }
        }
    }
}

template <int BM, bool AVEC>
cudaError_t launch_bm(int xmode, const float* X, const float* M, float* T, int64_t P, int64_t N, int64_t Q, int64_t J,
                      cudaStream_t s) {
    const dim3 grid((unsigned)(((P * Q + kTBN - 1) / kTBN) * ((J + BM - 1) / BM)));
    const dim3 block((BM / 8) * (kTBN / 8));
    switch (xmode) {
        case kColVecQ: ttm_kernel<BM, kColVecQ, AVEC><<<grid, block, 0, s>>>(X, M, T, P, N, Q, J); break;
        case kColScalarQ: ttm_kernel<BM, kColScalarQ, AVEC><<<grid, block, 0, s>>>(X, M, T, P, N, Q, J); break;
        case kColVecK: ttm_kernel<BM, kColVecK, AVEC><<<grid, block, 0, s>>>(X, M, T, P, N, Q, J); break;
        default: ttm_kernel<BM, kColScalarK, AVEC><<<grid, block, 0, s>>>(X, M, T, P, N, Q, J); break;
    }
    return cudaGetLastError();
}

}  // namespace

int ttm_row_tile(int64_t J) { return J <= 32 ? 32 : (J <= 64 ? 64 : 128); }

int64_t ttm_tiles(int64_t P, int64_t Q, int64_t J) {
    const int64_t bm = ttm_row_tile(J);
    return ((P * Q + kTBN - 1) / kTBN) * ((J + bm - 1) / bm);
}

cudaError_t launch_ttm(const float* X, const float* M, float* T, int64_t P, int64_t N, int64_t Q, int64_t J,
                       cudaStream_t s) {
    const bool xal = (reinterpret_cast<uintptr_t>(X) & 15) == 0;
    const bool aal = (reinterpret_cast<uintptr_t>(M) & 15) == 0 && N % 4 == 0;
    int xmode;
    if (Q % 4 == 0 && xal) xmode = kColVecQ;
    else if (Q >= 32) xmode = kColScalarQ;
    else if (Q == 1 && N % 4 == 0 && xal) xmode = kColVecK;
    else xmode = kColScalarK;
    const int bm = ttm_row_tile(J);
    if (bm == 32) return aal ? launch_bm<32, true>(xmode, X, M, T, P, N, Q, J, s)
                             : launch_bm<32, false>(xmode, X, M, T, P, N, Q, J, s);
    if (bm == 64) return aal ? launch_bm<64, true>(xmode, X, M, T, P, N, Q, J, s)
                             : launch_bm<64, false>(xmode, X, M, T, P, N, Q, J, s);
    return aal ? launch_bm<128, true>(xmode, X, M, T, P, N, Q, J, s)
               : launch_bm<128, false>(xmode, X, M, T, P, N, Q, J, s);
}

}  // namespace mk
