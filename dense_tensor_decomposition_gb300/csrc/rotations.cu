// Givens rotations along one mode ("An HPC Approach to Accelerate Tensor
// Decompositions", §2 and §4.3, "Application of Rotations"): Y is
// multiplied in mode n by R^T, R the identity except for 2 x 2 blocks
// [[c, -s], [s, c]] at rows and columns (p, q) of a group of disjoint pivot
// pairs.  For every fibre along mode n and every pair g:
//     new[p_g] = c_g old[p_g] + s_g old[q_g],   new[q_g] = c_g old[q_g] - s_g old[p_g].
// Y is viewed as [P, N, Q] (P: modes before n, Q: modes after).  Bandwidth
// bound: each rotated row of every [N, Q] slab is read and written once.
#include "internal.h"

namespace mk {
namespace {

__device__ __forceinline__ bool pair_ok(int p, int q, int N) { return p >= 0 && q >= 0 && p < N && q < N && p != q; }

// any Q: one element pair per item, items ordered q fastest, then pair, then slab
__global__ void __launch_bounds__(256) rotate_items_kernel(float* __restrict__ Y, int64_t P, int N, int64_t Q,
                                                           const int* __restrict__ pairs, const float* __restrict__ c,
                                                           const float* __restrict__ s, int G) {
    const int64_t n = P * G * Q;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < n; it += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rq = it / Q;
        const int64_t q = it - rq * Q;
        const int64_t p = rq / G;
        const int g = (int)(rq - p * G);
        const int pg = pairs[2 * g], qg = pairs[2 * g + 1];
        if (!pair_ok(pg, qg, N)) continue;
        const float cg = c[g], sg = s[g];
        float* a = Y + (p * N + pg) * Q + q;
        float* b = Y + (p * N + qg) * Q + q;
        const float x = *a, y = *b;
        *a = fmaf(cg, x, sg * y);
        *b = fmaf(cg, y, -sg * x);
    }
}

// Q a multiple of 4, rows 16-byte aligned: one float4 of one row pair per
// item, items ordered as above, so a warp reads contiguous 512-byte runs of
// each row and the grid covers all rows of all slabs at once
__global__ void __launch_bounds__(256) rotate_items4_kernel(float4* __restrict__ Y, int64_t P, int N, int64_t Q4,
                                                            const int* __restrict__ pairs, const float* __restrict__ c,
                                                            const float* __restrict__ s, int G) {
    const int64_t n = P * G * Q4;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < n; it += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rq = it / Q4;
        const int64_t t = it - rq * Q4;
        const int64_t p = rq / G;
        const int g = (int)(rq - p * G);
        const int pg = pairs[2 * g], qg = pairs[2 * g + 1];
        if (!pair_ok(pg, qg, N)) continue;
        const float cg = c[g], sg = s[g];
        float4* a = Y + (p * N + pg) * Q4 + t;
        float4* b = Y + (p * N + qg) * Q4 + t;
        const float4 x = __ldcs(a), y = __ldcs(b);
        __stcs(a, make_float4(fmaf(cg, x.x, sg * y.x), fmaf(cg, x.y, sg * y.y), fmaf(cg, x.z, sg * y.z),
                              fmaf(cg, x.w, sg * y.w)));
        __stcs(b, make_float4(fmaf(cg, y.x, -sg * x.x), fmaf(cg, y.y, -sg * x.y), fmaf(cg, y.z, -sg * x.z),
                              fmaf(cg, y.w, -sg * x.w)));
    }
}

// short slabs (N * Q <= kSlab floats, e.g. the innermost mode): T whole
// consecutive [N, Q] slabs are read flat into shared memory, rotated there and
// written back flat, so every global access is coalesced.  With VEC the host
// has chosen T so that every tile starts on a 16-byte boundary: the tile is
// loaded with cp.async 16-byte copies (straight into shared memory, no
// registers, the whole tile in flight at once) and stored as float4s; the
// tail of the last tile goes element by element.
constexpr int kSlab = 8192;
constexpr int kSlabThreads = 256;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

// waits for this thread's copies (a hardware wait, no polling)
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

template <bool VEC>
__device__ __forceinline__ void slab_load(float* __restrict__ sm, const float* __restrict__ src, int nv) {
    int done = 0;
    if constexpr (VEC) {
        const int nv4 = nv >> 2;
        for (int e = threadIdx.x; e < nv4; e += kSlabThreads) cp_async16(sm + 4 * e, src + 4 * e);
        done = nv4 << 2;
    }
    for (int e = done + threadIdx.x; e < nv; e += kSlabThreads) sm[e] = __ldcs(src + e);
    if constexpr (VEC) cp_async_wait_all();
}

template <bool VEC>
__device__ __forceinline__ void slab_store(float* __restrict__ dst, const float* __restrict__ sm, int nv) {
    int done = 0;
    if constexpr (VEC) {
        const int nv4 = nv >> 2;
        const float4* s4 = reinterpret_cast<const float4*>(sm);
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll 4
        for (int e = threadIdx.x; e < nv4; e += kSlabThreads) __stcs(d4 + e, s4[e]);
        done = nv4 << 2;
    }
    for (int e = done + threadIdx.x; e < nv; e += kSlabThreads) __stcs(dst + e, sm[e]);
}

template <bool VEC>
__global__ void __launch_bounds__(kSlabThreads) rotate_slabs_kernel(float* __restrict__ Y, int64_t P, int N, int64_t Q,
                                                                    const int* __restrict__ pairs,
                                                                    const float* __restrict__ c,
                                                                    const float* __restrict__ s, int G, int T) {
    __shared__ float4 sm4[kSlab / 4];
    float* sm = reinterpret_cast<float*>(sm4);
    const int S = (int)(N * Q);
    const int Qi = (int)Q;
    // items of a tile are (slab t, pair g, q), q fastest; a thread takes every
    // kSlabThreads-th one, so its first item and its stride are the same in
    // every tile and are split into (t, g, q) once, without divisions later
    const int q0 = (int)threadIdx.x % Qi, r0 = (int)threadIdx.x / Qi;
    const int g0 = r0 % G, t0 = r0 / G;
    const int dq = kSlabThreads % Qi, dr = kSlabThreads / Qi;
    const int dg = dr % G, dt = dr / G;
    const int64_t ntiles = (P + T - 1) / T;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t p0 = tile * T;
        const int nt = (int)(P - p0 < T ? P - p0 : T);
        const int nv = nt * S;
        slab_load<VEC>(sm, Y + p0 * S, nv);
        __syncthreads();
        for (int q = q0, g = g0, t = t0; t < nt;) {
            const int pg = pairs[2 * g], qg = pairs[2 * g + 1];
            if (pair_ok(pg, qg, N)) {
                const float cg = c[g], sg = s[g];
                float* a = sm + t * S + pg * Qi + q;
                float* b = sm + t * S + qg * Qi + q;
                const float x = *a, y = *b;
                *a = fmaf(cg, x, sg * y);
                *b = fmaf(cg, y, -sg * x);
            }
            q += dq;                             // advance by kSlabThreads items
            int carry = 0;
            if (q >= Qi) { q -= Qi; carry = 1; }
            g += dg + carry;                     // < 2G
            if (g >= G) { g -= G; ++t; }
            t += dt;
        }
        __syncthreads();
        slab_store<VEC>(Y + p0 * S, sm, nv);
        __syncthreads();
    }
}

template <bool VEC>
int slab_blocks_per_sm() {
    static int occ = 0;
    if (occ == 0) {
        // largest shared-memory carveout, so that shared memory is not what limits residency
        cudaFuncSetAttribute(rotate_slabs_kernel<VEC>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rotate_slabs_kernel<VEC>, kSlabThreads, 0) !=
                cudaSuccess ||
            occ < 1)
            occ = 1;
        cudaGetLastError();
    }
    return occ;
}

}  // namespace

cudaError_t launch_rotations(float* Y, int64_t P, int N, int64_t Q, const int* pairs, const float* c, const float* s,
                             int G, cudaStream_t stream) {
    if (P == 0 || G == 0 || Q == 0) return cudaSuccess;
    const bool aligned = (reinterpret_cast<uintptr_t>(Y) & 15) == 0;
    const int64_t S = (int64_t)N * Q;
    if (S <= kSlab && (Q < 32 || Q % 4 != 0 || !aligned)) {
        int64_t T = kSlab / S;
        bool vec = false;
        if (aligned && T >= 4) {
            T &= ~(int64_t)3;                    // T * S a multiple of 4: every tile 16-byte aligned
            vec = true;
        } else if (aligned && S % 4 == 0) {
            vec = true;
        }
        int64_t blocks = (P + T - 1) / T;
        const int64_t cap = 152 * (int64_t)(vec ? slab_blocks_per_sm<true>() : slab_blocks_per_sm<false>());
        if (blocks > cap) blocks = cap;
        if (vec)
            rotate_slabs_kernel<true><<<(unsigned)blocks, kSlabThreads, 0, stream>>>(Y, P, N, Q, pairs, c, s, G, (int)T);
        else
            rotate_slabs_kernel<false><<<(unsigned)blocks, kSlabThreads, 0, stream>>>(Y, P, N, Q, pairs, c, s, G,
                                                                                       (int)T);
    } else if (aligned && Q % 4 == 0) {
        int64_t blocks = (P * G * (Q / 4) + 255) / 256;
        if (blocks > 152 * 16) blocks = 152 * 16;
        rotate_items4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<float4*>(Y), P, N, Q / 4, pairs,
                                                                   c, s, G);
    } else {
        int64_t blocks = (P * G * Q + 255) / 256;
        if (blocks > 152 * 16) blocks = 152 * 16;
        rotate_items_kernel<<<(unsigned)blocks, 256, 0, stream>>>(Y, P, N, Q, pairs, c, s, G);
    }
    return cudaGetLastError();
}

}  // namespace mk
