// Small helper kernels of the MTTKRP path:
//  * prod_table_kernel builds the factor-product tables G (pre modes) and
//    Binner (inner group) that the main kernels combine into Khatri-Rao rows
//    on the fly, plus the Y base offset of every pre index;
//  * reduce_splits_kernel adds the per-split partial results in a fixed order
//    in fp64 and writes the fp32 output (no atomics anywhere, so results are
//    bitwise reproducible).
#include "internal.h"

namespace mk {

__global__ void prod_table_kernel(ProdTableArgs a) {
    const int64_t n = a.rows * a.R;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / a.R;
        const int64_t r = e - row * a.R;
        int64_t rem = row;
        int64_t base = 0;
        float prod = 1.0f;
        for (int m = a.nm - 1; m >= 0; --m) {
            const int64_t idx = rem % a.dim[m];
            rem /= a.dim[m];
            prod *= a.fac[m][idx * a.R + r];
            base += idx * a.ystride[m];
        }
        a.tab[e] = prod;
        if (a.base != nullptr && r == 0) a.base[row] = base;
    }
}

cudaError_t launch_prod_table(const ProdTableArgs& a, cudaStream_t s) {
    const int64_t n = a.rows * a.R;
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    prod_table_kernel<<<(unsigned)blocks, threads, 0, s>>>(a);
    return cudaGetLastError();
}

// out[e] = (float) sum_{s=0}^{splits-1} (double) part[s * n + e], s in increasing order.
__global__ void reduce_splits_kernel(const float* __restrict__ part, int64_t splits, int64_t n,
                                     float* __restrict__ out) {
    const bool vec = (n % 4 == 0) && ((reinterpret_cast<uintptr_t>(part) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (vec) {
        const int64_t n4 = n / 4;
        for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4; e += stride) {
            double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
            for (int64_t sp = 0; sp < splits; ++sp) {
                const float4 v = __ldcs(reinterpret_cast<const float4*>(part + sp * n) + e);
                s0 += (double)v.x;
                s1 += (double)v.y;
                s2 += (double)v.z;
                s3 += (double)v.w;
            }
            reinterpret_cast<float4*>(out)[e] = make_float4((float)s0, (float)s1, (float)s2, (float)s3);
        }
    } else {
        for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
            double acc = 0.0;
            for (int64_t sp = 0; sp < splits; ++sp) acc += (double)__ldcs(part + sp * n + e);
            out[e] = (float)acc;
        }
    }
}

cudaError_t launch_reduce_splits(const float* part, int64_t splits, int64_t n, float* out,
                                 cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    int64_t work = (n % 4 == 0) ? n / 4 : n;
    int64_t blocks = (work + threads - 1) / threads;
    if (blocks > 152 * 8) blocks = 152 * 8;
    reduce_splits_kernel<<<(unsigned)blocks, threads, 0, s>>>(part, splits, n, out);
    return cudaGetLastError();
}

}  // namespace mk
