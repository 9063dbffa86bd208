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

// out[e] = (float) sum over s of (double) part[s * n + e], summed in a fixed order
// that depends only on (splits, n): each block owns 32 consecutive outputs (one
// per lane); warp w adds the partials of splits [w*S/8, (w+1)*S/8) in
// increasing s; the eight warp sums are then added in warp order.  The result
// is therefore bitwise reproducible, and the S loads are spread over 8 warps
// instead of one serial loop per output.
constexpr int kRedWarps = 8;

__global__ void __launch_bounds__(kRedWarps * 32)
    reduce_splits_kernel(const float* __restrict__ part, int64_t splits, int64_t n,
                         float* __restrict__ out) {
    __shared__ double sums[kRedWarps][32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t s0 = splits * warp / kRedWarps;
    const int64_t s1 = splits * (warp + 1) / kRedWarps;
    for (int64_t base = (int64_t)blockIdx.x * 32; base < n; base += (int64_t)gridDim.x * 32) {
        const int64_t e = base + lane;
        double acc = 0.0;
        if (e < n) {
            const float* p = part + s0 * n + e;
            int64_t sp = s0;
            // four independent loads in flight, added in split order
            for (; sp + 4 <= s1; sp += 4, p += 4 * n) {
                const float a0 = __ldcs(p), a1 = __ldcs(p + n), a2 = __ldcs(p + 2 * n), a3 = __ldcs(p + 3 * n);
                acc += (double)a0;
                acc += (double)a1;
                acc += (double)a2;
                acc += (double)a3;
            }
            for (; sp < s1; ++sp, p += n) acc += (double)__ldcs(p);
        }
        sums[warp][lane] = acc;
        __syncthreads();
        if (warp == 0 && e < n) {
            double t = 0.0;
#pragma unroll
            for (int w = 0; w < kRedWarps; ++w) t += sums[w][lane];
            out[e] = (float)t;
        }
        __syncthreads();
    }
}

cudaError_t launch_reduce_splits(const float* part, int64_t splits, int64_t n, float* out,
                                 cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 31) / 32;
    if (blocks > 152 * 16) blocks = 152 * 16;
    reduce_splits_kernel<<<(unsigned)blocks, kRedWarps * 32, 0, s>>>(part, splits, n, out);
    return cudaGetLastError();
}

}  // namespace mk
