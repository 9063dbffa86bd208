// Power-of-two scaling of the two-term fp16 split (device helpers shared by the
// tensor-core kernels and the table kernels).
//
// The split writes x = v * s as hi = fp16(x) and lo = fp16(x - hi), where s is
// the power of two that maps the largest magnitude m of the values it scales
// into [2^13, 2^14): fp16 holds the scaled values with room to spare, and their
// lo parts stay normal down to 2^-11 of the largest.  Scaling by powers of two
// is exact, so a kernel undoes it exactly at the end.
//
// Y is scaled per slab of mode 0 (the entries with one value of i_0): each slab
// by the power of two of its own largest magnitude, so a slab whose entries are
// far below the rest of the tensor keeps its precision.  Mode 0 is never summed
// inside one tensor-memory accumulation: for the mode-0 MTTKRP it is the output
// row (the epilogue divides each row by its slab's scale), for every other mode
// it is a pre mode, whose factor-product table row G(pi, :) is multiplied by
// s_global / s_slab(pi) (a power of two <= 1), so that every accumulated term
// carries the global scale, which the epilogue divides out.
#pragma once

#include <cstdint>

namespace mk {

// s for the largest magnitude m (fp32 bits of a non-negative value); m = 0 or a
// non-finite m: 1 (nothing to scale; non-finite values propagate).  A subnormal
// m uses the exponent of its leading bit; the scale is clamped to the fp32 range.
__device__ __forceinline__ float pow2_scale(uint32_t mbits) {
    const uint32_t m = mbits & 0x7FFFFFFFu;
    int e = (int)(m >> 23);                       // biased exponent
    if (m == 0 || e == 255) return 1.f;
    if (e == 0) e = 1 - (__clz((int)m) - 9);      // subnormal: leading bit of the mantissa
    int se = 127 + 13 - (e - 127);               // biased exponent of 2^(13 - (e - 127))
    se = se < 1 ? 1 : (se > 254 ? 254 : se);
    return __uint_as_float((uint32_t)se << 23);
}

// 1 / x for x = 2^k with a biased exponent in [1, 254] (what pow2_scale
// returns), exactly: 2^-k, subnormal (2^-127) for the largest x
__device__ __forceinline__ float pow2_recip(float x) {
    const uint32_t e = __float_as_uint(x) >> 23;
    return __uint_as_float(e <= 253u ? (254u - e) << 23 : 0x00400000u);
}

// Scale of slab s: from the slab's own largest magnitude, or the global one for
// an all-zero slab (whose images are zero whatever the scale).
__device__ __forceinline__ float slab_scale(const uint32_t* slab_bits, int64_t s, uint32_t gmax_bits) {
    const uint32_t m = slab_bits[s];
    return pow2_scale(m != 0 ? m : gmax_bits);
}

}  // namespace mk
