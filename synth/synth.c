/*
 * Seeded, counter-based synthetic input generator.
 *
 * This module produces the test and benchmark inputs for both the fp64 oracle
 * and the GPU library.  It holds none of the MTTKRP arithmetic: it only draws
 * random numbers and, for the structured workloads, evaluates a tensor given
 * as a sum of rank-one terms (that is how those workloads are defined).
 *
 * Every value is a pure function of (seed, stream, index), so the output is
 * bitwise identical whatever the number of OpenMP threads.
 *
 *  - mix64 is the SplitMix64 output function (Steele, Lea, Flood,
 *    "Fast splittable pseudorandom number generators", OOPSLA 2014; the
 *    constants are those of the published definition).
 *  - draw(seed, stream, i) = mix64(key(seed, stream) + (i + 1) * GOLDEN), i.e.
 *    element i of the SplitMix64 sequence whose state starts at key.
 *  - uniform [0,1): the top 53 bits of a draw times 2^-53.
 *  - normal: Box-Muller in fp64 with the pair of draws (2i, 2i+1).
 *
 * Everything is computed in fp64 on the host and rounded once to fp32 where
 * an fp32 output is requested.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* SplitMix64 sequence: state += GOLDEN, then output mix64(state). */
uint64_t synth_splitmix_next(uint64_t* state) {
    *state += GOLDEN;
    return synth_mix64(*state);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return synth_mix64(synth_mix64(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL));
}

uint64_t synth_draw(uint64_t seed, uint64_t stream, uint64_t i) {
    return synth_mix64(stream_key(seed, stream) + (i + 1) * GOLDEN);
}

static inline double u01(uint64_t key, uint64_t i) {
    return (double)(synth_mix64(key + (i + 1) * GOLDEN) >> 11) * 0x1.0p-53;
}

/* uniform in (0, 1]: used for the logarithm in Box-Muller. */
static inline double u01_open0(uint64_t key, uint64_t i) {
    return (double)((synth_mix64(key + (i + 1) * GOLDEN) >> 11) + 1) * 0x1.0p-53;
}

static inline double normal01(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double a = u01_open0(key, 2 * i);
    double b = u01(key, 2 * i + 1);
    return sqrt(-2.0 * log(a)) * cos(two_pi * b);
}

void synth_uniform_f64(uint64_t seed, uint64_t stream, int64_t n, double lo, double hi,
                       double* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = lo + (hi - lo) * u01(key, (uint64_t)i);
}

void synth_uniform_f32(uint64_t seed, uint64_t stream, int64_t n, double lo, double hi,
                       float* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * u01(key, (uint64_t)i));
}

void synth_normal_f64(uint64_t seed, uint64_t stream, int64_t n, double mean, double stddev,
                      double* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = mean + stddev * normal01(key, (uint64_t)i);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double mean, double stddev,
                      float* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(mean + stddev * normal01(key, (uint64_t)i));
}

/*
 * Evaluate a d-way tensor given as a sum of S rank-one terms,
 *   Y(i_0..i_{d-1}) = sum_s prod_n B_n(i_n, s)   (+ optional N(0, noise_std) noise),
 * with B_n stored I_n x S row-major in fp64.  Y is written C-order (last index
 * fastest).  The noise uses (seed, noise_stream); noise_std = 0 disables it.
 * Output in fp32 (out32) or fp64 (out64); exactly one must be non-NULL.
 */
int synth_rank_sum(int d, const int64_t* dims, int64_t S, const double* const* B,
                   double noise_std, uint64_t seed, uint64_t noise_stream, float* out32,
                   double* out64) {
    if (d < 1 || d > 16 || S < 0 || (out32 == NULL) == (out64 == NULL)) return -1;
    int64_t total = 1;
    for (int n = 0; n < d; ++n) {
        if (dims[n] < 1) return -1;
        total *= dims[n];
    }
    uint64_t key = stream_key(seed, noise_stream);
    int64_t last = dims[d - 1];
    int64_t nfib = total / last;
#pragma omp parallel
    {
        double* prefix = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
#pragma omp for schedule(static)
        for (int64_t f = 0; f < nfib; ++f) {
            /* decode fibre index f into (i_0..i_{d-2}); the last index runs inside */
            int64_t rem = f;
            int64_t idx[16];
            for (int n = d - 2; n >= 0; --n) {
                idx[n] = rem % dims[n];
                rem /= dims[n];
            }
            for (int64_t s = 0; s < S; ++s) {
                double p = 1.0;
                for (int n = 0; n < d - 1; ++n) p *= B[n][idx[n] * S + s];
                prefix[s] = p;
            }
            for (int64_t j = 0; j < last; ++j) {
                double v = 0.0;
                for (int64_t s = 0; s < S; ++s) v += prefix[s] * B[d - 1][j * S + s];
                int64_t lin = f * last + j;
                if (noise_std != 0.0) v += noise_std * normal01(key, (uint64_t)lin);
                if (out32)
                    out32[lin] = (float)v;
                else
                    out64[lin] = v;
            }
        }
        free(prefix);
    }
    return 0;
}
