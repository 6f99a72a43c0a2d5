/*
 * Seeded synthetic operands for the dense projection Y = X·Wᵀ (+ bias).
 *
 * The same generator as synth/__init__.py (SplitMix64 counter stream,
 * Box–Muller, fp64 → fp32 → bf16 round-to-nearest-even), written in C so the
 * largest weight matrices (hundreds of millions of elements) are drawn in about
 * a second.  It contains no step of the projection itself.
 *
 * SplitMix64: G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; counter form: output j of the stream seeded with s
 * is mix(s + (j+1)·0x9E3779B97F4A7C15).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_stream_seed(uint64_t seed, int tensor) {
    return synth_mix64(seed * 256ULL + (uint64_t)tensor);
}

static inline double synth_uniform(uint64_t s, uint64_t j) {
    uint64_t bits = synth_mix64(s + (j + 1ULL) * SYNTH_GAMMA) >> 11;
    return ((double)bits + 1.0) * 0x1.0p-53;
}

static inline uint16_t synth_bf16_rne(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)(((uint64_t)u + 0x7FFFu + lsb) >> 16);
}

/* The j-th standard normal of stream s (Box–Muller on the pair j & ~1). */
static inline double synth_normal_at(uint64_t s, uint64_t j) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t pair = j & ~1ULL;
    double u1 = synth_uniform(s, pair);
    double u2 = synth_uniform(s, pair + 1ULL);
    double r = sqrt(-2.0 * log(u1));
    double th = two_pi * u2;
    return (j & 1ULL) ? r * sin(th) : r * cos(th);
}

/* out[i] = bf16(std · normal_j) for j = first + i, i < count. */
void synth_normal_bf16(uint64_t seed, int tensor, int64_t first, int64_t count,
                       double std, uint16_t *out) {
    const uint64_t s = synth_stream_seed(seed, tensor);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = synth_bf16_rne(synth_normal_at(s, (uint64_t)(first + i)) * std);
}

/* out[i] = fp32(std · normal_j) (round to nearest): fp32 weights. */
void synth_normal_f32(uint64_t seed, int tensor, int64_t first, int64_t count,
                      double std, float *out) {
    const uint64_t s = synth_stream_seed(seed, tensor);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = (float)(synth_normal_at(s, (uint64_t)(first + i)) * std);
}
