/*
 * Seeded synthetic input generator.
 *
 * This file only draws numbers: it holds none of the epilogue's arithmetic
 * (no products, sums, norms or rounding of results).  Both the CPU oracle's
 * tests and the GPU path's tests/bench take their inputs from here, so the two
 * sides always see identical bytes.
 *
 * Generator definition (counter based, so any element can be drawn alone and
 * the loops parallelise without changing a single value):
 *
 *   mix(z)        SplitMix64 finaliser (Steele, Lea, Flood 2014):
 *                   z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *                   z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   stream key    key = mix(mix(seed) ^ (tensor_id * 0xD1B54A32D192ED03)
 *                            ^ (rank * 0x8CB92BA72F3D8DD7))
 *   raw word i    w(i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 *                 (the i-th output of a SplitMix64 stream seeded with key)
 *   uniform       u(i) = (w(i) >> 11) * 2^-53            in [0, 1)
 *   normal        Box-Muller on the pair (2j, 2j+1):
 *                   rho = sqrt(-2 ln(1 - u(2j))), th = 2 pi u(2j+1)
 *                   z(2j) = rho cos th,  z(2j+1) = rho sin th
 *   to bf16       fp64 -> fp32 by the C cast (round to nearest even), then
 *                 fp32 -> bf16 round to nearest even on the bit pattern.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27; z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

uint64_t synth_stream_key(uint64_t seed, uint64_t tensor_id, uint64_t rank) {
    return mix64(mix64(seed) ^ (tensor_id * 0xD1B54A32D192ED03ull) ^ (rank * 0x8CB92BA72F3D8DD7ull));
}

static inline uint64_t word_at(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
}

static inline double u01_at(uint64_t key, uint64_t i) {
    return (double)(word_at(key, i) >> 11) * 0x1.0p-53;
}

static inline double normal_at(uint64_t key, uint64_t i) {
    uint64_t j = i >> 1;
    double u1 = 1.0 - u01_at(key, 2 * j);
    double u2 = u01_at(key, 2 * j + 1);
    double rho = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? rho * sin(th) : rho * cos(th);
}

static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x007FFFFFu)) return (uint16_t)((x >> 16) | 0x40u);
    uint32_t lsb = (x >> 16) & 1u;
    x += 0x7FFFu + lsb;
    return (uint16_t)(x >> 16);
}

/* Raw 64-bit words, for tests of the generator itself. */
void synth_words(uint64_t key, uint64_t start, int64_t n, uint64_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = word_at(key, start + (uint64_t)i);
}

/* bf16 ~ U[lo, hi). */
void synth_uniform_bf16(uint64_t key, int64_t n, double lo, double hi, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double v = lo + (hi - lo) * u01_at(key, (uint64_t)i);
        out[i] = f32_to_bf16_bits((float)v);
    }
}

/* bf16 ~ mean + std * N(0,1). */
void synth_normal_bf16(uint64_t key, int64_t n, double mean, double std, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double v = mean + std * normal_at(key, (uint64_t)i);
        out[i] = f32_to_bf16_bits((float)v);
    }
}

/* fp32 ~ mean + std * N(0,1). */
void synth_normal_f32(uint64_t key, int64_t n, double mean, double std, float *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + std * normal_at(key, (uint64_t)i));
}

/* Overwrite a fraction p of a bf16 array with the bit pattern `bits`
 * (element i is chosen when u(i) of the stream `key` is below p). Returns the
 * number of elements overwritten. */
int64_t synth_inject_bf16(uint64_t key, int64_t n, double p, uint16_t bits, uint16_t *data) {
    int64_t hit = 0;
#pragma omp parallel for schedule(static) reduction(+ : hit)
    for (int64_t i = 0; i < n; ++i) {
        if (u01_at(key, (uint64_t)i) < p) { data[i] = bits; ++hit; }
    }
    return hit;
}
