/*
 * Seeded synthetic input generator shared by the CPU oracle, the tests and the
 * benchmark.  It holds none of the decoder's arithmetic: it only draws numbers.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; finaliser constants as published by Vigna)
 * used in counter mode.  A tensor is identified by a 64-bit id; its stream
 * state starts at key = mix(seed ^ mix(id)) and the k-th output (k >= 1) is
 * mix(key + k * GOLDEN).  Element i of a tensor consumes outputs 2i+1 and 2i+2,
 * so any element can be drawn independently of the others (parallel fills are
 * bit-identical to serial ones, and a subset can be drawn on its own).
 *
 * Normals use the Box-Muller transform (cosine branch) in double precision,
 * then round to float (and from float to bfloat16 with round-to-nearest-even
 * for bf16 outputs).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(seed ^ mix64(tensor_id + GOLDEN));
}

static inline uint64_t draw(uint64_t key, uint64_t k) { return mix64(key + (k + 1) * GOLDEN); }

static inline double normal_at(uint64_t key, int64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t a = draw(key, 2 * (uint64_t)i);
    uint64_t b = draw(key, 2 * (uint64_t)i + 1);
    double u1 = ((double)(a >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0, 1] */
    double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);         /* [0, 1) */
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void synth_normal_f32(uint64_t seed, uint64_t tensor_id, int64_t n, double mean, double std,
                      float *out) {
    uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + std * normal_at(key, i));
}

void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, int64_t n, double mean, double std,
                       uint16_t *out) {
    uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne((float)(mean + std * normal_at(key, i)));
}

/* Uniform integers in [lo, hi] (inclusive); multiply-shift range reduction. */
void synth_uniform_int(uint64_t seed, uint64_t tensor_id, int64_t n, int32_t lo, int32_t hi,
                       int32_t *out) {
    uint64_t key = stream_key(seed, tensor_id);
    uint64_t range = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
    for (int64_t i = 0; i < n; ++i) {
        uint64_t r = draw(key, (uint64_t)i) >> 32;
        out[i] = lo + (int32_t)((r * range) >> 32);
    }
}

/* Raw 64-bit outputs, exposed so tests can check the generator against the
 * published SplitMix64 reference sequence. */
void synth_raw_u64(uint64_t state, int64_t n, uint64_t *out) {
    for (int64_t k = 0; k < n; ++k) out[k] = draw(state, (uint64_t)k);
}
