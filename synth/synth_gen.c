/*
 * Seeded synthetic-input generator shared by the tests, the bench and the
 * oracle-side checks.  It holds none of the MTP method's arithmetic: it only
 * turns (seed, stream, index) into numbers.
 *
 * Generator (counter based, so any sub-range can be regenerated alone):
 *   - SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): state_n = key + n * 0x9E3779B97F4A7C15,
 *     output = mix(state_n) with the published three-step xor-shift/multiply
 *     finaliser.
 *   - key = mix(mix(seed) ^ (stream * 0xD1B54A32D192ED03)), one key per tensor.
 *   - uniform double in [0,1): the top 53 bits times 2^-53.
 *   - normal: Box-Muller (Box & Muller 1958), cosine branch only, using the
 *     two outputs at counters 2i and 2i+1 for element i.
 *   - integers in [lo, hi): Lemire's multiply-shift on the top 32 bits.
 *   - bf16 outputs are the float32 value rounded to nearest-even on the upper
 *     16 bits.
 *
 * Portable C11 + OpenMP; no intrinsics, no architecture-specific code.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return sm_mix(sm_mix(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t n) {
    return sm_mix(key + (n + 1) * GOLDEN);
}

static inline double u01_open_low(uint64_t x) {   /* (0, 1] */
    return ((double)(x >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}
static inline double u01(uint64_t x) {            /* [0, 1) */
    return (double)(x >> 11) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = u01_open_low(draw(key, 2 * i));
    double u2 = u01(draw(key, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[j] = mean + std * N(0,1) for element index offset + j, as float32. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double mean, double std, float* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = (float)(mean + std * normal_at(key, offset + (uint64_t)j));
}

/* Same values as synth_normal_f32, rounded to bf16 (bit patterns). */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double mean, double std, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = f32_to_bf16_rne((float)(mean + std * normal_at(key, offset + (uint64_t)j)));
}

/* out[j] uniform integer in [lo, hi), hi - lo <= 2^32. */
void synth_uniform_i32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       int64_t lo, int64_t hi, int32_t* out) {
    uint64_t key = stream_key(seed, stream);
    uint64_t range = (uint64_t)(hi - lo);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        uint64_t x = draw(key, offset + (uint64_t)j) >> 32;
        out[j] = (int32_t)(lo + (int64_t)((x * range) >> 32));
    }
}

/* out[j] uniform double in [0, 1). */
void synth_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = u01(draw(key, offset + (uint64_t)j));
}

/* Raw 64-bit outputs, for tests of the generator itself. */
void synth_raw_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                   uint64_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t j = 0; j < n; ++j) out[j] = draw(key, offset + (uint64_t)j);
}

/* Plain SplitMix64 sequence from a state, for checking the published
 * reference values of the generator. */
void synth_splitmix64_seq(uint64_t state, int64_t n, uint64_t* out) {
    for (int64_t j = 0; j < n; ++j) {
        state += GOLDEN;
        out[j] = sm_mix(state);
    }
}
