/*
 * synth.c -- seeded, counter-based generator of synthetic input tensors.
 *
 * This file holds no arithmetic of the MoE layer: it only turns
 * (seed, tensor id, attempt, element index) into a normal deviate and rounds it
 * to the stored type.  Both the CUDA path's callers and the CPU oracle's tests
 * read the bytes it writes, so both see identical inputs.
 *
 * Definition (fixed; changing it changes every synthetic workload):
 *   splitmix64(z): z += 0x9E3779B97F4A7C15;
 *                  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                  z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *                  return z ^ (z >> 31)
 *   stream base  : b = splitmix64(splitmix64(splitmix64(seed) + tensor_id) + attempt)
 *   uniforms     : u1 = (splitmix64(b + 2i) >> 11) * 2^-53,
 *                  u2 = (splitmix64(b + 2i + 1) >> 11) * 2^-53        (in [0, 1))
 *   normal       : z_i = sqrt(-2 ln(1 - u1)) * cos(2 pi u2)      (Box-Muller, fp64)
 *   stored value : scale * z_i in fp64, rounded to fp32 (round-to-nearest-even),
 *                  and for bf16 storage that fp32 value rounded again RNE to bf16.
 */
#include <math.h>
#include <stdint.h>

static inline uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t tensor_id, uint64_t attempt) {
    return splitmix64(splitmix64(splitmix64(seed) + tensor_id) + attempt);
}

static inline double normal_at(uint64_t base, uint64_t i) {
    const double two_m53 = 1.0 / 9007199254740992.0;
    const double u1 = (double)(splitmix64(base + 2 * i) >> 11) * two_m53;
    const double u2 = (double)(splitmix64(base + 2 * i + 1) >> 11) * two_m53;
    const double two_pi = 6.283185307179586476925286766559;
    return sqrt(-2.0 * log(1.0 - u1)) * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    union {
        float f;
        uint32_t u;
    } v;
    v.f = f;
    const uint32_t lsb = (v.u >> 16) & 1u;
    return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

/* Elements [start, start+count) of tensor `tensor_id`, scaled by `scale`, as fp32. */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t attempt, int64_t start,
                      int64_t count, double scale, float *out) {
    const uint64_t b = stream_base(seed, tensor_id, attempt);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) out[i] = (float)(scale * normal_at(b, (uint64_t)(start + i)));
}

/* Same values as synth_normal_f32, then rounded RNE to bf16 (raw 16-bit patterns). */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t attempt, int64_t start,
                       int64_t count, double scale, uint16_t *out) {
    const uint64_t b = stream_base(seed, tensor_id, attempt);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = f32_to_bf16_rne((float)(scale * normal_at(b, (uint64_t)(start + i))));
}

/* Raw uniform 64-bit words (for tests of the generator itself). */
void synth_raw_u64(uint64_t seed, uint64_t tensor_id, uint64_t attempt, int64_t start,
                   int64_t count, uint64_t *out) {
    const uint64_t b = stream_base(seed, tensor_id, attempt);
    for (int64_t i = 0; i < count; ++i) out[i] = splitmix64(b + (uint64_t)(start + i));
}

/* The mixing function alone (for a test against its published outputs). */
uint64_t synth_splitmix64(uint64_t z) { return splitmix64(z); }
