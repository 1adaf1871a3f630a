/*
 * Seeded synthetic inputs for causal linear attention workloads.
 *
 * This module holds no arithmetic of the attention method itself. It only
 * turns (seed, tensor id, flat index) into a normally distributed value and
 * stores it in the storage format of the workload (bf16 or fp32). Both the
 * float64 oracle and the CUDA library read the arrays it writes, so the two
 * sides always see bit-identical inputs.
 *
 * Generator (counter based, so any element can be regenerated on its own):
 *   key   = mix(seed * 0x9E3779B97F4A7C15 + mix(tensor_id + 0xD1B54A32D192ED03))
 *   r0,r1 = mix(key + (2 i + 1) * 0x9E3779B97F4A7C15), mix(key + (2 i + 2) * ...)
 *   u1    = ((r0 >> 11) + 1) * 2^-53      in (0, 1]
 *   u2    = (r1 >> 11) * 2^-53            in [0, 1)
 *   x     = scale * sqrt(-2 ln u1) * cos(2 pi u2)            (Box-Muller)
 * where mix() is the SplitMix64 finaliser (Steele, Lea, Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; constants as
 * published by Vigna for splitmix64). x is rounded to float (RNE) and then,
 * for bf16 storage, to bf16 with round-to-nearest-even on the float bits.
 */
#include <math.h>
#include <stdint.h>

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(seed * 0x9E3779B97F4A7C15ULL + mix64(tensor_id + 0xD1B54A32D192ED03ULL));
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const uint64_t g = 0x9E3779B97F4A7C15ULL;
    uint64_t r0 = mix64(key + (2 * i + 1) * g);
    uint64_t r1 = mix64(key + (2 * i + 2) * g);
    double u1 = (double)((r0 >> 11) + 1) * 0x1.0p-53;
    double u2 = (double)(r1 >> 11) * 0x1.0p-53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    union { float f; uint32_t u; } c;
    c.f = f;
    uint32_t u = c.u;
    if ((u & 0x7f800000u) == 0x7f800000u) {          /* inf / nan: keep, quiet nan */
        return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* Fill out[0..n) with shift + scale * N(0,1) for flat indices [first, first + n) of
 * tensor (seed, tensor_id), computed in float64 and rounded once to float32 (RNE),
 * then for bf16 storage to bf16 bits. dtype 0 writes float32, dtype 1 bf16 bits. */
void synth_normal_affine(uint64_t seed, uint64_t tensor_id, uint64_t first, int64_t n,
                         double scale, double shift, int dtype, void* out) {
    const uint64_t key = stream_key(seed, tensor_id);
    if (dtype == 1) {
        uint16_t* o = (uint16_t*)out;
        #pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < n; ++j)
            o[j] = f32_to_bf16_rne((float)(shift + scale * normal_at(key, first + (uint64_t)j)));
    } else {
        float* o = (float*)out;
        #pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < n; ++j)
            o[j] = (float)(shift + scale * normal_at(key, first + (uint64_t)j));
    }
}

/* The plain recipe: scale * N(0,1) (shift 0 adds an exact zero, so the values are
 * those of the affine form). */
void synth_normal(uint64_t seed, uint64_t tensor_id, uint64_t first, int64_t n,
                  double scale, int dtype, void* out) {
    synth_normal_affine(seed, tensor_id, first, n, scale, 0.0, dtype, out);
}

/* Widen bf16 bits to float32 (storage-format conversion only). */
void synth_bf16_to_f32(const uint16_t* in, float* out, int64_t n) {
    #pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        union { uint32_t u; float f; } c;
        c.u = (uint32_t)in[j] << 16;
        out[j] = c.f;
    }
}
