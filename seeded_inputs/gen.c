/*
 * Counter-based Gaussian generator shared by the fp64 oracle and the CUDA path's tests/bench.
 *
 * It holds no FAVOR+ arithmetic: it only turns (seed, tensor id, flat element index) into an
 * N(0, sigma^2) sample, optionally rounded to fp32 or bf16.  Any element of any tensor can be
 * regenerated on its own, so a single head of a multi-GB workload can be rebuilt for checking.
 *
 * Definition (both halves are published algorithms, written here from their definitions):
 *   key  = splitmix64(splitmix64(seed) ^ (tensor_id * 0xD1B54A32D192ED03))
 *   h1   = splitmix64(key + 2*i),  h2 = splitmix64(key + 2*i + 1)
 *   u1   = ((h1 >> 11) + 1) * 2^-53   in (0, 1]
 *   u2   =  (h2 >> 11)      * 2^-53   in [0, 1)
 *   z    = sqrt(-2 ln u1) * cos(2 pi u2)          (Box-Muller, cosine branch only)
 *   out  = sigma * z, rounded fp64 -> fp32 (round to nearest) -> bf16 (round to nearest even)
 * splitmix64 is Steele, Lea & Flood's SplitMix finaliser (the 64-bit variant Vigna publishes).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
    return splitmix64(splitmix64(seed) ^ (tensor_id * 0xD1B54A32D192ED03ull));
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const double two_m53 = 1.1102230246251565404236316680908203125e-16; /* 2^-53 */
    uint64_t h1 = splitmix64(key + 2 * i);
    uint64_t h2 = splitmix64(key + 2 * i + 1);
    double u1 = (double)((h1 >> 11) + 1) * two_m53;
    double u2 = (double)(h2 >> 11) * two_m53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void si_normal_f64(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t count, double sigma,
                   double* out) {
    uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) out[t] = sigma * normal_at(key, offset + (uint64_t)t);
}

void si_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t count, double sigma,
                   float* out) {
    uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) out[t] = (float)(sigma * normal_at(key, offset + (uint64_t)t));
}

void si_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t count, double sigma,
                    uint16_t* out) {
    uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t)
        out[t] = f32_to_bf16_rne((float)(sigma * normal_at(key, offset + (uint64_t)t)));
}

/* fp32 -> bf16 (round to nearest even), used to round a built Omega to the workload dtype. */
void si_f32_to_bf16(const float* in, int64_t count, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) out[t] = f32_to_bf16_rne(in[t]);
}

/* bf16 -> fp32 widening (exact). */
void si_bf16_to_f32(const uint16_t* in, int64_t count, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        uint32_t u = (uint32_t)in[t] << 16;
        memcpy(&out[t], &u, 4);
    }
}
