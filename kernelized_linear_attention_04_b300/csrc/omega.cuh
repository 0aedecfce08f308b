// On-device construction of the random projection Omega [m x d] ("Performer for vision", *What Is
// Performer?*, Orthogonal Features: the rows of Omega are drawn Gaussian and made exactly orthogonal
// within each block of d rows, which lowers the variance of the softmax-kernel estimate; the
// "Performer" paper note, FAVOR+ section: positive orthogonal random features). Redrawing Omega
// during training is a call of this kernel with a new seed.
//
// Definition built here, for blocks b = 0 .. ceil(m/d) - 1 of d rows each:
//   G_b     d x d iid N(0, 1): element (b d + i) d + j of the Gaussian stream (seed, 4)
//   E_b     the rows of G_b orthonormalised in order by modified Gram-Schmidt
//   chi_r   || (x_{r d}, ..., x_{r d + d - 1}) ||, x the Gaussian stream (seed, 5): the length of an
//           independent N(0, I_d) vector, so row r of Omega is again marginally N(0, I_d)
//   Omega_r = chi_r * E_{b, i} for r = b d + i < m  (rounded fp64 -> fp32 -> bf16 for bf16 output)
// Unstructured (orthogonal = 0): Omega_r = G_{b, i}, the iid Gaussian rows.
//
// The Gaussian stream is a counter-based generator (each element a function of seed, stream and
// index alone), written from the published definitions of its two halves: SplitMix64's finaliser
// (Steele, Lea and Flood) hashes (key + 2i) and (key + 2i + 1) into two uniforms, and the cosine
// branch of the Box-Muller transform turns them into one N(0, 1) sample.
//
// One CTA per block: the d x d block in shared memory as fp64, right-looking Gram-Schmidt (after row
// i is normalised every later row loses its component along it, so each row sees the projections
// of e_0, e_1, ... in order, as the left-looking form computes them), one warp per row, one barrier
// per row. Nothing waits on another CTA.
#pragma once

#include "common.cuh"

namespace favor {
namespace omg {

constexpr int kThreads = 256;
constexpr uint64_t kStreamGauss = 4, kStreamChi = 5;

__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

// Key of stream `id` of a seed: the hashed seed, mixed with the stream id by an odd constant.
__host__ __device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t id) {
    return splitmix64(splitmix64(seed) ^ (id * 0xD1B54A32D192ED03ull));
}

// Element i of a stream: u1 in (0, 1] and u2 in [0, 1) from the top 53 bits of two hashes, then
// sqrt(-2 ln u1) cos(2 pi u2).
__device__ __forceinline__ double gauss_at(uint64_t key, uint64_t i) {
    const double two_m53 = 1.0 / 9007199254740992.0;
    const uint64_t h1 = splitmix64(key + 2 * i), h2 = splitmix64(key + 2 * i + 1);
    const double u1 = (double)((h1 >> 11) + 1) * two_m53;
    const double u2 = (double)(h2 >> 11) * two_m53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void store_round(float* p, double x) { *p = __double2float_rn(x); }
__device__ __forceinline__ void store_round(__nv_bfloat16* p, double x) {
    *p = __float2bfloat16_rn(__double2float_rn(x));
}

template <int D>
constexpr size_t omega_smem_bytes() {
    return sizeof(double) * ((size_t)D * D + D);
}

// Grid: ceil(m / D) CTAs of kThreads threads; dynamic shared memory omega_smem_bytes<D>().
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    omega_build(uint64_t key_g, uint64_t key_chi, int m, int orthogonal, T* __restrict__ Om) {
    static_assert(D % 32 == 0, "rows are processed a warp at a time");
    extern __shared__ double se[];  // [D][D] the block, then chi [D]
    double* chi = se + D * D;
    constexpr int kWarps = kThreads / 32;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t row0 = (int64_t)blockIdx.x * D;
    const int64_t left = (int64_t)m - row0;
    const int rows = left < D ? (int)left : D;  // rows of this block that Omega keeps

    for (int e = threadIdx.x; e < D * D; e += kThreads) se[e] = gauss_at(key_g, (uint64_t)(row0 * D + e));
    if (orthogonal) {
        for (int i = warp; i < rows; i += kWarps) {
            double s = 0.0;
            for (int j = lane; j < D; j += 32) {
                const double x = gauss_at(key_chi, (uint64_t)((row0 + i) * D + j));
                s = fma(x, x, s);
            }
            s = warp_sum_d(s);
            if (lane == 0) chi[i] = sqrt(s);
        }
    }
    __syncthreads();

    if (orthogonal) {
        // normalise row 0; afterwards the warp that finishes row i + 1's last projection normalises it
        if (warp == 0) {
            double s = 0.0;
            for (int j = lane; j < D; j += 32) s = fma(se[j], se[j], s);
            const double nrm = sqrt(warp_sum_d(s));
            for (int j = lane; j < D; j += 32) se[j] = se[j] / nrm;
        }
        __syncthreads();
        // only the rows Omega keeps need their projections: row k depends on rows < k alone
        for (int i = 0; i + 1 < rows; ++i) {
            const double* ei = se + i * D;
            for (int k = i + 1 + warp; k < rows; k += kWarps) {
                double* vk = se + k * D;
                double p = 0.0;
                for (int j = lane; j < D; j += 32) p = fma(vk[j], ei[j], p);
                p = warp_sum_d(p);
                double s = 0.0;
                for (int j = lane; j < D; j += 32) {
                    const double x = fma(-p, ei[j], vk[j]);
                    vk[j] = x;
                    s = fma(x, x, s);
                }
                if (k == i + 1) {  // row i + 1 is now orthogonal to rows 0 .. i: normalise it
                    const double nrm = sqrt(warp_sum_d(s));
                    for (int j = lane; j < D; j += 32) vk[j] = vk[j] / nrm;
                }
            }
            __syncthreads();
        }
    }

    for (int e = threadIdx.x; e < rows * D; e += kThreads) {
        const int i = e / D;
        const double x = orthogonal ? se[e] * chi[i] : se[e];
        store_round(Om + row0 * D + e, x);
    }
}

}  // namespace omg
}  // namespace favor
