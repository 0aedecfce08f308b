// Shared device helpers of the FAVOR+ kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace favor {

constexpr int kKindExp = 0;
constexpr int kKindRelu = 1;
constexpr int kStabNone = 0;
constexpr int kStabRow = 1;
constexpr int kStabHead = 2;

constexpr float kLog2e = 1.4426950408889634f;

// Device error word: set (never trapped on) by a kernel whose bounded wait gave up.
constexpr unsigned kDevErrTimeout = 1u;
__device__ unsigned int g_favor_error;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Order-preserving map float -> uint32 (monotone; 0 is below every float), for atomicMax on floats.
__device__ __forceinline__ unsigned ordered_encode(float f) {
    unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ordered_decode(unsigned e) {
    unsigned u = (e & 0x80000000u) ? (e & 0x7FFFFFFFu) : ~e;
    return __uint_as_float(u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// exp(u - stab) for the exp family, evaluated as 2^((u - stab) * log2 e).
__device__ __forceinline__ float exp_shift(float u, float stab) { return exp2f((u - stab) * kLog2e); }

}  // namespace favor
