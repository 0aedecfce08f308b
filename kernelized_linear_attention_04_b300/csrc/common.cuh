// Shared device helpers of the FAVOR+ kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace favor {

constexpr int kKindExp = 0;
constexpr int kKindRelu = 1;
constexpr int kKindElu = 2;
constexpr int kStabNone = 0;
constexpr int kStabRow = 1;
constexpr int kStabHead = 2;

constexpr float kLog2e = 1.4426950408889634f;

// Device error word: set (never trapped on) by a kernel whose bounded wait gave up, or, in a debug
// build, whose bounds check failed.
constexpr unsigned kDevErrTimeout = 1u;
constexpr unsigned kDevErrBounds = 2u;
__device__ unsigned int g_favor_error;

// Debug builds (-DFAVOR_DEBUG, the stand-in for a memory checker) test the index of every
// computed-address access to global memory, shared memory and tensor memory against its buffer:
// a failed check records kDevErrBounds in the device error word and the guarded access is skipped.
// Release builds compile the checks away (the guard is the constant true).
#ifdef FAVOR_DEBUG
__device__ __forceinline__ bool favor_in_bounds(bool ok) {
    if (!ok) atomicOr(&g_favor_error, kDevErrBounds);
    return ok;
}
#define FAVOR_IN_BOUNDS(cond) (::favor::favor_in_bounds(static_cast<bool>(cond)))
#else
#define FAVOR_IN_BOUNDS(cond) true
#endif

// Test hook, 0 (off) unless a caller arms it through favor_test_set_wait_limit: while it holds a
// nonzero value, every bounded wait gives up after that many nanoseconds instead of its normal limit,
// and the causal tensor-core scan withholds the first arrival its MMA issuer waits for, so that the
// timeout path (error word, abort of the other roles, TMA drain, TMEM release) runs on demand
// without any fault or hang.
__device__ unsigned long long g_favor_test_wait_ns;

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

// Feature of a family without a stabiliser, from the projection a: generalized ReLU
// max(0, a) * g + eps (a = w_r . x^); elu + 1 (whose projection is the identity and whose input is
// the raw x, so a = x_r): a + 1 for a > 0, exp(a) otherwise (g and eps unused).
__device__ __forceinline__ float phi_plain(float a, int kind, float g, float eps) {
    if (kind != kKindElu) return fmaxf(a, 0.f) * g + eps;
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fminf(a, 0.f) * kLog2e));
    return a > 0.f ? a + 1.f : e;
}

// exp(u - stab) for the exp family, evaluated as 2^((u - stab) * log2 e).
__device__ __forceinline__ float exp_shift(float u, float stab) { return exp2f((u - stab) * kLog2e); }

}  // namespace favor
