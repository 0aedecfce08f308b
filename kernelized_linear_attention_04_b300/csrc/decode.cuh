// Streaming decode step of causal FAVOR+ ("Performer for vision", *What Is Performer?*, Key
// Feature 2: attention accumulated incrementally, which enables streaming inference; *Why
// Performer Matters*, Streaming and Sampling: autoregressive decoding with an unbounded context).
// Per head, for one new token with query q, key k and value v:
//   S <- f S + phi(k) v^T,   z <- f z + phi(k),   y = phi(q)^T S / phi(q)^T z,
// one step of the causal recurrence (the new token attends to itself and every earlier token).
//
// The m features are processed in blocks of 64, one CTA per (head, block), each block with its own
// stabilisers (all cancel in the ratio; the common 1/sqrt(m) is dropped, so the ReLU family's
// epsilon is scaled by sqrt(m)). Block b of a head keeps a running key constant st_b in the state: a
// new key whose largest exponent over the block, max_r (w_r . k^) - |k^|^2 / 2, exceeds it raises
// it, and f = exp(old - new) rescales the block's S and z (f = 0 for the first token). The query
// uses its largest exponent over the block, c_b. With num_b = phi_b(q)^T S_b and den_b = phi_b(q)^T z_b,
//   y = sum_b w_b num_b / sum_b w_b den_b,   w_b = exp(c_b + st_b - max_b' (c_b' + st_b')),
// which the last block of the head to finish computes (a per-head counter in the state, no waits).
//
// Each CTA reads and writes its 64 x d fp32 block of the state once (a memory-bound update) and
// reads its 64 rows of Omega from L2.
#pragma once

#include "common.cuh"

namespace favor {
namespace dec {

constexpr int kThreads = 256;

// Block-wide reductions over the CTA's kThreads threads; `red` holds kThreads / 32 floats.
__device__ __forceinline__ float block_reduce_max(float v, float* red) {
    v = warp_max(v);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
    return r;
}
__device__ __forceinline__ float block_reduce_sum(float v, float* red) {
    v = warp_sum(v);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) r += red[w];  // fixed order
    return r;
}

constexpr int kBlk = 64;  // features per CTA

// State of every head: S [BH][m][D], z [BH][m], stab [BH][m/64] (fp32; -inf before the first
// token), partials [BH][m/64][D + 2], counter [BH] (u32; 0 between steps).
__global__ void decode_init(float* __restrict__ S, float* __restrict__ z, float* __restrict__ stab,
                            unsigned* __restrict__ cnt, int64_t nS, int64_t nz, int64_t nst, int64_t nh) {
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, di = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = i0; i < nS; i += di) S[i] = 0.f;
    for (int64_t i = i0; i < nz; i += di) z[i] = 0.f;
    for (int64_t i = i0; i < nst; i += di) stab[i] = -INFINITY;
    for (int64_t i = i0; i < nh; i += di) cnt[i] = 0u;
}

// Shared memory: q^, k^, v (D each), phi(q), phi(k) (64 each), numerator partials (4 kThreads),
// reduction scratch (kThreads / 32).
template <int D>
constexpr size_t decode_smem_floats() {
    return 3 * (size_t)D + 2 * kBlk + 4 * kThreads + kThreads / 32;
}

// 8 consecutive elements of a row of Omega as fp32 (one 16-byte load for bf16, two for fp32).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Grid (B*H heads, m / 64 blocks), kThreads threads.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    decode_step(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ Om,
                T* __restrict__ y, float* __restrict__ S, float* __restrict__ z, float* __restrict__ stabs,
                float* __restrict__ part, unsigned* __restrict__ cnt, int m, int kind, float relu_eps_s, float scale) {
    static_assert(kThreads % (D / 4) == 0 && D % 64 == 0 && kBlk % (kThreads / (D / 4)) == 0 && kBlk <= kThreads,
                  "rows of D/4 float4 columns; Omega rows of 8 x 16 bytes; one z entry per thread");
    extern __shared__ float sm[];
    float* sq = sm;            // scale * q
    float* sk = sq + D;        // scale * k
    float* sv = sk + D;        // v
    float* pq = sv + D;        // phi(q) of the block's 64 features
    float* pk = pq + kBlk;     // phi(k)
    float* nump = pk + kBlk;   // [kThreads / (D / 4)][D] = 4 kThreads numerator partials
    float* red = nump + 4 * kThreads;
    __shared__ bool s_last;
    const int nb = m / kBlk;
    const int blk = blockIdx.y;
    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    const bool exp_kind = kind == kKindExp;
    const int f0 = blk * kBlk;  // first feature of this block
    q += bh * D;
    k += bh * D;
    v += bh * D;
    y += bh * D;
    S += (bh * (int64_t)m + f0) * D;
    z += bh * (int64_t)m + f0;

    // the block's state does not depend on the new token: its loads go out first, so that their
    // latency overlaps the token and Omega loads and the projections. Thread tid keeps columns
    // c4 .. c4 + 3 (c4 = 4 (tid mod D/4)) of the rows tid / (D/4) + i kThreads / (D/4).
    constexpr int kTpr = D / 4;
    constexpr int kRows = kThreads / kTpr;
    constexpr int kPer = kBlk / kRows;
    const int c4 = 4 * (tid % kTpr), r0s = tid / kTpr;
    float4 xs[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) xs[i] = *reinterpret_cast<const float4*>(S + (int64_t)(r0s + i * kRows) * D + c4);
    const float zold = tid < kBlk ? z[tid] : 0.f;

    for (int c = tid; c < D; c += kThreads) {
        sq[c] = scale * to_f32(q[c]);
        sk[c] = scale * to_f32(k[c]);
        sv[c] = to_f32(v[c]);
    }
    __syncthreads();
    // |k^|^2 / 2 (every warp computes it from shared memory)
    float hk = 0.f;
    for (int c = tid % 32; c < D; c += 32) hk = fmaf(sk[c], sk[c], hk);
    hk = 0.5f * warp_sum(hk);

    // projections u_r = w_r . x^ of the query and the key for the block's rows: a row of Omega per
    // group of 8 lanes, D / 8 consecutive elements per lane (coalesced 16-byte loads), shuffle sums
    constexpr int kLpr = 8;
    constexpr int kEl = D / kLpr;
    const int lr = (tid % 32) / kLpr, lc = tid % kLpr;
    float qmax = -INFINITY, kmax = -INFINITY;
    for (int r0 = (tid / 32) * (32 / kLpr); r0 < kBlk; r0 += kThreads / kLpr) {
        const int r = r0 + lr;
        const T* w = Om + (int64_t)(f0 + r) * D + lc * kEl;
        float uq = 0.f, uk = 0.f;
#pragma unroll
        for (int e = 0; e < kEl; e += 8) {
            float x[8];
            load8(w + e, x);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uq = fmaf(x[i], sq[lc * kEl + e + i], uq);
                uk = fmaf(x[i], sk[lc * kEl + e + i], uk);
            }
        }
#pragma unroll
        for (int o = kLpr / 2; o > 0; o >>= 1) {
            uq += __shfl_xor_sync(0xffffffffu, uq, o);
            uk += __shfl_xor_sync(0xffffffffu, uk, o);
        }
        if (lc == 0) {
            pq[r] = uq;
            pk[r] = uk;
        }
        qmax = fmaxf(qmax, uq);
        kmax = fmaxf(kmax, uk);
    }
    __syncthreads();
    float f = 1.f, new_stab = 0.f;
    if (exp_kind) {
        qmax = block_reduce_max(qmax, red);
        kmax = block_reduce_max(kmax, red) - hk;  // the new key's largest exponent in this block
        const float old = stabs[bh * nb + blk];
        new_stab = fmaxf(old, kmax);
        f = old == -INFINITY ? 0.f : exp_shift(old, new_stab);
    }
    for (int r = tid; r < kBlk; r += kThreads) {
        if (exp_kind) {
            pq[r] = exp_shift(pq[r], qmax);
            pk[r] = exp_shift(pk[r] - hk, new_stab);
        } else {
            pq[r] = phi_plain(pq[r], kind, 1.f, relu_eps_s);
            pk[r] = phi_plain(pk[r], kind, 1.f, relu_eps_s);
        }
    }
    __syncthreads();

    // state update and the block's numerator (float4 stores)
    const float4 v4 = make_float4(sv[c4], sv[c4 + 1], sv[c4 + 2], sv[c4 + 3]);
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int r = r0s + i * kRows;
        float4* sp = reinterpret_cast<float4*>(S + (int64_t)r * D + c4);
        float4 x = xs[i];
        const float p = pk[r], g = pq[r];
        x.x = fmaf(f, x.x, p * v4.x);
        x.y = fmaf(f, x.y, p * v4.y);
        x.z = fmaf(f, x.z, p * v4.z);
        x.w = fmaf(f, x.w, p * v4.w);
        *sp = x;
        num.x = fmaf(g, x.x, num.x);
        num.y = fmaf(g, x.y, num.y);
        num.z = fmaf(g, x.z, num.z);
        num.w = fmaf(g, x.w, num.w);
    }
    float den = 0.f;
    if (tid < kBlk) {
        const float zr = fmaf(f, zold, pk[tid]);
        z[tid] = zr;
        den = pq[tid] * zr;
    }
    *reinterpret_cast<float4*>(nump + (tid / kTpr) * D + c4) = num;
    den = block_reduce_sum(den, red);  // its barriers also publish nump
    float* mine = part + (bh * nb + blk) * (int64_t)(D + 2);
    if (tid < D) {
        float acc = 0.f;
#pragma unroll 8
        for (int g = 0; g < kRows; ++g) acc += nump[g * D + tid];  // fixed order
        mine[tid] = acc;
    }
    if (tid == 0) {
        mine[D] = den;
        mine[D + 1] = exp_kind ? qmax + new_stab : 0.f;  // log of the block's weight, up to a common constant
        if (exp_kind) stabs[bh * nb + blk] = new_stab;
    }
    // the last block of the head to finish combines the partials
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(cnt + bh, 1u) == (unsigned)(nb - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* hp = part + bh * nb * (int64_t)(D + 2);
    float M = -INFINITY;
    for (int b = 0; b < nb; ++b) M = fmaxf(M, __ldcg(hp + b * (D + 2) + D + 1));
    if (tid < D) {
        float nsum = 0.f, dsum = 0.f;
        for (int b = 0; b < nb; ++b) {  // fixed order
            const float wb = exp_shift(__ldcg(hp + b * (D + 2) + D + 1), M);
            nsum = fmaf(wb, __ldcg(hp + b * (D + 2) + tid), nsum);
            dsum = fmaf(wb, __ldcg(hp + b * (D + 2) + D), dsum);
        }
        store_elem(y + tid, nsum / dsum);
    }
    if (tid == 0) cnt[bh] = 0u;  // ready for the next step (launches on a stream run in order)
}

}  // namespace dec
}  // namespace favor
