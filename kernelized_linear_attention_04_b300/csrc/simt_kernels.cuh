// CUDA-core (SIMT) FAVOR+ kernels: fp32 FFMA arithmetic for fp32 or bf16 inputs.
//
// These carry the fp32 workloads (a 1e-4 max-abs tolerance rules out tf32/bf16 tensor cores) and
// every shape the tensor-core kernels do not take. Structure per operation:
//   features : one CTA per 16-token tile of one head; Omega streamed through shared memory in
//              64-row chunks; stabiliser per row in the CTA, per head through an atomic max.
//   state    : one CTA per (token split, head, 64-feature slice); phi(K) tile kept in shared memory,
//              S/z slice accumulated in registers with a running key stabiliser (rescaled when the
//              running max grows), partials written to the workspace.
//   combine  : one CTA per head, rescales partials to the head's largest stabiliser, sums in a
//              fixed order (deterministic).
//   readout  : one CTA per 16-token tile; phi(Q) with per-row stabiliser, Y = phi(Q)S / phi(Q)z.
//   causal   : one CTA per head walking 16-token sub-chunks in order; the prefix state lives in
//              the workspace (L2-resident), intra-chunk lower-triangular block in shared memory.
#pragma once

#include "common.cuh"

namespace favor {
namespace simt {

constexpr int kTok = 16;       // tokens per tile
constexpr int kThreads = 256;  // threads per CTA
constexpr int kOmChunk = 64;   // Omega rows per shared-memory chunk
constexpr int kSlice = 64;     // features per state slice

// Loads a [kTok, D] tile of rows [t0, t0+kTok) (rows >= n are zero) into shared memory as fp32.
template <typename T, int D>
__device__ __forceinline__ void load_tile(const T* __restrict__ X, int64_t n, int64_t t0, float* xs) {
    for (int e = threadIdx.x; e < kTok * D; e += kThreads) {
        int t = e / D, c = e % D;
        int64_t row = t0 + t;
        xs[t * D + c] = row < n ? to_f32(X[row * D + c]) : 0.f;
    }
}

// hs[t] = |x^_t|^2 / 2 = scale^2 |x_t|^2 / 2 for the kTok rows of a tile.
template <int D>
__device__ __forceinline__ void half_norms(const float* xs, float scale, float* hs) {
    int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int t = warp; t < kTok; t += kThreads / 32) {
        float s = 0.f;
        for (int c = lane; c < D; c += 32) s += xs[t * D + c] * xs[t * D + c];
        s = warp_sum(s);
        if (lane == 0) hs[t] = 0.5f * scale * scale * s;
    }
}

// ps[t * ldp + r] = scale * (w_r . x_t) for r in [r0, r0 + nr), Omega rows staged in `oms` chunks.
template <typename T, int D>
__device__ __forceinline__ void project_rows(const T* __restrict__ Om, int r0, int nr, const float* xs, float scale,
                                             float* oms, float* ps, int ldp) {
    for (int f0 = 0; f0 < nr; f0 += kOmChunk) {
        __syncthreads();
        for (int e = threadIdx.x; e < kOmChunk * D; e += kThreads) {
            int r = e / D, c = e % D;
            oms[r * (D + 1) + c] = to_f32(Om[(int64_t)(r0 + f0 + r) * D + c]);
        }
        __syncthreads();
        int r = threadIdx.x % kOmChunk;
        for (int t = threadIdx.x / kOmChunk; t < kTok; t += kThreads / kOmChunk) {
            float acc = 0.f;
#pragma unroll 16
            for (int c = 0; c < D; ++c) acc = fmaf(oms[r * (D + 1) + c], xs[t * D + c], acc);
            ps[t * ldp + f0 + r] = scale * acc;
        }
    }
    __syncthreads();
}

__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
    return r;
}

// ------------------------------------------------------------------------------------------------
// Feature map. Phi [BH, n, m] fp32. For STAB_HEAD the exponents are written and a second pass
// (features_head_apply) subtracts the head maximum gathered in head_max (ordered-encoded uints).
// ------------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) features_kernel(const T* __restrict__ X, const T* __restrict__ Om,
                                                            float* __restrict__ Phi, int64_t n, int m, int kind,
                                                            float relu_eps, int stab, float scale,
                                                            unsigned* __restrict__ head_max) {
    extern __shared__ float smem[];
    float* xs = smem;                          // kTok * D
    float* oms = xs + kTok * D;                // kOmChunk * (D + 1)
    float* ps = oms + kOmChunk * (D + 1);      // kTok * m
    float* hs = ps + kTok * m;                 // kTok
    const int64_t bh = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    X += bh * n * D;
    Phi += bh * n * m;

    load_tile<T, D>(X, n, t0, xs);
    __syncthreads();
    half_norms<D>(xs, scale, hs);
    project_rows<T, D>(Om, 0, m, xs, scale, oms, ps, m);
    const float inv_sqrt_m = rsqrtf((float)m);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float local_max = -INFINITY;
    for (int t = warp; t < kTok; t += kThreads / 32) {
        int64_t row = t0 + t;
        if (row >= n) continue;
        float* pr = ps + t * m;
        float* out = Phi + row * m;
        if (kind != kKindExp) {
            for (int r = lane; r < m; r += 32) out[r] = phi_plain(pr[r], kind, inv_sqrt_m, relu_eps);
            continue;
        }
        float rmax = -INFINITY;
        for (int r = lane; r < m; r += 32) {
            pr[r] -= hs[t];
            rmax = fmaxf(rmax, pr[r]);
        }
        rmax = warp_max(rmax);
        if (stab == kStabHead) {
            local_max = fmaxf(local_max, rmax);
            for (int r = lane; r < m; r += 32) out[r] = pr[r];
        } else {
            float st = stab == kStabRow ? rmax : 0.f;
            for (int r = lane; r < m; r += 32) out[r] = exp_shift(pr[r], st) * inv_sqrt_m;
        }
    }
    if (kind == kKindExp && stab == kStabHead && lane == 0 && local_max > -INFINITY)
        atomicMax(head_max + bh, ordered_encode(local_max));
}

__global__ void features_head_apply_kernel(float* __restrict__ Phi, int64_t per_head, int m,
                                           const unsigned* __restrict__ head_max) {
    const int64_t bh = blockIdx.y;
    const float st = ordered_decode(head_max[bh]);
    const float inv_sqrt_m = rsqrtf((float)m);
    float* p = Phi + bh * per_head;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < per_head; e += (int64_t)gridDim.x * blockDim.x)
        p[e] = exp_shift(p[e], st) * inv_sqrt_m;
}

// ------------------------------------------------------------------------------------------------
// Non-causal state: partial S (kSlice x D), z (kSlice) and key stabiliser per (split, head, slice).
// Workspace layout: pS [BH][splits][m][D], pz [BH][splits][m], pstab [BH][splits][m / kSlice].
// ------------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) state_kernel(const T* __restrict__ K, const T* __restrict__ V,
                                                         const T* __restrict__ Om, int64_t n, int m, int kind,
                                                         float relu_eps, float scale, int64_t tokens_per_split,
                                                         float* __restrict__ pS, float* __restrict__ pz,
                                                         float* __restrict__ pstab) {
    extern __shared__ float smem[];
    float* ks = smem;                         // kTok * D
    float* vs = ks + kTok * D;                // kTok * D
    float* oms = vs + kTok * D;               // kOmChunk * (D + 1)
    float* ps = oms + kOmChunk * (D + 1);     // kTok * kSlice
    float* hs = ps + kTok * kSlice;           // kTok
    float* red = hs + kTok;                   // 8
    const int split = blockIdx.x, splits = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int slice = blockIdx.z, slices = gridDim.z;
    const int r0 = slice * kSlice;
    const int64_t j0 = (int64_t)split * tokens_per_split;
    const int64_t j1 = min(n, j0 + tokens_per_split);
    K += bh * n * D;
    V += bh * n * D;
    const float inv_sqrt_m = rsqrtf((float)m);

    constexpr int kPerRow = kThreads / kSlice;  // threads per feature row
    constexpr int kCols = D / kPerRow;          // columns each of them accumulates
    const int my_r = threadIdx.x / kPerRow;     // feature within the slice
    const int my_c0 = (threadIdx.x % kPerRow) * kCols;
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
    float zacc = 0.f;
    float stab = -INFINITY;                   // running key stabiliser (exp family)

    for (int64_t t0 = j0; t0 < j1; t0 += kTok) {
        __syncthreads();
        load_tile<T, D>(K, j1, t0, ks);       // rows past the split end read as zero...
        load_tile<T, D>(V, j1, t0, vs);
        __syncthreads();
        half_norms<D>(ks, scale, hs);
        project_rows<T, D>(Om, r0, kSlice, ks, scale, oms, ps, kSlice);
        const int nvalid = (int)(j1 - t0 < kTok ? j1 - t0 : kTok);  // ...and get phi = 0 below
        if (kind == kKindExp) {
            float tmax = -INFINITY;
            for (int e = threadIdx.x; e < kTok * kSlice; e += kThreads) {
                int t = e / kSlice;
                float u = ps[e] - hs[t];
                ps[e] = u;
                if (t < nvalid) tmax = fmaxf(tmax, u);
            }
            tmax = block_max(tmax, red);
            if (tmax > stab) {                 // running max grew: rescale what is accumulated
                float f = stab == -INFINITY ? 0.f : exp_shift(stab, tmax);
#pragma unroll
                for (int c = 0; c < kCols; ++c) acc[c] *= f;
                zacc *= f;
                stab = tmax;
            }
            for (int e = threadIdx.x; e < kTok * kSlice; e += kThreads) {
                int t = e / kSlice;
                ps[e] = t < nvalid ? exp_shift(ps[e], stab) * inv_sqrt_m : 0.f;
            }
        } else {
            for (int e = threadIdx.x; e < kTok * kSlice; e += kThreads) {
                int t = e / kSlice;
                ps[e] = t < nvalid ? phi_plain(ps[e], kind, inv_sqrt_m, relu_eps) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int t = 0; t < kTok; ++t) {
            float p = ps[t * kSlice + my_r];
            zacc += p;
#pragma unroll
            for (int c = 0; c < kCols; ++c) acc[c] = fmaf(p, vs[t * D + my_c0 + c], acc[c]);
        }
    }
    const int64_t base = (bh * splits + split);
    float* outS = pS + (base * m + r0 + my_r) * D + my_c0;
#pragma unroll
    for (int c = 0; c < kCols; ++c) outS[c] = acc[c];
    if (my_c0 == 0) pz[base * m + r0 + my_r] = zacc;
    if (threadIdx.x == 0) pstab[base * slices + slice] = kind == kKindExp ? stab : 0.f;
}

// Sums the partial states of one head: S = sum_s exp(stab_s - M) S_s (fixed order), same for z.
// Grid: (head, chunk of kCombineChunk elements of S); chunk 0 also sums z.
constexpr int kCombineChunk = 1024;
template <int D>
__global__ void __launch_bounds__(kThreads) combine_kernel(const float* __restrict__ pS, const float* __restrict__ pz,
                                                           const float* __restrict__ pstab, int splits, int m,
                                                           float* __restrict__ S, float* __restrict__ z) {
    __shared__ float wts[64 * 8];             // splits * slices weights (<= 64 splits, <= 8 slices)
    const int64_t bh = blockIdx.x;
    const int e0 = blockIdx.y * kCombineChunk;
    const int e1 = min(m * D, e0 + kCombineChunk);
    const int slices = m / kSlice;
    const float* st = pstab + bh * splits * slices;
    float M = -INFINITY;
    for (int i = 0; i < splits * slices; ++i) M = fmaxf(M, st[i]);
    for (int i = threadIdx.x; i < splits * slices; i += kThreads)
        wts[i] = st[i] == -INFINITY ? 0.f : exp_shift(st[i], M);
    __syncthreads();
    for (int e = e0 + threadIdx.x; e < e1; e += kThreads) {
        int r = e / D;
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) acc = fmaf(wts[s * slices + r / kSlice], pS[((bh * splits + s) * m) * D + e], acc);
        S[bh * m * D + e] = acc;
    }
    if (blockIdx.y != 0) return;
    for (int r = threadIdx.x; r < m; r += kThreads) {
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) acc = fmaf(wts[s * slices + r / kSlice], pz[(bh * splits + s) * m + r], acc);
        z[bh * m + r] = acc;
    }
}

// Y tile = phi(Q) S / phi(Q) z with per-row query stabilisers.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) readout_kernel(const T* __restrict__ Q, const T* __restrict__ Om,
                                                           const float* __restrict__ S, const float* __restrict__ z,
                                                           T* __restrict__ Y, int64_t n, int m, int kind,
                                                           float relu_eps, float scale) {
    extern __shared__ float smem[];
    float* qs = smem;                          // kTok * D
    float* oms = qs + kTok * D;                // kOmChunk * (D + 1)
    float* ps = oms + kOmChunk * (D + 1);      // kTok * m
    float* hs = ps + kTok * m;                 // kTok
    float* den = hs + kTok;                    // kTok
    const int64_t bh = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    Q += bh * n * D;
    Y += bh * n * D;
    S += bh * m * D;
    z += bh * m;

    load_tile<T, D>(Q, n, t0, qs);
    __syncthreads();
    half_norms<D>(qs, scale, hs);
    project_rows<T, D>(Om, 0, m, qs, scale, oms, ps, m);
    const float inv_sqrt_m = rsqrtf((float)m);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int t = warp; t < kTok; t += kThreads / 32) {
        float* pr = ps + t * m;
        float dsum = 0.f;
        if (kind != kKindExp) {
            for (int r = lane; r < m; r += 32) {
                pr[r] = phi_plain(pr[r], kind, inv_sqrt_m, relu_eps);
                dsum = fmaf(pr[r], z[r], dsum);
            }
        } else {
            float rmax = -INFINITY;
            for (int r = lane; r < m; r += 32) {
                pr[r] -= hs[t];
                rmax = fmaxf(rmax, pr[r]);
            }
            rmax = warp_max(rmax);
            for (int r = lane; r < m; r += 32) {
                pr[r] = exp_shift(pr[r], rmax) * inv_sqrt_m;
                dsum = fmaf(pr[r], z[r], dsum);
            }
        }
        dsum = warp_sum(dsum);
        if (lane == 0) den[t] = dsum;
    }
    __syncthreads();
    const int c = threadIdx.x % D;
    for (int t = threadIdx.x / D; t < kTok; t += kThreads / D) {
        int64_t row = t0 + t;
        // four independent partial sums keep several loads of S in flight (m is a multiple of 64)
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        const float* pr = ps + t * m;
#pragma unroll 4
        for (int r = 0; r < m; r += 4) {
            a0 = fmaf(pr[r], S[(int64_t)r * D + c], a0);
            a1 = fmaf(pr[r + 1], S[(int64_t)(r + 1) * D + c], a1);
            a2 = fmaf(pr[r + 2], S[(int64_t)(r + 2) * D + c], a2);
            a3 = fmaf(pr[r + 3], S[(int64_t)(r + 3) * D + c], a3);
        }
        const float acc = (a0 + a1) + (a2 + a3);
        if (row < n) store_elem(Y + row * D + c, acc / den[t]);
    }
}

// ------------------------------------------------------------------------------------------------
// Causal scan: one CTA per head; per 16-token sub-chunk
//   Y = (phi(Q) S_prev + tril(phi(Q) phi(K)^T) V) / (phi(Q) z_prev + tril(...) 1),
//   then S += phi(K)^T V, z += phi(K)^T 1.  S, z live in the workspace [BH][m][D], [BH][m].
// ------------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) causal_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                          const T* __restrict__ V, const T* __restrict__ Om,
                                                          T* __restrict__ Y, int64_t n, int m, int kind,
                                                          float relu_eps, float scale, float* __restrict__ Sg,
                                                          float* __restrict__ zg) {
    extern __shared__ float smem[];
    float* qs = smem;                          // kTok * D
    float* ks = qs + kTok * D;                 // kTok * D
    float* vs = ks + kTok * D;                 // kTok * D
    float* pq = vs + kTok * D;                 // kTok * m
    float* pk = pq + kTok * m;                 // kTok * m
    float* P = pk + kTok * m;                  // kTok * kTok
    float* hq = P + kTok * kTok;               // kTok
    float* hk = hq + kTok;                     // kTok
    float* oms = hk + kTok;                    // kOmChunk * (D + 1)
    float* red = oms + kOmChunk * (D + 1);     // 8
    const int64_t bh = blockIdx.x;
    Q += bh * n * D;
    K += bh * n * D;
    V += bh * n * D;
    Y += bh * n * D;
    float* S = Sg + bh * m * D;
    float* z = zg + bh * m;
    const float inv_sqrt_m = rsqrtf((float)m);
    for (int e = threadIdx.x; e < m * D; e += kThreads) S[e] = 0.f;
    for (int e = threadIdx.x; e < m; e += kThreads) z[e] = 0.f;
    float stab = -INFINITY;

    for (int64_t t0 = 0; t0 < n; t0 += kTok) {
        __syncthreads();
        load_tile<T, D>(Q, n, t0, qs);
        load_tile<T, D>(K, n, t0, ks);
        load_tile<T, D>(V, n, t0, vs);
        __syncthreads();
        half_norms<D>(qs, scale, hq);
        half_norms<D>(ks, scale, hk);
        project_rows<T, D>(Om, 0, m, qs, scale, oms, pq, m);
        project_rows<T, D>(Om, 0, m, ks, scale, oms, pk, m);
        const int nvalid = (int)(n - t0 < kTok ? n - t0 : kTok);
        if (kind == kKindExp) {
            float cmax = -INFINITY;
            for (int e = threadIdx.x; e < kTok * m; e += kThreads) {
                int t = e / m;
                float u = pk[e] - hk[t];
                pk[e] = u;
                if (t < nvalid) cmax = fmaxf(cmax, u);
            }
            cmax = block_max(cmax, red);
            if (cmax > stab) {
                float f = stab == -INFINITY ? 0.f : exp_shift(stab, cmax);
                for (int e = threadIdx.x; e < m * D; e += kThreads) S[e] *= f;
                for (int e = threadIdx.x; e < m; e += kThreads) z[e] *= f;
                stab = cmax;
            }
            for (int e = threadIdx.x; e < kTok * m; e += kThreads) {
                int t = e / m;
                pk[e] = t < nvalid ? exp_shift(pk[e], stab) * inv_sqrt_m : 0.f;
            }
            const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
            for (int t = warp; t < kTok; t += kThreads / 32) {
                float* pr = pq + t * m;
                float rmax = -INFINITY;
                for (int r = lane; r < m; r += 32) {
                    pr[r] -= hq[t];
                    rmax = fmaxf(rmax, pr[r]);
                }
                rmax = warp_max(rmax);
                for (int r = lane; r < m; r += 32) pr[r] = exp_shift(pr[r], rmax) * inv_sqrt_m;
            }
        } else {
            for (int e = threadIdx.x; e < kTok * m; e += kThreads) {
                int t = e / m;
                pk[e] = t < nvalid ? phi_plain(pk[e], kind, inv_sqrt_m, relu_eps) : 0.f;
                pq[e] = phi_plain(pq[e], kind, inv_sqrt_m, relu_eps);
            }
        }
        __syncthreads();
        {   // intra-chunk block, lower triangular (j <= i)
            int i = threadIdx.x / kTok, j = threadIdx.x % kTok;
            float acc = 0.f;
            if (j <= i)
                for (int r = 0; r < m; ++r) acc = fmaf(pq[i * m + r], pk[j * m + r], acc);
            P[i * kTok + j] = acc;
        }
        __syncthreads();
        const int c = threadIdx.x % D;
        for (int i = threadIdx.x / D; i < kTok; i += kThreads / D) {
            float num = 0.f, dn = 0.f;
            const float* pr = pq + i * m;
            for (int r = 0; r < m; ++r) {
                num = fmaf(pr[r], S[(int64_t)r * D + c], num);
                dn = fmaf(pr[r], z[r], dn);
            }
            for (int j = 0; j <= i; ++j) {
                num = fmaf(P[i * kTok + j], vs[j * D + c], num);
                dn += P[i * kTok + j];
            }
            if (t0 + i < n) store_elem(Y + (t0 + i) * D + c, num / dn);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < m * D; e += kThreads) {
            int r = e / D, cc = e % D;
            float acc = S[e];
            for (int j = 0; j < kTok; ++j) acc = fmaf(pk[j * m + r], vs[j * D + cc], acc);
            S[e] = acc;
        }
        for (int r = threadIdx.x; r < m; r += kThreads) {
            float acc = z[r];
            for (int j = 0; j < kTok; ++j) acc += pk[j * m + r];
            z[r] = acc;
        }
    }
}

}  // namespace simt
}  // namespace favor
