// Tensor-core (tcgen05 + TMA + TMEM) kernels of the non-causal FAVOR+ path, bf16 in / fp32 accumulate.
//
//   nc_state_tc   key side. One CTA per (head, token split, feature slice). For every 128-token
//                 tile it projects the keys onto up to four 128-feature groups of Omega with the
//                 features on the TMEM lanes (U^T = Omega_g K_tile^T), turns U^T into
//                 phi(K)^T in place (bf16, packed two per TMEM column) and accumulates
//                 S_g += phi(K)^T V_tile with phi(K)^T read straight from TMEM. z = Phi(K)^T 1 is a
//                 per-lane running sum in the epilogue. phi(K) never leaves the SM.
//   nc_combine    sums the partial (S, z) of all splits in a fixed order after rescaling each to
//                 the head's largest key stabiliser, and writes S as the bf16 operand image the
//                 readout copies into shared memory unchanged.
//   nc_readout_tc query side. Per 128-token tile: U = Q_tile Omega^T (tokens on the lanes),
//                 phi(Q) in place with an exact per-row stabiliser, den = phi(Q) z on the CUDA
//                 cores, num = phi(Q) S on the tensor cores, Y = num / den stored by TMA.
//
// Stabilisers. A query row may use any constant of its own and a head's keys any one constant:
// both cancel between numerator and denominator. Queries use their exact row maximum. Keys use
// the bound  u_r(k) <= W |k^| - |k^|^2 / 2  (Cauchy-Schwarz, W = largest row norm of Omega), held
// per CTA as a running value that only moves (with a rescale of the accumulated S and z) when a
// tile's bound exceeds it by more than kStabSlackHi; the common factor 1/sqrt(m) is dropped on both
// sides for the same reason.
#pragma once

#include "tc.cuh"

namespace favor {
namespace tcnc {

using namespace favor::tc;

constexpr int kTile = 128;            // tokens per tile (the MMA M or N extent)
constexpr int kThreads = 192;         // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue
constexpr int kEpiThreads = 128;
constexpr float kStabSlackLo = 12.f;  // after a (re)set, the key stabiliser sits this far below the bound
constexpr float kStabSlackHi = 24.f;  // ... and is raised once a tile's bound exceeds it by this much

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Squared norm of row `row` of a [128 x D] bf16 tile stored as D/64 swizzled regions of 16 KB.
template <int D>
__device__ __forceinline__ float tile_row_sqnorm(const uint8_t* tile, int row) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int a = 0; a < D / 64; ++a) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 v = *reinterpret_cast<const uint4*>(tile + a * 16384 + sw128_offset(row, c));
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
                s0 = fmaf(lo, lo, s0);
                s1 = fmaf(hi, hi, s1);
            }
        }
    }
    return s0 + s1;
}

// =============================================================================================
// Key-side state kernel
// =============================================================================================
struct StateParams {
    int n;              // tokens per head
    int m_pad;          // features, padded to a multiple of 128
    int groups;         // 128-feature groups handled by this CTA (1..4, D=128: 1..2)
    int tokens_per_split;
    int kind;           // kKindExp / kKindRelu
    float relu_eps_s;   // relu_eps * sqrt(m)
    float scale;        // d^(-1/4)
    float* pS;          // [BH][splits][m_pad][D] fp32
    float* pz;          // [BH][splits][m_pad]
    float* pstab;       // [BH][splits][fslices]
};

template <int D>
struct StateSmem {
    static constexpr int kStages = (D == 64) ? 4 : 2;
    static constexpr int kTileBytes = kTile * D * 2;  // one [128 x D] bf16 tile
    // Omega region: D/64 swizzled regions of (groups * 128) rows, each row 128 B.
    __host__ __device__ static size_t omega_bytes(int groups) { return (size_t)groups * 128 * D * 2; }
    static size_t bytes(int groups) { return 1024 + omega_bytes(groups) + (size_t)kStages * 2 * kTileBytes + 1024; }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    nc_state_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                const __grid_constant__ CUtensorMap mOm, StateParams p) {
    using SM = StateSmem<D>;
    constexpr int NS = SM::kStages;
    constexpr int kAtoms = D / 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int G = p.groups;
    uint8_t* sOm = smem;                                   // kAtoms regions of G*128 rows
    uint8_t* sStage = sOm + SM::omega_bytes(G);            // NS x {K tile, V tile}
    float* sC = reinterpret_cast<float*>(sStage + (size_t)NS * 2 * SM::kTileBytes);  // [128] per-token constants
    __shared__ uint64_t bar_full[NS], bar_empty[NS], bar_om, bar_ufull[2], bar_ufree[2], bar_phi[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float red[4];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int split = blockIdx.x, splits = gridDim.x;
    const int bh = blockIdx.y;
    const int fslice = blockIdx.z, fslices = gridDim.z;
    const int f0 = fslice * G * 128;  // first feature of this CTA
    const int j0 = split * p.tokens_per_split;
    const int j1 = min(p.n, j0 + p.tokens_per_split);
    const int T = (j1 - j0 + kTile - 1) / kTile;
    const int U = T * G;  // units = (tile, group) pairs

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1 + 4);  // MMA commit + one arrive per epilogue warp
        }
        mbar_init(&bar_om, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_ufull[i], 1);
            mbar_init(&bar_ufree[i], 1);
            mbar_init(&bar_phi[i], 4);
        }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    // TMEM: S_g at columns [g*D, (g+1)*D); U slots at 256 and 384.
    auto u_col = [](int s) { return 256u + 128u * (uint32_t)s; };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mV);
            tma_prefetch_desc(&mOm);
            mbar_arrive_expect_tx(&bar_om, (uint32_t)SM::omega_bytes(G));
            for (int g = 0; g < G; ++g)
                for (int a = 0; a < kAtoms; ++a)
                    tma_load_2d(sOm + (size_t)a * G * 16384 + g * 16384, &mOm, &bar_om, a * 64, f0 + g * 128);
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int st = t % NS;
                if (!mbar_wait(&bar_empty[st], ((t / NS) & 1) ^ 1, &abort_flag)) break;
                uint8_t* kt = sStage + (size_t)st * 2 * SM::kTileBytes;
                uint8_t* vt = kt + SM::kTileBytes;
                mbar_arrive_expect_tx(&bar_full[st], 2 * SM::kTileBytes);
                for (int a = 0; a < kAtoms; ++a) {
                    tma_load_3d(kt + a * 16384, &mK, &bar_full[st], a * 64, j0 + t * kTile, bh);
                    tma_load_3d(vt + a * 16384, &mV, &bar_full[st], a * 64, j0 + t * kTile, bh);
                }
                issued = t + 1;
            }
            // Drain: every issued load must land before the CTA may exit.
            for (int t = max(0, issued - NS); t < issued; ++t) {
                volatile int never = 0;
                mbar_wait(&bar_full[t % NS], (t / NS) & 1, &never);
            }
            volatile int never = 0;
            mbar_wait(&bar_om, 0, &never);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_p = idesc_bf16(128, 128, false, false);  // U^T = Om_g K^T
            constexpr uint32_t idesc_s = idesc_bf16(128, D, false, true);     // S_g += phi^T V
            bool ok = mbar_wait(&bar_om, 0, &abort_flag);
            tc_fence_after();
            // Unit u = (tile u / G, group u % G) uses U slot u % 2.
            auto issue_proj = [&](int u) -> bool {
                const int t = u / G, g = u % G, s = u & 1, st = t % NS;
                if (g == 0 && !mbar_wait(&bar_full[st], (t / NS) & 1, &abort_flag)) return false;
                if (!mbar_wait(&bar_ufree[s], ((u >> 1) & 1) ^ 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* kt = sStage + (size_t)st * 2 * SM::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int a = ks / 4, w = ks % 4;
                    uint64_t ad = sdesc_sw128(smem_u32(sOm + (size_t)a * G * 16384 + g * 16384 + w * 32), 16, 1024);
                    uint64_t bd = sdesc_sw128(smem_u32(kt + a * 16384 + w * 32), 16, 1024);
                    mma_ss(tbase + u_col(s), ad, bd, idesc_p, ks > 0);
                }
                mma_commit(&bar_ufull[s]);
                return true;
            };
            auto issue_state = [&](int u) -> bool {
                const int t = u / G, g = u % G, s = u & 1, st = t % NS;
                if (!mbar_wait(&bar_phi[s], (u >> 1) & 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* vt = sStage + (size_t)st * 2 * SM::kTileBytes + SM::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks) {
                    uint64_t bd = sdesc_sw128(smem_u32(vt + ks * 2048), 16384, 1024);
                    mma_ts(tbase + (uint32_t)(g * D), tbase + u_col(s) + ks * 8, bd, idesc_s, (t > 0 || ks > 0));
                }
                mma_commit(&bar_ufree[s]);
                if (g == G - 1) mma_commit(&bar_empty[st]);
                return true;
            };
            if (ok) {
                for (int u = 0; u < U; ++u) {
                    if (!issue_proj(u)) break;
                    if (u >= 1 && !issue_state(u - 1)) break;
                }
                if (!abort_flag && U > 0) issue_state(U - 1);
            }
        }
    } else {
        // ---------------- epilogue (warps 2-5) ----------------
        const int q = warp & 3;
        const int r = q * 32 + lane;  // TMEM lane = feature row within a group; also the token row for norms
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const float A2 = p.scale * kLog2e;
        float zacc[4] = {0.f, 0.f, 0.f, 0.f};
        float stab = 0.f;
        bool failed = !mbar_wait(&bar_om, 0, &abort_flag);
        __syncwarp();
        // W = largest row norm of this CTA's Omega rows (zero rows past m do not matter).
        float W = 0.f;
        if (p.kind == kKindExp) {
            float w2 = 0.f;
            for (int g = 0; g < G; ++g) {
                float s = 0.f;
                for (int a = 0; a < kAtoms; ++a) s += tile_row_sqnorm<64>(sOm + (size_t)a * G * 16384 + g * 16384, r);
                w2 = fmaxf(w2, s);
            }
            w2 = warp_max(w2);
            if (lane == 0) red[q] = w2;
            named_bar(1, kEpiThreads);
            W = sqrtf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])));
            named_bar(1, kEpiThreads);
        }
        // On a failed wait the loop keeps running (the waits then return at once) so that every
        // epilogue thread passes the same named barriers; only the results are garbage.
        for (int t = 0; t < T; ++t) {
            const int st = t % NS;
            failed |= !mbar_wait(&bar_full[st], (t / NS) & 1, &abort_flag);
            __syncwarp();
            const uint8_t* kt = sStage + (size_t)st * 2 * SM::kTileBytes;
            const int j = j0 + t * kTile + r;
            const bool valid = j < j1;
            float cj = INFINITY;
            if (p.kind == kKindExp) {
                const float xn2 = p.scale * p.scale * tile_row_sqnorm<D>(kt, r);  // |k^|^2
                const float h = 0.5f * xn2;
                const float b = valid ? W * sqrtf(xn2) - h : -INFINITY;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_empty[st]);
                const float bm = warp_max(b);
                if (lane == 0) red[q] = bm;
                named_bar(1, kEpiThreads);
                const float Bt = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
                named_bar(1, kEpiThreads);
                if (t == 0) {
                    stab = Bt - kStabSlackLo;
                } else if (Bt > stab + kStabSlackHi) {
                    // Raise the stabiliser: wait for every state MMA issued so far, rescale S and z.
                    const float nst = Bt - kStabSlackLo;
                    const float f = ex2((stab - nst) * kLog2e);
                    const int ul = t * G - 1;  // last unit of the previous tile
                    failed |= !mbar_wait(&bar_ufree[ul & 1], (ul >> 1) & 1, &abort_flag);
                    __syncwarp();
                    tc_fence_after();
                    for (int g = 0; g < G; ++g) {
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t v[32];
                            tmem_ld32(tbase + lane_off + g * D + c0, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                            tmem_st32(tbase + lane_off + g * D + c0, v);
                        }
                        zacc[g] *= f;
                    }
                    tmem_st_wait();
                    stab = nst;
                }
                cj = valid ? (h + stab) * kLog2e : INFINITY;
            } else {
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_empty[st]);
                cj = valid ? 0.f : INFINITY;
                named_bar(1, kEpiThreads);  // previous tile's readers of sC are done
            }
            sC[r] = cj;
            named_bar(1, kEpiThreads);
            for (int g = 0; g < G; ++g) {
                const int u = t * G + g, s = u & 1;
                failed |= !mbar_wait(&bar_ufull[s], (u >> 1) & 1, &abort_flag);
                __syncwarp();
                tc_fence_after();
                const uint32_t ua = tbase + lane_off + u_col(s);
                float z = zacc[g];
#pragma unroll
                for (int c = 0; c < kTile / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(ua + 32 * c, v);
                    tmem_ld_wait();
                    float ph[32];
                    if (p.kind == kKindExp) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 c4 = *reinterpret_cast<const float4*>(sC + 32 * c + i);
                            ph[i + 0] = ex2(fmaf(__uint_as_float(v[i + 0]), A2, -c4.x));
                            ph[i + 1] = ex2(fmaf(__uint_as_float(v[i + 1]), A2, -c4.y));
                            ph[i + 2] = ex2(fmaf(__uint_as_float(v[i + 2]), A2, -c4.z));
                            ph[i + 3] = ex2(fmaf(__uint_as_float(v[i + 3]), A2, -c4.w));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 c4 = *reinterpret_cast<const float4*>(sC + 32 * c + i);
                            ph[i + 0] = c4.x == 0.f ? fmaxf(__uint_as_float(v[i + 0]) * p.scale, 0.f) + p.relu_eps_s : 0.f;
                            ph[i + 1] = c4.y == 0.f ? fmaxf(__uint_as_float(v[i + 1]) * p.scale, 0.f) + p.relu_eps_s : 0.f;
                            ph[i + 2] = c4.z == 0.f ? fmaxf(__uint_as_float(v[i + 2]) * p.scale, 0.f) + p.relu_eps_s : 0.f;
                            ph[i + 3] = c4.w == 0.f ? fmaxf(__uint_as_float(v[i + 3]) * p.scale, 0.f) + p.relu_eps_s : 0.f;
                        }
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t w = pack_bf16(ph[2 * i], ph[2 * i + 1]);
                        pk[i] = w;
                        // z sums the bf16-rounded features the MMA sees.
                        z += __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
                    }
                    tmem_st16(ua + 16 * c, pk);
                }
                zacc[g] = z;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_phi[s]);
            }
        }
        // Final state: wait for the last state MMA, then write this CTA's partial S, z and stabiliser.
        if (__all_sync(0xffffffffu, !failed) && U > 0) {
            const int ul = U - 1;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_ufree[ul & 1], (ul >> 1) & 1, &abort_flag));
            if (ok) {
                tc_fence_after();
                const size_t part = (size_t)bh * splits + split;
                for (int g = 0; g < G; ++g) {
                    const int feat = f0 + g * 128 + r;
                    float* out = p.pS + (part * p.m_pad + feat) * D;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tbase + lane_off + g * D + c0, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(out + c0 + i) =
                                make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                                            __uint_as_float(v[i + 3]));
                    }
                    p.pz[part * p.m_pad + feat] = zacc[g];
                }
                if (threadIdx.x == 64) p.pstab[part * fslices + fslice] = p.kind == kKindExp ? stab : 0.f;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// =============================================================================================
// Combine: S = sum_s w_s S_s, z = sum_s w_s z_s with w_s = exp(stab_s - max stab); S written as the
// readout's B operand image: D/64 regions of [m_pad rows x 128 B], 128-byte swizzled, bf16.
// Grid (m_pad / 16, BH), 128 threads: thread = (row in the block of 16, 16-byte chunk).
// =============================================================================================
template <int D>
__global__ void __launch_bounds__(128) nc_combine(const float* __restrict__ pS, const float* __restrict__ pz,
                                                  const float* __restrict__ pstab, int splits, int fslices,
                                                  int m, int m_pad, int feats_per_slice, uint8_t* __restrict__ Simg,
                                                  float* __restrict__ zout) {
    constexpr int kChunks = D / 8;  // 16-byte bf16 chunks per row
    __shared__ float wts[1024];
    const int bh = blockIdx.y;
    const int nst = splits * fslices;
    const float* st = pstab + (size_t)bh * nst;
    float M = -INFINITY;
    for (int i = 0; i < nst; ++i) M = fmaxf(M, st[i]);
    for (int i = threadIdx.x; i < nst; i += blockDim.x) wts[i] = ex2((st[i] - M) * kLog2e);
    __syncthreads();
    const int rows_per_block = 128 / kChunks;  // D=64: 16 rows, D=128: 8 rows
    const int row = blockIdx.x * rows_per_block + threadIdx.x / kChunks;
    const int ch = threadIdx.x % kChunks;
    if (row >= m_pad) return;
    const int fs = row / feats_per_slice;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float zs = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float w = wts[s * fslices + fs];
        const float* src = pS + (((size_t)bh * splits + s) * m_pad + row) * D + ch * 8;
        const float4 a = *reinterpret_cast<const float4*>(src);
        const float4 b = *reinterpret_cast<const float4*>(src + 4);
        acc[0] = fmaf(w, a.x, acc[0]); acc[1] = fmaf(w, a.y, acc[1]);
        acc[2] = fmaf(w, a.z, acc[2]); acc[3] = fmaf(w, a.w, acc[3]);
        acc[4] = fmaf(w, b.x, acc[4]); acc[5] = fmaf(w, b.y, acc[5]);
        acc[6] = fmaf(w, b.z, acc[6]); acc[7] = fmaf(w, b.w, acc[7]);
        if (ch == 0) zs = fmaf(w, pz[((size_t)bh * splits + s) * m_pad + row], zs);
    }
    if (row >= m) {  // padding features: no contribution to the readout
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        zs = 0.f;
    }
    uint4 o = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                         pack_bf16(acc[6], acc[7]));
    const int a = ch / 8, c = ch % 8;
    uint8_t* img = Simg + (size_t)bh * m_pad * D * 2 + (size_t)a * m_pad * 128;
    *reinterpret_cast<uint4*>(img + row * 128 + ((c ^ (row & 7)) << 4)) = o;
    if (ch == 0) zout[(size_t)bh * m_pad + row] = zs;
}

// =============================================================================================
// Query-side readout kernel
// =============================================================================================
struct ReadoutParams {
    int n;
    int m_pad;
    int m;
    int tiles_per_cta;
    int kind;
    float relu_eps_s;
    float scale;
    const uint8_t* Simg;  // [BH][m_pad * D * 2] from nc_combine
    const float* z;       // [BH][m_pad]
};

template <int D>
struct ReadoutSmem {
    static constexpr int kStages = (D == 64) ? 4 : 2;
    static constexpr int kTileBytes = kTile * D * 2;
    static size_t bytes(int m_pad) {
        return 1024 + (size_t)m_pad * D * 2 /*Omega*/ + (size_t)m_pad * D * 2 /*S image*/ + (size_t)m_pad * 4 /*z*/ +
               (size_t)kStages * kTileBytes + kTileBytes /*Y staging*/;
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    nc_readout_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mOm,
                  const __grid_constant__ CUtensorMap mY, ReadoutParams p) {
    using SM = ReadoutSmem<D>;
    constexpr int NS = SM::kStages;
    constexpr int kAtoms = D / 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int MP = p.m_pad;
    uint8_t* sOm = smem;                                   // kAtoms regions of MP rows x 128 B
    uint8_t* sS = sOm + (size_t)MP * D * 2;                // S image: kAtoms regions of MP rows x 128 B
    uint8_t* sQ = sS + (size_t)MP * D * 2;                 // NS stages
    uint8_t* sY = sQ + (size_t)NS * SM::kTileBytes;        // Y staging tile
    float* sz = reinterpret_cast<float*>(sY + SM::kTileBytes);  // [MP]
    __shared__ uint64_t bar_full[NS], bar_empty[NS], bar_const, bar_ufull[2], bar_ufree[2], bar_phi[2], bar_num[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y;
    const int tiles_head = (p.n + kTile - 1) / kTile;
    const int t0 = blockIdx.x * p.tiles_per_cta;
    const int T = max(0, min(tiles_head, t0 + p.tiles_per_cta) - t0);
    const int nslot = MP <= 256 ? 2 : 1;
    const uint32_t slot_cols = MP <= 256 ? 256u : 512u;
    const uint32_t num_off = MP <= 256 ? 128u : 256u;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_const, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_ufull[i], 1);
            mbar_init(&bar_ufree[i], 4);
            mbar_init(&bar_phi[i], 4);
            mbar_init(&bar_num[i], 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&mQ);
            tma_prefetch_desc(&mOm);
            tma_prefetch_desc(&mY);
            const uint32_t sbytes = (uint32_t)MP * D * 2;
            mbar_arrive_expect_tx(&bar_const, sbytes * 2 + (uint32_t)MP * 4);
            for (int a = 0; a < kAtoms; ++a)
                for (int r0 = 0; r0 < MP; r0 += 128)
                    tma_load_2d(sOm + (size_t)a * MP * 128 + r0 * 128, &mOm, &bar_const, a * 64, r0);
            bulk_load(sS, p.Simg + (size_t)bh * sbytes, sbytes, &bar_const);
            bulk_load(sz, p.z + (size_t)bh * MP, (uint32_t)MP * 4, &bar_const);
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int st = t % NS;
                if (!mbar_wait(&bar_empty[st], ((t / NS) & 1) ^ 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&bar_full[st], SM::kTileBytes);
                for (int a = 0; a < kAtoms; ++a)
                    tma_load_3d(sQ + (size_t)st * SM::kTileBytes + a * 16384, &mQ, &bar_full[st], a * 64,
                                (t0 + t) * kTile, bh);
                issued = t + 1;
            }
            for (int t = max(0, issued - NS); t < issued; ++t) {
                volatile int never = 0;
                mbar_wait(&bar_full[t % NS], (t / NS) & 1, &never);
            }
            volatile int never = 0;
            mbar_wait(&bar_const, 0, &never);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const int nN = MP <= 256 ? 1 : 2;    // N blocks of the projection
            const int Nb = MP <= 256 ? MP : MP / 2;
            const uint32_t idesc_p = idesc_bf16(128, Nb, false, false);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
            bool ok = mbar_wait(&bar_const, 0, &abort_flag);
            tc_fence_after();
            auto issue_proj = [&](int t) -> bool {
                const int s = t % nslot, st = t % NS;
                const int k = t / nslot;  // use count of slot s
                if (!mbar_wait(&bar_full[st], (t / NS) & 1, &abort_flag)) return false;
                if (!mbar_wait(&bar_ufree[s], (k & 1) ^ 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* qt = sQ + (size_t)st * SM::kTileBytes;
                for (int nb = 0; nb < nN; ++nb) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const int a = ks / 4, w = ks % 4;
                        uint64_t ad = sdesc_sw128(smem_u32(qt + a * 16384 + w * 32), 16, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(sOm + (size_t)a * MP * 128 + (size_t)nb * Nb * 128 + w * 32),
                                                  16, 1024);
                        mma_ss(tbase + s * slot_cols + nb * Nb, ad, bd, idesc_p, ks > 0);
                    }
                }
                mma_commit(&bar_ufull[s]);
                mma_commit(&bar_empty[st]);
                return true;
            };
            auto issue_out = [&](int t) -> bool {
                const int s = t % nslot, k = t / nslot;
                if (!mbar_wait(&bar_phi[s], k & 1, &abort_flag)) return false;
                tc_fence_after();
                for (int ks = 0; ks < MP / 16; ++ks) {
                    uint64_t bd = sdesc_sw128(smem_u32(sS + ks * 2048), (uint32_t)MP * 128, 1024);
                    mma_ts(tbase + s * slot_cols + num_off, tbase + s * slot_cols + ks * 8, bd, idesc_o, ks > 0);
                }
                mma_commit(&bar_num[s]);
                return true;
            };
            if (ok) {
                if (nslot == 2) {
                    for (int t = 0; t < T; ++t) {
                        if (!issue_proj(t)) break;
                        if (t >= 1 && !issue_out(t - 1)) break;
                    }
                    if (!abort_flag && T > 0) issue_out(T - 1);
                } else {
                    for (int t = 0; t < T; ++t)
                        if (!issue_proj(t) || !issue_out(t)) break;
                }
            }
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;
        const int r = q * 32 + lane;  // token row of the tile
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const float A2 = p.scale * kLog2e;
        const bool is_issuer = (warp == 2 && lane == 0);
        float den[2] = {0.f, 0.f};
        bool failed = !mbar_wait(&bar_const, 0, &abort_flag);
        __syncwarp();

        auto epi1 = [&](int t) -> bool {
            const int s = t % nslot, k = t / nslot;
            const bool ok = mbar_wait(&bar_ufull[s], k & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            const uint32_t ua = tbase + lane_off + s * slot_cols;
            float rmax = 0.f;
            if (p.kind == kKindExp) {
                rmax = -INFINITY;
                for (int c0 = 0; c0 < MP; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(ua + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        rmax = fmaxf(rmax, fmaxf(__uint_as_float(v[i]), __uint_as_float(v[i + 1])));
                }
            }
            const float cst = A2 * rmax;
            float dsum = 0.f;
            for (int c0 = 0; c0 < MP; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(ua + c0, v);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 z4 = *reinterpret_cast<const float4*>(sz + c0 + i);
                    float f0, f1, f2, f3;
                    if (p.kind == kKindExp) {
                        f0 = ex2(fmaf(__uint_as_float(v[i + 0]), A2, -cst));
                        f1 = ex2(fmaf(__uint_as_float(v[i + 1]), A2, -cst));
                        f2 = ex2(fmaf(__uint_as_float(v[i + 2]), A2, -cst));
                        f3 = ex2(fmaf(__uint_as_float(v[i + 3]), A2, -cst));
                    } else {
                        f0 = fmaxf(__uint_as_float(v[i + 0]) * p.scale, 0.f) + p.relu_eps_s;
                        f1 = fmaxf(__uint_as_float(v[i + 1]) * p.scale, 0.f) + p.relu_eps_s;
                        f2 = fmaxf(__uint_as_float(v[i + 2]) * p.scale, 0.f) + p.relu_eps_s;
                        f3 = fmaxf(__uint_as_float(v[i + 3]) * p.scale, 0.f) + p.relu_eps_s;
                    }
                    const uint32_t w0 = pack_bf16(f0, f1), w1 = pack_bf16(f2, f3);
                    pk[i / 2] = w0;
                    pk[i / 2 + 1] = w1;
                    // den uses the same bf16-rounded features as the numerator MMA.
                    dsum = fmaf(__uint_as_float(w0 << 16), z4.x, dsum);
                    dsum = fmaf(__uint_as_float(w0 & 0xFFFF0000u), z4.y, dsum);
                    dsum = fmaf(__uint_as_float(w1 << 16), z4.z, dsum);
                    dsum = fmaf(__uint_as_float(w1 & 0xFFFF0000u), z4.w, dsum);
                }
                tmem_st16(ua + c0 / 2, pk);
            }
            den[t & 1] = dsum;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_phi[s]);
            return ok;
        };
        auto epi2 = [&](int t) -> bool {
            const int s = t % nslot, k = t / nslot;
            const bool ok = mbar_wait(&bar_num[s], k & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            const uint32_t na = tbase + lane_off + s * slot_cols + num_off;
            const float inv = 1.f / den[t & 1];
            // The staging tile is free once the previous TMA store has read it.
            if (is_issuer) bulk_wait_read0();
            named_bar(2, kEpiThreads);
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(na + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint4 o;
                    o.x = pack_bf16(__uint_as_float(v[8 * cc + 0]) * inv, __uint_as_float(v[8 * cc + 1]) * inv);
                    o.y = pack_bf16(__uint_as_float(v[8 * cc + 2]) * inv, __uint_as_float(v[8 * cc + 3]) * inv);
                    o.z = pack_bf16(__uint_as_float(v[8 * cc + 4]) * inv, __uint_as_float(v[8 * cc + 5]) * inv);
                    o.w = pack_bf16(__uint_as_float(v[8 * cc + 6]) * inv, __uint_as_float(v[8 * cc + 7]) * inv);
                    const int chunk = (c0 / 8 + cc);  // 16-byte chunk index along the row (0..D/8)
                    *reinterpret_cast<uint4*>(sY + (chunk / 8) * 16384 + sw128_offset(r, chunk % 8)) = o;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_ufree[s]);
            fence_async_smem();
            named_bar(2, kEpiThreads);
            if (is_issuer) {
                for (int a = 0; a < kAtoms; ++a) tma_store_3d(&mY, sY + a * 16384, a * 64, (t0 + t) * kTile, bh);
                bulk_commit();
            }
            return ok;
        };
        // Every epilogue thread runs the whole schedule (failed waits return at once), so the named
        // barriers inside epi2 always see all 128 threads.
        if (T > 0) {
            if (nslot == 2) {
                failed |= !epi1(0);
                for (int t = 0; t < T; ++t) {
                    if (t + 1 < T) failed |= !epi1(t + 1);
                    failed |= !epi2(t);
                }
            } else {
                for (int t = 0; t < T; ++t) {
                    failed |= !epi1(t);
                    failed |= !epi2(t);
                }
            }
        }
        (void)failed;
        if (is_issuer) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace tcnc
}  // namespace favor
