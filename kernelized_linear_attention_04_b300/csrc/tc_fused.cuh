// Single-launch non-causal FAVOR+ for short sequences (bf16, d = 64, m <= 256, n <= 8 * 128).
//
// One thread-block cluster per head, one CTA per 128-token tile. Each CTA
//   1. projects its key tile with the features on the TMEM lanes, turns U^T into phi(K)^T in place
//      and accumulates its partial S = phi(K)^T V (tcgen05, A from TMEM) and z (per-lane sums), with
//      a key stabiliser of its own (12 nats below the tile's largest bound W |k^| - |k^|^2 / 2);
//   2. publishes the partial (fp32) in its shared memory; after a cluster barrier, CTA c sums the
//      feature rows [c R, (c + 1) R) over the cluster in rank order, each partial rescaled to the
//      cluster's largest stabiliser, and writes the bf16 rows of S (in the readout MMA's swizzled
//      operand layout) and z into every CTA of the cluster through distributed shared memory;
//   3. after a second cluster barrier, projects its query tile (tokens on the lanes), forms phi(Q)
//      in place with the exact row stabiliser, den = phi(Q) . z on the CUDA cores and
//      num = phi(Q) S on the tensor cores, and stores Y = num / den.
// S never goes through global memory and the whole call is one launch.
#pragma once

#include "tc.cuh"
#include "tc_noncausal.cuh"  // ex2, kStabSlackLo, tile_row_sqnorm, phi_col

namespace favor {
namespace tcfu {

using namespace favor::tc;
using tcnc::ex2;
using tcnc::kStabSlackLo;
using tcnc::tile_row_sqnorm;

constexpr int kTile = 128;
constexpr int kD = 64;
constexpr int kMaxCluster = 8;
constexpr int kEpiWarps = 16;
constexpr int kThreads = 32 * (1 + kEpiWarps);  // warp 0: TMA + MMA issue; warps 1..16: epilogue
constexpr int kTileBytes = kTile * kD * 2;

struct FusedParams {
    int n, m, m_pad;
    int kind;
    float relu_eps_s;  // relu_eps * sqrt(m)
    float scale;       // d^(-1/4)
    __nv_bfloat16* Y;
};

struct FusedSmem {
    // Omega (m_pad x 128 B), K, V, Q tiles, partial S (m_pad x 64 fp32), S image (m_pad x 128 B),
    // z (m_pad fp32), z partials (2 x m_pad fp32), per-token constants, row-max / den exchange.
    static size_t bytes(int m_pad) {
        return 1024 + (size_t)m_pad * 128 + 3 * kTileBytes + (size_t)m_pad * 256 + (size_t)m_pad * 128 +
               (size_t)m_pad * 4 + 2 * (size_t)m_pad * 4 + 128 * 4 + 2 * 4 * 128 * 4;
    }
};

__global__ void __launch_bounds__(kThreads, 1)
    nc_fused_small(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                   const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mOm, FusedParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 by hand below
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int MP = p.m_pad;
    const int G = MP / 128;
    uint8_t* sOm = smem;                                   // MP rows x 128 B (K-major, features = rows)
    uint8_t* sK = sOm + (size_t)MP * 128;
    uint8_t* sV = sK + kTileBytes;
    uint8_t* sQ = sV + kTileBytes;
    float* sP = reinterpret_cast<float*>(sQ + kTileBytes);  // [MP][64] partial S of this CTA
    uint8_t* sS = reinterpret_cast<uint8_t*>(sP + (size_t)MP * 64);  // bf16 S image, MP rows x 128 B
    float* sz = reinterpret_cast<float*>(sS + (size_t)MP * 128);     // [MP] z of the head
    float* sZp = sz + MP;                                  // [2][MP] z partials of the two token halves
    float* sC = sZp + 2 * MP;                              // [128] per-key constants
    float* sMax = sC + 128;                                // [4][128] row-max shares
    float* sDen = sMax + 4 * 128;                          // [4][128] denominator shares
    __shared__ uint64_t bar_load, bar_q, bar_u, bar_phi, bar_s, bar_pq, bar_phiq, bar_num;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float sStab;
    __shared__ float red[kEpiWarps];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int T = (int)cluster_size();   // tiles of the head = CTAs of the cluster
    const int rank = (int)cluster_rank();
    const int bh = blockIdx.x / T;
    const int j0 = rank * kTile;         // this CTA's tile
    const int nvalid = min(kTile, p.n - j0);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_load, 1);
        mbar_init(&bar_q, 1);
        mbar_init(&bar_u, 1);
        mbar_init(&bar_phi, kEpiWarps);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_pq, 1);
        mbar_init(&bar_phiq, kEpiWarps);
        mbar_init(&bar_num, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    // TMEM: S_g at [64 g, 64 g + 64); U^T of group g at 256 + 128 g; later U(Q) at [256, 256 + MP)
    // with phi(Q) packed in its first MP/2 columns, and num at [0, 64).

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&mQ);
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mV);
            tma_prefetch_desc(&mOm);
            mbar_arrive_expect_tx(&bar_load, (uint32_t)MP * 128 + 2 * kTileBytes);
            for (int r0 = 0; r0 < MP; r0 += 128) tma_load_2d(sOm + (size_t)r0 * 128, &mOm, &bar_load, 0, r0);
            tma_load_3d(sK, &mK, &bar_load, 0, j0, bh);
            tma_load_3d(sV, &mV, &bar_load, 0, j0, bh);
            mbar_arrive_expect_tx(&bar_q, kTileBytes);
            tma_load_3d(sQ, &mQ, &bar_q, 0, j0, bh);
            bool ok = mbar_wait(&bar_load, 0, &abort_flag);
            tc_fence_after();
            // key projections U^T_g = Omega_g K^T (M = 128 features, N = 128 tokens, K = 64)
            constexpr uint32_t id_p = idesc_bf16(128, 128, false, false);
            if (ok) {
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        uint64_t ad = sdesc_sw128(smem_u32(sOm + (size_t)g * 16384 + ks * 32), 16, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(sK + ks * 32), 16, 1024);
                        mma_ss(tbase + 256 + 128 * g, ad, bd, id_p, ks > 0);
                    }
                }
            }
            mma_commit(&bar_u);
            // state S_g = phi_g(K)^T V (A = phi^T packed in TMEM, B = V MN-major)
            ok = ok && mbar_wait(&bar_phi, 0, &abort_flag);
            tc_fence_after();
            constexpr uint32_t id_s = idesc_bf16(128, kD, false, true);
            if (ok) {
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks) {
                        uint64_t bd = sdesc_sw128(smem_u32(sV + ks * 2048), 16384, 1024);
                        mma_ts(tbase + 64 * g, tbase + 256 + 128 * g + tcnc::phi_col(ks), bd, id_s, ks > 0);
                    }
                }
            }
            mma_commit(&bar_s);
            // query projection U = Q Omega^T (M = 128 tokens, N = MP features) into the U^T columns
            ok = ok && mbar_wait(&bar_s, 0, &abort_flag) && mbar_wait(&bar_q, 0, &abort_flag);
            tc_fence_after();
            const uint32_t id_q = idesc_bf16(128, MP, false, false);
            if (ok) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint64_t ad = sdesc_sw128(smem_u32(sQ + ks * 32), 16, 1024);
                    uint64_t bd = sdesc_sw128(smem_u32(sOm + ks * 32), 16, 1024);
                    mma_ss(tbase + 256, ad, bd, id_q, ks > 0);
                }
            }
            mma_commit(&bar_pq);
        }
        __syncwarp();
    }
    const float A2 = p.scale * kLog2e;
    const bool exp_kind = p.kind == kKindExp;
    const int ew = warp - 1;  // epilogue warp index (warp 0 has -1)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    bool failed = false;
    float W = 0.f;
    if (warp > 0) {
        // ---------------- key side ----------------
        failed |= !mbar_wait(&bar_load, 0, &abort_flag);
        __syncwarp();
        if (exp_kind) {  // W = largest row norm of Omega (identical in every CTA of the cluster)
            float w2 = 0.f;
            for (int row = ew * 32 + lane; row < MP; row += 32 * kEpiWarps)
                w2 = fmaxf(w2, tile_row_sqnorm<64>(sOm + (size_t)(row >> 7) * 16384, row & 127));
            w2 = warp_max(w2);
            if (lane == 0) red[ew] = w2;
        }
        named_bar(1, 32 * kEpiWarps);
        if (exp_kind) {
            float m2 = 0.f;
#pragma unroll
            for (int i = 0; i < kEpiWarps; ++i) m2 = fmaxf(m2, red[i]);
            W = sqrtf(m2);
        }
        named_bar(1, 32 * kEpiWarps);
        // key norms and the tile's stabiliser (warps of column group 0 own the 128 key rows)
        if (ew < 4) {
            const bool valid = r < nvalid;
            const float kn2 = exp_kind ? p.scale * p.scale * tile_row_sqnorm<64>(sK, r) : 0.f;
            const float b = valid ? W * sqrtf(kn2) - 0.5f * kn2 : -INFINITY;
            const float bm = warp_max(b);
            if (lane == 0) red[ew] = bm;
            sC[r] = kn2;  // temporarily |k^|^2
        }
        named_bar(1, 32 * kEpiWarps);
        const float stab = exp_kind ? fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])) - kStabSlackLo : 0.f;
        named_bar(1, 32 * kEpiWarps);
        if (ew < 4) {
            const float kn2 = sC[r];
            sC[r] = r < nvalid ? (exp_kind ? (0.5f * kn2 + stab) * kLog2e : 0.f) : INFINITY;
            if (ew == 0 && lane == 0) sStab = stab;
        }
        named_bar(1, 32 * kEpiWarps);
        // phi^T for group tm (team of 8 warps), tokens [64 cg, 64 cg + 64) of the tile
        const int tm = ew / 8, cg = (ew % 8) >> 2;
        float zpart = 0.f;
        failed |= !mbar_wait(&bar_u, 0, &abort_flag);
        __syncwarp();
        tc_fence_after();
        if (tm < G) {
            const uint32_t ua = tbase + lane_off + 256 + 128 * tm + 64 * cg;
            uint32_t v[64];
            tmem_ld32(ua, *reinterpret_cast<uint32_t(*)[32]>(v));
            tmem_ld32(ua + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
            tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float* cj = sC + 64 * cg + 32 * hh;
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float a0 = __uint_as_float(v[32 * hh + i]), a1 = __uint_as_float(v[32 * hh + i + 1]);
                    float f0, f1;
                    if (exp_kind) {
                        f0 = ex2(fmaf(a0, A2, -cj[i]));
                        f1 = ex2(fmaf(a1, A2, -cj[i + 1]));
                    } else {
                        f0 = cj[i] == 0.f ? fmaxf(a0 * p.scale, 0.f) + p.relu_eps_s : 0.f;
                        f1 = cj[i + 1] == 0.f ? fmaxf(a1 * p.scale, 0.f) + p.relu_eps_s : 0.f;
                    }
                    zpart += f0 + f1;
                    pk[i / 2] = pack_bf16(f0, f1);
                }
                tmem_st16(ua + 16 * hh, pk);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_phi);
        // partial S (fp32) and z of this CTA into shared memory for the cluster reduction
        failed |= !mbar_wait(&bar_s, 0, &abort_flag);
        __syncwarp();
        tc_fence_after();
        if (tm < G) {
            sZp[cg * MP + tm * 128 + r] = zpart;
            const int feat = tm * 128 + r;
            uint32_t v[32];
            tmem_ld32(tbase + lane_off + 64 * tm + 32 * cg, v);
            tmem_ld_wait();
            float* dst = sP + (size_t)feat * 64 + 32 * cg;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + i) =
                    make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                                __uint_as_float(v[i + 3]));
        }
        tc_fence_before();
        __syncwarp();
    }
    cluster_sync();  // every CTA's partial S, z and stabiliser are in place

    // ---------------- cluster reduction: CTA rank owns feature rows [rank * R, rank * R + R) ----------------
    if (warp > 0) {
        float stabs[kMaxCluster];
        float M = -INFINITY;
        for (int c = 0; c < T; ++c) {
            stabs[c] = ld_cluster_f32(mapa(smem_u32(&sStab), c));
            M = fmaxf(M, stabs[c]);
        }
        const int R = (MP + T - 1) / T;
        const int e = ew * 32 + lane;
        const int part = e % 8;  // 8 threads per row, 8 columns each; 64 rows per pass
        for (int rr = e / 8; rr < R; rr += 32 * kEpiWarps / 8) {
            const int row = rank * R + rr;
            if (row >= MP) break;
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float zs = 0.f;
            for (int c = 0; c < T; ++c) {
                const float wgt = ex2((stabs[c] - M) * kLog2e);
                const uint32_t base = mapa(smem_u32(sP + (size_t)row * 64 + 8 * part), c);
                const uint4 a = ld_cluster_v4(base), b = ld_cluster_v4(base + 16);
                acc[0] = fmaf(wgt, __uint_as_float(a.x), acc[0]);
                acc[1] = fmaf(wgt, __uint_as_float(a.y), acc[1]);
                acc[2] = fmaf(wgt, __uint_as_float(a.z), acc[2]);
                acc[3] = fmaf(wgt, __uint_as_float(a.w), acc[3]);
                acc[4] = fmaf(wgt, __uint_as_float(b.x), acc[4]);
                acc[5] = fmaf(wgt, __uint_as_float(b.y), acc[5]);
                acc[6] = fmaf(wgt, __uint_as_float(b.z), acc[6]);
                acc[7] = fmaf(wgt, __uint_as_float(b.w), acc[7]);
                if (part == 0) {
                    const float z0 = ld_cluster_f32(mapa(smem_u32(sZp + row), c));
                    const float z1 = ld_cluster_f32(mapa(smem_u32(sZp + MP + row), c));
                    zs = fmaf(wgt, z0 + z1, zs);
                }
            }
            if (row >= p.m) {  // padding features contribute nothing
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                zs = 0.f;
            }
            const uint4 o = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                                       pack_bf16(acc[6], acc[7]));
            const uint32_t off = sw128_offset(row, part);
            for (int c = 0; c < T; ++c) {
                st_cluster_v4(mapa(smem_u32(sS + off), c), o);
                if (part == 0) st_cluster_f32(mapa(smem_u32(sz + row), c), zs);
            }
        }
        // the S image is read by the tensor cores (async proxy) of the receiving CTAs
        asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
        __syncwarp();
    }
    cluster_sync();  // every CTA holds the head's S image and z
    if (warp == 0) {
        if (lane == 0) {
            // numerator num = phi(Q) S (A = phi(Q) packed in TMEM, B = the S image, MN-major)
            fence_async_smem();
            constexpr uint32_t id_n = idesc_bf16(128, kD, false, true);
            const bool ok = mbar_wait(&bar_phiq, 0, &abort_flag);
            tc_fence_after();
            if (ok) {
                for (int ks = 0; ks < MP / 16; ++ks) {
                    uint64_t bd = sdesc_sw128(smem_u32(sS + ks * 2048), (uint32_t)MP * 128, 1024);
                    mma_ts(tbase, tbase + 256 + ks * 8, bd, id_n, ks > 0);
                }
            }
            mma_commit(&bar_num);
        }
        __syncwarp();
    }

    // ---------------- query side ----------------
    if (warp > 0) {
        const int cg4 = ew >> 2;  // column group: features [cg4 Wf, cg4 Wf + Wf), outputs [16 cg4, 16 cg4 + 16)
        const int Wf = MP / 4;
        failed |= !mbar_wait(&bar_pq, 0, &abort_flag);
        __syncwarp();
        tc_fence_after();
        const uint32_t ua = tbase + lane_off + 256 + cg4 * Wf;
        uint32_t v0[32], v1[32];
        tmem_ld32(ua, v0);
        if (Wf == 64) tmem_ld32(ua + 32, v1);
        tmem_ld_wait();
        float rmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) rmax = fmaxf(rmax, __uint_as_float(v0[i]));
        if (Wf == 64) {
#pragma unroll
            for (int i = 0; i < 32; ++i) rmax = fmaxf(rmax, __uint_as_float(v1[i]));
        }
        sMax[cg4 * 128 + r] = rmax;
        named_bar(1, 32 * kEpiWarps);  // every warp holds its U values: U may be overwritten now
        rmax = fmaxf(fmaxf(sMax[r], sMax[128 + r]), fmaxf(sMax[256 + r], sMax[384 + r]));
        const float cst = exp_kind ? A2 * rmax : 0.f;
        float dsum = 0.f;
        auto feat32 = [&](const uint32_t (&v)[32], int h) {
            const float* zr = sz + cg4 * Wf + 32 * h;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float f0, f1;
                if (exp_kind) {
                    f0 = ex2(fmaf(__uint_as_float(v[i]), A2, -cst));
                    f1 = ex2(fmaf(__uint_as_float(v[i + 1]), A2, -cst));
                } else {
                    f0 = fmaxf(__uint_as_float(v[i]) * p.scale, 0.f) + p.relu_eps_s;
                    f1 = fmaxf(__uint_as_float(v[i + 1]) * p.scale, 0.f) + p.relu_eps_s;
                }
                const uint32_t w = pack_bf16(f0, f1);
                pk[i / 2] = w;
                dsum = fmaf(__uint_as_float(w << 16), zr[i], dsum);
                dsum = fmaf(__uint_as_float(w & 0xFFFF0000u), zr[i + 1], dsum);
            }
            tmem_st16(tbase + lane_off + 256 + cg4 * (Wf / 2) + 16 * h, pk);
        };
        feat32(v0, 0);
        if (Wf == 64) feat32(v1, 1);
        tmem_st_wait();
        sDen[cg4 * 128 + r] = dsum;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_phiq);
        named_bar(1, 32 * kEpiWarps);  // denominator shares visible
        const float den = ((sDen[r] + sDen[128 + r]) + sDen[256 + r]) + sDen[384 + r];
        failed |= !mbar_wait(&bar_num, 0, &abort_flag);
        __syncwarp();
        tc_fence_after();
        uint32_t nv[16];
        tmem_ld16(tbase + lane_off + 16 * cg4, nv);
        tmem_ld_wait();
        if (r < nvalid) {
            const float inv = 1.f / den;
            uint4* dst = reinterpret_cast<uint4*>(p.Y + ((size_t)bh * p.n + j0 + r) * kD + 16 * cg4);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint4 o;
                o.x = pack_bf16(__uint_as_float(nv[8 * c + 0]) * inv, __uint_as_float(nv[8 * c + 1]) * inv);
                o.y = pack_bf16(__uint_as_float(nv[8 * c + 2]) * inv, __uint_as_float(nv[8 * c + 3]) * inv);
                o.z = pack_bf16(__uint_as_float(nv[8 * c + 4]) * inv, __uint_as_float(nv[8 * c + 5]) * inv);
                o.w = pack_bf16(__uint_as_float(nv[8 * c + 6]) * inv, __uint_as_float(nv[8 * c + 7]) * inv);
                dst[c] = o;
            }
        }
    }
    (void)failed;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
    cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

}  // namespace tcfu
}  // namespace favor
