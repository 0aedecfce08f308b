// Single-launch non-causal FAVOR+ for short sequences (bf16, d = 64, m <= 256, n <= 8 * 128).
//
// One thread-block cluster per head, one CTA per 128-token tile. Each CTA
//   1. projects its key tile with the features on the TMEM lanes, turns U^T into phi(K)^T in place
//      and accumulates its partial S = phi(K)^T V (tcgen05, A from TMEM) and z (per-lane sums), with
//      a key stabiliser of its own (the tile's exact largest exponent w_r . k^_j - |k^_j|^2 / 2);
//   2. writes the partial (fp32, straight from TMEM), its z and its stabiliser to the workspace in
//      global memory (L2) and arrives on a cluster barrier; while the barrier completes it projects
//      its query tile (tokens on the lanes) and forms phi(Q) in place with the exact row stabiliser;
//   3. sums the feature rows it owns ([c R, (c + 1) R) for CTA c) over the cluster's partials in
//      rank order, each rescaled to the cluster's largest stabiliser, writes the bf16 rows into its
//      own copy of the readout MMA's operand (swizzled, MN-major) and bulk-copies that contiguous
//      block into every peer (completing on the peer's mbarrier); z it sums for all rows itself and
//      stores as a bf16 hi + lo pair in two extra operand columns; for the exp family the rounding
//      remainder of S (S - bf16(S), itself in bf16) goes the same way in a second operand;
//   4. once the peers' blocks have landed, takes [num | den] = phi(Q) [S | z_hi + z_lo] in one MMA
//      chain (N = 64 + 16), adds phi(Q) S_lo (exp family) and stores Y = num / den.
// Distributed shared memory carries only the bf16 rows (per SM its bandwidth is far below L2's), in
// bulk copies of whole row blocks.
#pragma once

#include "tc.cuh"
#include "tc_noncausal.cuh"  // ex2, tile_row_sqnorm, phi_col

namespace favor {
namespace tcfu {

using namespace favor::tc;
using tcnc::ex2;
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
    float4* Pp;        // [BH][T][16][m_pad] partial S: float4 column group c4 of feature row f at (c4, f)
    float* Zp;         // [BH][T][2][m_pad] partial z of the two 64-token halves
    float* Stab;       // [BH][kMaxCluster] key stabiliser of each CTA
};

// Workspace of one call: the partials of every CTA, 256-byte aligned pieces.
inline size_t fused_ws_part(size_t b) { return (b + 255) & ~size_t(255); }
inline size_t fused_ws_pp_bytes(int BH, int T, int m_pad) { return (size_t)BH * T * m_pad * 256; }
inline size_t fused_ws_bytes(int BH, int T, int m_pad) {
    return fused_ws_part(fused_ws_pp_bytes(BH, T, m_pad)) + fused_ws_part((size_t)BH * T * 2 * m_pad * 4) +
           fused_ws_part((size_t)BH * kMaxCluster * 4);
}

struct FusedSmem {
    // Omega (m_pad x 128 B), K, V, Q tiles, the readout's B operand (two 64-column MN regions of
    // m_pad x 128 B: S, then z_hi, z_lo and zeros), per-key constants, row-max exchange.
    static size_t bytes(int m_pad) {
        return 1024 + (size_t)m_pad * 128 + 3 * kTileBytes + 3 * (size_t)m_pad * 128 + 128 * 4 + 4 * 128 * 4;
    }
};

template <int KIND>
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
    uint8_t* sS = sQ + kTileBytes;                         // bf16 [S | z] operand, 2 x MP x 128 B
    uint8_t* sSlo = sS + 2 * (size_t)MP * 128;             // bf16 S - bf16(S) operand, MP x 128 B
    float* sC = reinterpret_cast<float*>(sSlo + (size_t)MP * 128);  // [128] per-key constants
    float* sMax = sC + 128;                                // [4][128] row-max shares
    __shared__ uint64_t bar_load, bar_q, bar_u, bar_phi, bar_s, bar_pq, bar_phiq, bar_num, bar_own, bar_img;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float red[kEpiWarps];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int T = (int)cluster_size();   // tiles of the head = CTAs of the cluster
    const int rank = (int)cluster_rank();
    const int bh = blockIdx.x / T;
    const int j0 = rank * kTile;         // this CTA's tile
    const int nvalid = min(kTile, p.n - j0);
    const int R = (MP + T - 1) / T;      // feature rows owned by each CTA
    const int own_lo = min(MP, rank * R);
    const int own_rows = min(MP, own_lo + R) - own_lo;

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
        mbar_init(&bar_own, kEpiWarps);
        mbar_init(&bar_img, 1);
        fence_mbar_init();
        // the peers' rows of the operand (and of the remainder, exp family) arrive by bulk copies
        // (after the first cluster barrier)
        mbar_arrive_expect_tx(&bar_img, (uint32_t)(MP - own_rows) * 128 * (KIND == kKindExp ? 2u : 1u));
        // the loads start before the TMEM allocation and the CTA barrier
        tma_prefetch_desc(&mQ);
        tma_prefetch_desc(&mK);
        tma_prefetch_desc(&mV);
        tma_prefetch_desc(&mOm);
        mbar_arrive_expect_tx(&bar_load, (uint32_t)MP * 128 + 2 * kTileBytes);
        tma_load_3d(sK, &mK, &bar_load, 0, j0, bh);
        for (int r0 = 0; r0 < MP; r0 += 128) tma_load_2d(sOm + (size_t)r0 * 128, &mOm, &bar_load, 0, r0);
        tma_load_3d(sV, &mV, &bar_load, 0, j0, bh);
        mbar_arrive_expect_tx(&bar_q, kTileBytes);
        tma_load_3d(sQ, &mQ, &bar_q, 0, j0, bh);
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(&tmem_base, 512);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    // TMEM: S_g at [64 g, 64 g + 64); U^T of group g at 256 + 128 g; later U(Q) at [256, 256 + MP)
    // with phi(Q) packed in its first MP/2 columns, and [num | den] at [0, 80).

    if (warp == 0) {
        if (lane == 0) {
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
    const bool exp_kind = KIND == kKindExp;
    const int ew = warp - 1;  // epilogue warp index (warp 0 has -1)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int cg4 = ew >> 2;  // query side column group: features [cg4 Wf, cg4 Wf + Wf), outputs [16 cg4, +16)
    const int Wf = MP / 4;
    bool failed = false;
    if (warp > 0) {
        // ---------------- key side ----------------
        failed |= !mbar_wait(&bar_load, 0, &abort_flag);
        __syncwarp();
        // warps 1..4 own the tile's 128 keys: the per-key part of the exponent, |k^|^2 / 2 (binary
        // orders of magnitude), +inf for keys past n
        if (ew < 4) {
            const float kn2 = exp_kind ? p.scale * p.scale * tile_row_sqnorm<64>(sK, r) : 0.f;
            sC[r] = r < nvalid ? 0.5f * kn2 * kLog2e : INFINITY;
        }
        named_bar(1, 32 * kEpiWarps);
        // phi^T for group tm (team of 8 warps), tokens [64 cg, 64 cg + 64) of the tile
        const int tm = ew / 8, cg = (ew % 8) >> 2;
        float zpart = 0.f;
        failed |= !mbar_wait(&bar_u, 0, &abort_flag);
        __syncwarp();
        tc_fence_after();
        uint32_t v[64];
        if (tm < G) {
            const uint32_t ua = tbase + lane_off + 256 + 128 * tm + 64 * cg;
            tmem_ld32(ua, *reinterpret_cast<uint32_t(*)[32]>(v));
            tmem_ld32(ua + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
            tmem_ld_wait();
        }
        // The tile's key stabiliser: the exact largest exponent w_r . k^_j - |k^_j|^2 / 2 over its
        // valid keys and real features (the tile's largest key feature is then 1).
        float stab = 0.f;  // binary orders of magnitude
        if (exp_kind) {
            float mx = -INFINITY;
            if (tm < G && tm * 128 + r < p.m) {
#pragma unroll
                for (int i = 0; i < 64; ++i) mx = fmaxf(mx, fmaf(__uint_as_float(v[i]), A2, -sC[64 * cg + i]));
            }
            mx = warp_max(mx);
            if (lane == 0) red[ew] = mx;
            named_bar(1, 32 * kEpiWarps);
            stab = -INFINITY;
#pragma unroll
            for (int i = 0; i < kEpiWarps; ++i) stab = fmaxf(stab, red[i]);
        }
        const bool real_feat = tm * 128 + r < p.m;  // padding features get phi = 0
        if (tm < G) {
            const uint32_t ua = tbase + lane_off + 256 + 128 * tm + 64 * cg;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float* cj = sC + 64 * cg + 32 * hh;
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float a0 = __uint_as_float(v[32 * hh + i]), a1 = __uint_as_float(v[32 * hh + i + 1]);
                    float f0, f1;
                    if (exp_kind) {
                        f0 = ex2(fmaf(a0, A2, -(cj[i] + stab)));
                        f1 = ex2(fmaf(a1, A2, -(cj[i + 1] + stab)));
                    } else {
                        f0 = cj[i] == 0.f ? phi_plain(a0 * p.scale, KIND, 1.f, p.relu_eps_s) : 0.f;
                        f1 = cj[i + 1] == 0.f ? phi_plain(a1 * p.scale, KIND, 1.f, p.relu_eps_s) : 0.f;
                    }
                    if (!real_feat) f0 = f1 = 0.f;
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
        // the partial S row (fp32) and z of feature tm*128 + r to the workspace; a warp's 32 rows of
        // one float4 column group are 512 contiguous bytes
        failed |= !mbar_wait(&bar_s, 0, &abort_flag);
        __syncwarp();
        tc_fence_after();
        if (tm < G && FAVOR_IN_BOUNDS(bh * T + rank < (int)gridDim.x && tm * 128 + r < MP)) {
            const int feat = tm * 128 + r;
            uint32_t v[32];
            tmem_ld32(tbase + lane_off + 64 * tm + 32 * cg, v);
            tmem_ld_wait();
            float4* dst = p.Pp + ((size_t)(bh * T + rank) * 16 + 8 * cg) * MP + feat;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                __stcg(dst + (size_t)c * MP, make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                                         __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3])));
            __stcg(p.Zp + ((size_t)(bh * T + rank) * 2 + cg) * MP + feat, zpart);
        }
        if (ew == 0 && lane == 0) __stcg(p.Stab + bh * kMaxCluster + rank, stab / kLog2e);
        tc_fence_before();
        __syncwarp();
    }

    // ---------------- phi(Q), while the workspace stores drain ----------------
    if (warp > 0) {
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
        auto feat32 = [&](const uint32_t (&v)[32], int h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float f0, f1;
                if (exp_kind) {
                    f0 = ex2(fmaf(__uint_as_float(v[i]), A2, -cst));
                    f1 = ex2(fmaf(__uint_as_float(v[i + 1]), A2, -cst));
                } else {
                    f0 = phi_plain(__uint_as_float(v[i]) * p.scale, KIND, 1.f, p.relu_eps_s);
                    f1 = phi_plain(__uint_as_float(v[i + 1]) * p.scale, KIND, 1.f, p.relu_eps_s);
                }
                pk[i / 2] = pack_bf16(f0, f1);
            }
            tmem_st16(tbase + lane_off + 256 + cg4 * (Wf / 2) + 16 * h, pk);
        };
        feat32(v0, 0);
        if (Wf == 64) feat32(v1, 1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_phiq);
        __syncwarp();
    }
    cluster_arrive();  // (partials) this CTA's workspace writes are visible to the peers after the wait
    cluster_wait();    // every CTA's partial S, z and stabiliser are in the workspace

    // ---------------- reduction: z of every row, S of the owned rows [rank R, rank R + R) ----------------
    if (warp > 0) {
        // every load of this phase (stabilisers, z partials, S partials) is issued before the first
        // use of any of them: one L2 round trip
        float wgt[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) wgt[c] = c < T ? __ldcg(p.Stab + bh * kMaxCluster + c) : -INFINITY;
        bool have_w = false;
        auto weights = [&] {  // each partial's scale: exp(stab_c - largest stab)
            if (have_w) return;
            have_w = true;
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) M = fmaxf(M, wgt[c]);
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) wgt[c] = c < T ? ex2((wgt[c] - M) * kLog2e) : 0.f;
        };
        // z (every CTA sums the head's z partials itself; thread ew * 32 + lane takes feature row
        // fz, m_pad <= 512 threads) as operand columns 64 (hi) and 65 (lo) of the second MN region,
        // columns 66..79 zero. Its loads are issued with those of the S rows below.
        const int fz = ew * 32 + lane;
        float zl[2 * kMaxCluster];
        {
            const float* zsrc = p.Zp + (size_t)bh * T * 2 * MP + fz;
#pragma unroll
            for (int c = 0; c < 2 * kMaxCluster; ++c) zl[c] = (fz < MP && c < 2 * T) ? __ldcg(zsrc + (size_t)c * MP) : 0.f;
        }
        const int c4 = ew;  // this warp's float4 column group: S columns [4 c4, 4 c4 + 4)
        const float4* src = p.Pp + (size_t)bh * T * 16 * MP + (size_t)c4 * MP;
        for (int i = lane; i < own_rows; i += 32) {
            const int row = own_lo + i;
            float4 a[kMaxCluster];
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)  // all loads in flight
                if (c < T) a[c] = __ldcg(src + (size_t)c * 16 * MP + row);
            weights();
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) {  // rank order
                if (c < T) {
                    acc[0] = fmaf(wgt[c], a[c].x, acc[0]);
                    acc[1] = fmaf(wgt[c], a[c].y, acc[1]);
                    acc[2] = fmaf(wgt[c], a[c].z, acc[2]);
                    acc[3] = fmaf(wgt[c], a[c].w, acc[3]);
                }
            }
            if (row >= p.m) {  // padding features contribute nothing
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = 0.f;
            }
            const uint32_t off = sw128_offset(row, c4 >> 1) + 8 * (c4 & 1);
            const uint2 hi = make_uint2(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]));
            *reinterpret_cast<uint2*>(sS + off) = hi;
            if (exp_kind)
                *reinterpret_cast<uint2*>(sSlo + off) =
                    make_uint2(pack_bf16(acc[0] - __uint_as_float(hi.x << 16), acc[1] - __uint_as_float(hi.x & 0xFFFF0000u)),
                               pack_bf16(acc[2] - __uint_as_float(hi.y << 16), acc[3] - __uint_as_float(hi.y & 0xFFFF0000u)));
        }
        if (fz < MP) {
            weights();
            float z = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) z = fmaf(wgt[c], zl[2 * c] + zl[2 * c + 1], z);
            if (fz >= p.m) z = 0.f;  // padding features contribute nothing
            const float zh = __bfloat162float(__float2bfloat16_rn(z));
            uint8_t* zrow = sS + (size_t)MP * 128 + (size_t)fz * 128;
            *reinterpret_cast<uint4*>(zrow + ((0u ^ (fz & 7u)) << 4)) = make_uint4(pack_bf16(zh, z - zh), 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(zrow + ((1u ^ (fz & 7u)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();  // the rows are read by the bulk-copy engine and the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_own);
        named_bar(1, 32 * kEpiWarps);  // the owned rows are complete
        if (ew == 0 && lane == 0 && own_rows > 0) {
            // the owned rows are one contiguous block of the operand: copy it into every peer
            const uint32_t off = (uint32_t)own_lo * 128;
            for (int c = 0; c < T; ++c)
                if (c != rank) {
                    bulk_copy_to_peer(mapa(smem_u32(sS + off), c), sS + off, (uint32_t)own_rows * 128,
                                      mapa(smem_u32(&bar_img), c));
                    if (exp_kind)
                        bulk_copy_to_peer(mapa(smem_u32(sSlo + off), c), sSlo + off, (uint32_t)own_rows * 128,
                                          mapa(smem_u32(&bar_img), c));
                }
        }
        __syncwarp();
    }
    if (warp == 0) {
        if (lane == 0) {
            // [num | den] = phi(Q) [S | z] (A = phi(Q) packed in TMEM, B = the operand, MN-major,
            // N = 80: the S region and the first 16 columns of the z region)
            constexpr uint32_t id_n = idesc_bf16(128, kD + 16, false, true);
            const bool ok = mbar_wait(&bar_own, 0, &abort_flag) && mbar_wait(&bar_img, 0, &abort_flag) &&
                            mbar_wait(&bar_phiq, 0, &abort_flag);
            tc_fence_after();
            if (ok) {
                for (int ks = 0; ks < MP / 16; ++ks) {
                    uint64_t bd = sdesc_sw128(smem_u32(sS + ks * 2048), (uint32_t)MP * 128, 1024);
                    mma_ts(tbase, tbase + 256 + ks * 8, bd, id_n, ks > 0);
                }
                if (KIND == kKindExp) {
                    constexpr uint32_t id_lo = idesc_bf16(128, kD, false, true);
                    for (int ks = 0; ks < MP / 16; ++ks) {
                        uint64_t bd = sdesc_sw128(smem_u32(sSlo + ks * 2048), 16, 1024);
                        mma_ts(tbase, tbase + 256 + ks * 8, bd, id_lo, 1u);
                    }
                }
            }
            mma_commit(&bar_num);
        }
        __syncwarp();
        // every peer's bulk copy into this CTA has landed (bar_img); arrive for the closing barrier
        cluster_arrive();
    }

    // ---------------- the output ----------------
    if (warp > 0) {
        failed |= !mbar_wait(&bar_num, 0, &abort_flag);
        __syncwarp();
        cluster_arrive();  // the MMA has consumed the peers' rows: this CTA needs nothing more from them
        tc_fence_after();
        uint32_t nv[16], d0, d1;
        tmem_ld16(tbase + lane_off + 16 * cg4, nv);
        tmem_ld2(tbase + lane_off + kD, d0, d1);
        tmem_ld_wait();
        if (r < nvalid && FAVOR_IN_BOUNDS(j0 + r < p.n && bh * T + rank < (int)gridDim.x && 16 * cg4 + 16 <= kD)) {
            const float inv = 1.f / (__uint_as_float(d0) + __uint_as_float(d1));
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
    // no CTA leaves while a bulk copy out of its shared memory may still be running: every CTA
    // arrives only once all copies into it have landed
    cluster_wait();
}

}  // namespace tcfu
}  // namespace favor
