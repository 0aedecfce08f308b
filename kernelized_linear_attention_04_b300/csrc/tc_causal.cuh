// Tensor-core (tcgen05 + TMA + TMEM) causal FAVOR+ scan, bf16 in / fp32 accumulate, d = 64.
//
// One CTA walks the 128-token tiles of one head in order. Per tile t (rows i, keys j of the tile):
//   num_i = phi(q_i) S_<t + sum_{j <= i} (phi(q_i) . phi(k_j)) v_j
//   den_i = phi(q_i) z_<t + sum_{j <= i}  phi(q_i) . phi(k_j)
//   y_i   = num_i / den_i;   then S_<t+1 = S_<t + Phi(K_t)^T V_t,  z_<t+1 = z_<t + Phi(K_t)^T 1.
// The prefix state is carried at every tile boundary (128 tokens); within a tile the keys are
// masked by j <= i, which for two 64-token chunks is exactly their chunked prefix-sum result.
//
// Each CTA holds one 128-feature group of the head; a head of 256 features is spread over a
// thread-block cluster of 2 CTAs whose partial numerators and denominators are summed through
// distributed shared memory once per tile (wider heads run the one-tile-at-a-time scan of
// tc_causal_wide.cuh).
//
// The tiles run as a software pipeline over four roles:
//   warp 0      TMA producer: Q, K (single buffers) and V (two buffers) of the coming tiles;
//   warp 1      MMA issuer, in the order [inter(t)] [intra(t-1)] [proj Q(t+1)] [scores(t), state(t)]
//               [proj K(t+1)]: the inter numerator runs while phi(K_t) is formed, the previous
//               tile's intra numerator as soon as its masked scores are in place, and phi(Q_{t+1})
//               is computed while tile t's MMAs run;
//   warps 2-9   feature team: phi(Q_t), phi(K_t) from the projections (TMEM) into shared memory, and
//               the inter-tile part of the denominator, phi(q) . z_<t;
//   warps 10-17 output team: the masked scores A~ (converted in place in TMEM into bf16 hi + lo, the
//               A operand of the intra MMA), the bf16 hi + lo snapshot of the state for the next
//               tile, and the output (cluster sum, num / den, Y).
// The numerator has two TMEM buffers, so the inter MMA of tile t+1 need not wait for the output of
// tile t. Tensor-core work per tile: U = X Omega^T (two projections), scores phi(Q) phi(K)^T, inter
// phi(Q) (S_hi + S_lo), state [S | z] += phi(K)^T [V | 1], intra (A~hi + A~lo) V.
//
// Stabilisers: a query row uses c_i = W |q^_i| (W = largest row norm of Omega; Cauchy-Schwarz bounds
// every w_r . q^_i by it). Keys use one constant per head, 12 nats below the largest bound
// W |k^_j| - |k^_j|^2 / 2 over all of the head's keys, found by a pass over K before the scan. Both
// cancel in num / den; the common 1/sqrt(m) is dropped.
#pragma once

#include "tc.cuh"
#include "tc_noncausal.cuh"  // shared helpers: ex2, tile_row_sqnorm, sq_acc_bf16x2, slack constant

namespace favor {
namespace tcc {

using namespace favor::tc;
using tcnc::ex2;
using tcnc::kStabSlackLo;
using tcnc::sq_acc_bf16x2;
using tcnc::tile_row_sqnorm;

constexpr int kTile = 128;
constexpr int kD = 64;                       // head dimension handled by this kernel
constexpr int kFeat = 128;                   // features per CTA
constexpr int kTeamWarps = 8;                // warps of the feature team and of the output team
constexpr int kThreads = 64 + 2 * 32 * kTeamWarps;
constexpr int kTileBytes = kTile * kD * 2;   // 16 KB: one [128 x 64] bf16 tile
constexpr int kPhiBytes = kTile * 128 * 2;   // 32 KB: [128 tokens x 128 features] bf16, two K atoms
constexpr int kXStride = 84;                 // floats per row of the cluster exchange buffer (64 + den + pad)

// TMEM columns
constexpr uint32_t kColS = 0;      // S: 64 columns, then z (column 64) and 15 zero columns
constexpr uint32_t kColU = 128;    // projection output, 128 columns
constexpr uint32_t kColSc = 256;   // scores; then A~ in place: keys [16 s, 16 s + 16) -> hi at 16 s, lo at 16 s + 8
constexpr uint32_t kColNum = 384;  // numerator, two buffers of 64 columns

struct CausalParams {
    int n;
    int m;
    int kind;
    float relu_eps_s;
    float scale;
    const __nv_bfloat16* K;  // [BH][n][64] keys, read directly by the stabiliser pass
    __nv_bfloat16* Y;
};

struct CausalSmem {
    // Omega rows of the CTA (128 x 64, K-major), Q, K, two V tiles, the state snapshot as hi and lo
    // bf16 images (128 x 64, MN-major), phi(Q), phi(K), the ones column (128 x 64 bf16, MN-major:
    // the second N region of the state MMA's B operand [V | 1]), z snapshots (2 x 128 fp32),
    // denominator shares (6 x 128 fp32), cluster exchange buffer.
    static size_t x_bytes(int cs) { return cs > 1 ? (size_t)(cs - 1) * (kTile / cs) * kXStride * 4 : 0; }
    static size_t bytes(int cs) {
        return 1024 + 8 * (size_t)kTileBytes + 2 * (size_t)kPhiBytes + 8 * 128 * 4 + x_bytes(cs);
    }
};

__global__ void __launch_bounds__(kThreads, 1)
    causal_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
              const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mOm, CausalParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 by hand below
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // A head's features are split over the CS CTAs of a cluster: CTA `rank` owns features
    // [rank * 128, rank * 128 + 128). The partial numerators and denominators of a tile are summed
    // in the CTA that finalises the row: CTA `rank` owns the rows [rank * RP, (rank + 1) * RP).
    const int CS = (int)cluster_size();
    const int rank = (int)cluster_rank();
    const int RP = kTile / CS;
    const int feat0 = rank * kFeat;
    uint8_t* sOm = smem;                       // 128 rows x 128 B
    uint8_t* sQ = sOm + kTileBytes;
    uint8_t* sK = sQ + kTileBytes;
    uint8_t* sV0 = sK + kTileBytes;            // V of even tiles, then V of odd tiles
    uint8_t* sS = sV0 + 2 * kTileBytes;        // state snapshot hi: 128 feature rows x 128 B (MN-major)
    uint8_t* sSl = sS + kTileBytes;            // state snapshot lo (S - hi, rounded)
    uint8_t* sPQ = sSl + kTileBytes;           // phi(Q): 2 K-atom regions of 128 rows x 128 B
    uint8_t* sPK = sPQ + kPhiBytes;            // phi(K)
    uint8_t* sOnes = sPK + kPhiBytes;          // 128 token rows x 128 B: column 0 = 1, the rest 0
    float* sZ = reinterpret_cast<float*>(sOnes + kTileBytes);  // [2][128] z snapshot by tile parity
    float* sDenF = sZ + 2 * 128;               // [2 parity][2 half][128] phi(q) . z_<t shares
    float* sDenO = sDenF + 4 * 128;            // [2 half][128] masked score row sums
    float* sX = sDenO + 2 * 128;               // [CS - 1][RP][kXStride] partial sums from the peers
    __shared__ uint64_t bar_om, bar_qfull, bar_kfull, bar_qkempty, bar_vfull[2], bar_vempty[2];
    __shared__ uint64_t bar_ufull, bar_ufree, bar_phq, bar_phk, bar_snap, bar_grp, bar_atil, bar_num;
    __shared__ uint64_t bar_dfree[2], bar_den[2];
    __shared__ uint64_t bar_xfree, bar_xfull;  // cluster exchange of the partial sums
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float sWred[kThreads / 32];
    __shared__ float sW[4];   // per-rank largest squared row norm of Omega
    __shared__ float sKB[4];  // per-rank largest key bound

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x / CS;
    const int T = (p.n + kTile - 1) / kTile;
    const bool exp_kind = p.kind == kKindExp;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_om, 1);
        mbar_init(&bar_qfull, 1);
        mbar_init(&bar_kfull, 1);
        mbar_init(&bar_qkempty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar_vfull[b], 1);
            mbar_init(&bar_vempty[b], 1);
            mbar_init(&bar_dfree[b], kTeamWarps);
            mbar_init(&bar_den[b], kTeamWarps);
        }
        mbar_init(&bar_ufull, 1);
        mbar_init(&bar_ufree, kTeamWarps);
        mbar_init(&bar_phq, kTeamWarps);
        mbar_init(&bar_phk, kTeamWarps);
        mbar_init(&bar_snap, kTeamWarps);
        mbar_init(&bar_grp, 1);
        mbar_init(&bar_atil, kTeamWarps);
        mbar_init(&bar_num, 1);
        mbar_init(&bar_xfree, CS > 1 ? CS - 1 : 1);
        mbar_init(&bar_xfull, CS > 1 ? (CS - 1) * (RP / 32) * 2 : 1);
        fence_mbar_init();
    }
    // the ones column: z = phi(K)^T 1 comes out of the state MMA as its 65th output column. In the
    // 128-byte-swizzled MN-major layout, column 0 of token row k sits in 16-byte chunk (k mod 8).
    for (int i = threadIdx.x; i < kTileBytes / 16; i += blockDim.x) {
        const int row = i >> 3, chunk = i & 7;
        reinterpret_cast<uint4*>(sOnes)[i] = make_uint4(chunk == (row & 7) ? 0x00003F80u : 0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    if (warp == 1) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    cluster_sync();  // every CTA's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tbase = tmem_base;

    // Omega rows of this CTA, then W = largest row norm of Omega over the whole cluster: the query
    // stabiliser c_i = W |q^_i| and the key bound must be the same in every CTA of the cluster.
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&mOm);
        mbar_arrive_expect_tx(&bar_om, (uint32_t)kTileBytes);
        tma_load_2d(sOm, &mOm, &bar_om, 0, feat0);
    }
    bool om_ok = mbar_wait(&bar_om, 0, &abort_flag);
    {
        float w2 = 0.f;
        if (exp_kind && threadIdx.x < kFeat) w2 = tile_row_sqnorm<64>(sOm, threadIdx.x);
        w2 = warp_max(w2);
        if (lane == 0) sWred[warp] = w2;
        __syncthreads();
        if (threadIdx.x == 0) {
            float m2 = 0.f;
            for (int i = 0; i < kThreads / 32; ++i) m2 = fmaxf(m2, sWred[i]);
            for (int c = 0; c < CS; ++c) st_cluster_f32(mapa(smem_u32(&sW[rank]), c), m2);
        }
        cluster_sync();
    }
    float W = 0.f;
    for (int c = 0; c < CS; ++c) W = fmaxf(W, sW[c]);
    W = sqrtf(W);
    (void)om_ok;

    // Key stabiliser of the head: the CTAs of the cluster take the tiles t = rank (mod CS) and read
    // the keys straight from global memory (four tiles of loads in flight per thread), then
    // exchange their maxima.
    float stab = 0.f;
    const float s2 = p.scale * p.scale;
    if (exp_kind) {
        float kb = -INFINITY;
        if (warp >= 2) {
            const int e = threadIdx.x - 64;
            const int sub = e & 7, rr = e >> 3;  // 16-byte chunk of the row, row within a 64-row step
            const uint4* Kh = reinterpret_cast<const uint4*>(p.K + (size_t)bh * p.n * kD);
            constexpr int kU = 4;
            for (int t0 = rank; t0 < T; t0 += kU * CS) {
                uint4 v[2 * kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int tt = t0 + u * CS;
                        const int j = tt * kTile + s * 64 + rr;
                        v[2 * u + s] = (tt < T && j < p.n) ? __ldg(Kh + (size_t)j * 8 + sub) : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int tt = t0 + u * CS;
                        const int j = tt * kTile + s * 64 + rr;
                        float a0 = 0.f, a1 = 0.f;
                        sq_acc_bf16x2(v[2 * u + s].x, a0, a1);
                        sq_acc_bf16x2(v[2 * u + s].y, a0, a1);
                        sq_acc_bf16x2(v[2 * u + s].z, a0, a1);
                        sq_acc_bf16x2(v[2 * u + s].w, a0, a1);
                        float ss = a0 + a1;  // the 8 lanes of a row hold its 8 chunks
                        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                        const float kn2 = s2 * ss;
                        if (tt < T && j < p.n) kb = fmaxf(kb, W * sqrtf(kn2) - 0.5f * kn2);
                    }
                }
            }
        }
        kb = warp_max(kb);
        if (lane == 0) sWred[warp] = kb;
        __syncthreads();
        if (threadIdx.x == 0) {
            float mx = -INFINITY;
            for (int i = 0; i < kThreads / 32; ++i) mx = fmaxf(mx, sWred[i]);
            for (int c = 0; c < CS; ++c) st_cluster_f32(mapa(smem_u32(&sKB[rank]), c), mx);
        }
        cluster_sync();
        float Bk = -INFINITY;
        for (int c = 0; c < CS; ++c) Bk = fmaxf(Bk, sKB[c]);
        stab = Bk - kStabSlackLo;
    }

    if (warp == 0) {
        // ---------------- TMA producer (lane 0) ----------------
        if (lane == 0) {
            tma_prefetch_desc(&mQ);
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mV);
            bool ok = true;
            for (int t = 0; t < T && ok; ++t) {
                const int b = t & 1;
                // Q and K of tile t once both projections of tile t-1 are done; V of tile t once the
                // intra MMA of tile t-2 (the last reader of its buffer) is done.
                if (!(ok = mbar_wait(&bar_qkempty, (t & 1) ^ 1, &abort_flag))) break;
                mbar_arrive_expect_tx(&bar_qfull, kTileBytes);
                tma_load_3d(sQ, &mQ, &bar_qfull, 0, t * kTile, bh);
                mbar_arrive_expect_tx(&bar_kfull, kTileBytes);
                tma_load_3d(sK, &mK, &bar_kfull, 0, t * kTile, bh);
                if (!(ok = mbar_wait(&bar_vempty[b], ((t >> 1) & 1) ^ 1, &abort_flag))) break;
                mbar_arrive_expect_tx(&bar_vfull[b], kTileBytes);
                tma_load_3d(sV0 + b * kTileBytes, &mV, &bar_vfull[b], 0, t * kTile, bh);
            }
            // Drain the loads in flight before the CTA may exit.
            volatile int never = 0;
            if (T > 0) {
                mbar_wait(&bar_qfull, (T - 1) & 1, &never);
                mbar_wait(&bar_kfull, (T - 1) & 1, &never);
                mbar_wait(&bar_vfull[(T - 1) & 1], ((T - 1) >> 1) & 1, &never);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (lane 0) ----------------
        if (lane == 0) {
            constexpr uint32_t id_proj = idesc_bf16(128, 128, false, false);  // U = X Om^T
            constexpr uint32_t id_sc = idesc_bf16(128, 128, false, false);    // phi(Q) phi(K)^T
            constexpr uint32_t id_num = idesc_bf16(128, kD, false, true);     // phi(Q) S, A~ V
            constexpr uint32_t id_st = idesc_bf16(128, kD + 16, true, true);  // phi(K)^T [V | 1]
            bool ok = true;
            int pu = 0;  // projections issued into the one U slot
            auto proj = [&](const uint8_t* x, uint64_t* full, uint32_t parity) -> bool {
                if (!mbar_wait(full, parity, &abort_flag)) return false;
                if (pu > 0 && !mbar_wait(&bar_ufree, (pu - 1) & 1, &abort_flag)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    uint64_t ad = sdesc_sw128(smem_u32(x + ks * 32), 16, 1024);
                    uint64_t bd = sdesc_sw128(smem_u32(sOm + ks * 32), 16, 1024);
                    mma_ss(tbase + kColU, ad, bd, id_proj, ks > 0);
                }
                mma_commit(&bar_ufull);
                ++pu;
                return true;
            };
            // intra numerator of tile u: Num += (A~hi + A~lo) V_u, A from TMEM (K = 128 keys); A~ must be
            // consumed before the next scores MMA overwrites it
            auto intra = [&](int u) -> bool {
                if (!mbar_wait(&bar_atil, u & 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* vu = sV0 + (u & 1) * kTileBytes;
                const uint32_t nu = tbase + kColNum + 64 * (u & 1);
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        uint64_t bd = sdesc_sw128(smem_u32(vu + ks * 2048), 16, 1024);
                        mma_ts(nu, tbase + kColSc + 16 * ks + 8 * part, bd, id_num, 1);
                    }
                }
                mma_commit(&bar_num);
                mma_commit(&bar_vempty[u & 1]);
                return true;
            };
            if (T > 0) {
                ok = proj(sQ, &bar_qfull, 0) && proj(sK, &bar_kfull, 0);
                if (ok) mma_commit(&bar_qkempty);
            }
            for (int t = 0; t < T && ok; ++t) {
                const int b = t & 1;
                const uint8_t* vt = sV0 + b * kTileBytes;
                const uint32_t nb = tbase + kColNum + 64 * b;
                // inter numerator phi(Q) (S_hi + S_lo) (the state as taken at the tile start) as soon
                // as phi(Q) and the snapshot are in place: it runs while phi(K) is formed
                ok = mbar_wait(&bar_phq, t & 1, &abort_flag) && mbar_wait(&bar_snap, t & 1, &abort_flag) &&
                     mbar_wait(&bar_dfree[b], ((t >> 1) & 1) ^ 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                for (int part = 0; part < 2; ++part) {
                    const uint8_t* sp = part == 0 ? sS : sSl;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int a = ks / 4, w = ks % 4;
                        uint64_t ad = sdesc_sw128(smem_u32(sPQ + a * 16384 + w * 32), 16, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(sp + ks * 16 * 128), 16, 1024);
                        mma_ss(nb, ad, bd, id_num, part > 0 || ks > 0);
                    }
                }
                // the previous tile's intra numerator (its A~ is ready by now, or soon)
                if (t > 0 && !(ok = intra(t - 1))) break;
                // projection of the next tile's queries as soon as U is free (the feature team has read
                // tile t's keys from it), so that phi(Q_{t+1}) is computed while tile t's MMAs run
                if (t + 1 < T && !(ok = proj(sQ, &bar_qfull, (t + 1) & 1))) break;
                ok = mbar_wait(&bar_phk, t & 1, &abort_flag) && mbar_wait(&bar_vfull[b], (t >> 1) & 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                // scores (K = 128 features, two K atoms)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int a = ks / 4, w = ks % 4;
                    uint64_t ad = sdesc_sw128(smem_u32(sPQ + a * 16384 + w * 32), 16, 1024);
                    uint64_t bd = sdesc_sw128(smem_u32(sPK + a * 16384 + w * 32), 16, 1024);
                    mma_ss(tbase + kColSc, ad, bd, id_sc, ks > 0);
                }
                // state update: [S | z] += phi(K)^T [V_t | 1] (K = 128 tokens, N = 64 + 16; the ones
                // column is the B operand's second N region, LBO bytes after the V tile)
                const uint32_t lbo_ones = (uint32_t)(sOnes - vt);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint64_t ad = sdesc_sw128(smem_u32(sPK + ks * 2048), 16384, 1024);
                    uint64_t bd = sdesc_sw128(smem_u32(vt + ks * 2048), lbo_ones, 1024);
                    mma_ss(tbase + kColS, ad, bd, id_st, t > 0 || ks > 0);
                }
                mma_commit(&bar_grp);
                // projection of the next tile's keys while the output team forms A~
                if (t + 1 < T) {
                    if (!(ok = proj(sK, &bar_kfull, (t + 1) & 1))) break;
                    mma_commit(&bar_qkempty);
                }
            }
            if (ok && T > 0) intra(T - 1);
        }
    } else if (warp < 2 + kTeamWarps) {
        // ---------------- feature team: 8 warps ----------------
        // Warp w reads TMEM lane quarter q = w % 4 (a hardware rule) and features [64 h, 64 h + 64)
        // of the projection; its lane is token row r of the tile.
        const int fw = warp - 2;
        const int q = warp & 3, h = fw >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const float A2 = p.scale * kLog2e;
        bool failed = false;
        int pu = 0;  // projections consumed
        const int fvalid = p.m - (feat0 + 64 * h);  // real (not padding) features among this warp's 64
        // phi of this warp's 64 projections in U, as 32 packed bf16 pairs, read in two halves of 32
        // columns (U is released once the second half is loaded). For exp features a row that must be
        // zero gets cst = +inf (ex2(-inf) = 0); the per-feature padding test is skipped when all 64
        // features are real (a warp-uniform branch).
        auto phi_from_u = [&](uint32_t (&w)[32], float cst, bool zero_row) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[32];
                tmem_ld32(tbase + lane_off + kColU + 64 * h + 32 * hh, v);
                tmem_ld_wait();
                if (hh == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_ufree);  // the next projection may overwrite U
                }
                if (exp_kind && fvalid >= 64) {
                    const float c = zero_row ? INFINITY : cst;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        float x0 = __uint_as_float(v[2 * k]), x1 = __uint_as_float(v[2 * k + 1]);
                        fma2(x0, x1, A2, -c);
                        w[16 * hh + k] = pack_bf16(ex2(x0), ex2(x1));
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        float x[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float a = __uint_as_float(v[2 * k + e]);
                            x[e] = exp_kind ? ex2(fmaf(a, A2, -cst)) : fmaxf(a * p.scale, 0.f) + p.relu_eps_s;
                            if (zero_row || 32 * hh + 2 * k + e >= fvalid) x[e] = 0.f;
                        }
                        w[16 * hh + k] = pack_bf16(x[0], x[1]);
                    }
                }
            }
            ++pu;
        };
        // row r of `dst` (K-major, atom region h)
        auto store_phi = [&](uint8_t* dst, const uint32_t (&w)[32]) {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4*>(dst + h * 16384 + sw128_offset(r, ch)) =
                    make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
        };
        for (int t = 0; t < T; ++t) {
            const int b = t & 1;
            const bool valid = t * kTile + r < p.n;
            // ---- phi(Q_t); the norms of row r first (Q and K of tile t stay in shared memory until
            // both projections of the tile are done)
            failed |= !mbar_wait(&bar_ufull, pu & 1, &abort_flag);
            failed |= !mbar_wait(&bar_qfull, t & 1, &abort_flag);
            failed |= !mbar_wait(&bar_kfull, t & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            float cq = 0.f, ck = 0.f;
            if (exp_kind) {
                const float qn2 = s2 * tile_row_sqnorm<64>(sQ, r);
                const float kn2 = s2 * tile_row_sqnorm<64>(sK, r);
                cq = W * sqrtf(qn2) * kLog2e;
                ck = (0.5f * kn2 + stab) * kLog2e;
            }
            uint32_t pq[32];
            phi_from_u(pq, cq, false);
            if (t > 0) {  // the MMAs of tile t-1 have read the phi buffers
                failed |= !mbar_wait(&bar_grp, (t - 1) & 1, &abort_flag);
                __syncwarp();
            }
            store_phi(sPQ, pq);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_phq);
            // ---- den share phi(q_r) . z_<t over this warp's features, with the bf16-rounded phi
            // (both waits come before this tile's phi(K) is published, so neither barrier can have
            // moved on by two phases)
            failed |= !mbar_wait(&bar_snap, t & 1, &abort_flag);
            failed |= !mbar_wait(&bar_dfree[b], ((t >> 1) & 1) ^ 1, &abort_flag);  // tile t-2's shares read
            __syncwarp();
            const float* zr = sZ + b * 128 + 64 * h;
            float den = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 o = *reinterpret_cast<const uint4*>(sPQ + h * 16384 + sw128_offset(r, c));
                const float4 za = *reinterpret_cast<const float4*>(zr + 8 * c);
                const float4 zb = *reinterpret_cast<const float4*>(zr + 8 * c + 4);
                den = fmaf(__uint_as_float(o.x << 16), za.x, den);
                den = fmaf(__uint_as_float(o.x & 0xFFFF0000u), za.y, den);
                den = fmaf(__uint_as_float(o.y << 16), za.z, den);
                den = fmaf(__uint_as_float(o.y & 0xFFFF0000u), za.w, den);
                den = fmaf(__uint_as_float(o.z << 16), zb.x, den);
                den = fmaf(__uint_as_float(o.z & 0xFFFF0000u), zb.y, den);
                den = fmaf(__uint_as_float(o.w << 16), zb.z, den);
                den = fmaf(__uint_as_float(o.w & 0xFFFF0000u), zb.w, den);
            }
            sDenF[(b * 2 + h) * 128 + r] = den;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_den[b]);
            // ---- phi(K_t)
            failed |= !mbar_wait(&bar_ufull, pu & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            phi_from_u(pq, ck, !valid);
            store_phi(sPK, pq);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_phk);
        }
        (void)failed;
    } else {
        // ---------------- output team: 8 warps ----------------
        // Warp w reads TMEM lane quarter q = w % 4 and half h of the columns: keys [64 h, 64 h + 64)
        // of the scores, state columns [32 h, 32 h + 32) (lane = feature), output columns
        // [32 h, 32 h + 32) (lane = token row).
        const int ow = warp - 2 - kTeamWarps;
        const int q = warp & 3, h = ow >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        constexpr int NO = 32 * kTeamWarps;  // named barrier 2: the output team
        bool failed = false;
        // the state before tile 0 is zero
        {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                *reinterpret_cast<uint4*>(sS + sw128_offset(r, 4 * h + c)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sSl + sw128_offset(r, 4 * h + c)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (h == 0) sZ[r] = 0.f;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_snap);
        }
        for (int t = 0; t < T; ++t) {
            const int b = t & 1;
            failed |= !mbar_wait(&bar_grp, t & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            // ---- snapshot of the state after this tile's update, for the next tile (lane = feature r);
            // first, as the next tile's inter MMA and denominator wait for it
            if (t + 1 < T) {
                const int b1 = (t + 1) & 1;
                uint32_t sv[32];
                tmem_ld32(tbase + lane_off + kColS + 32 * h, sv);
                uint32_t z0 = 0u, z1 = 0u;
                if (h == 0) tmem_ld2(tbase + lane_off + kColS + 64, z0, z1);
                tmem_ld_wait();
                (void)z1;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float x[8], l[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) x[k] = __uint_as_float(sv[8 * c + k]);
                    uint4 o;
                    o.x = pack_bf16(x[0], x[1]);
                    o.y = pack_bf16(x[2], x[3]);
                    o.z = pack_bf16(x[4], x[5]);
                    o.w = pack_bf16(x[6], x[7]);
                    const uint32_t hw[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        l[2 * k] = x[2 * k] - __uint_as_float(hw[k] << 16);
                        l[2 * k + 1] = x[2 * k + 1] - __uint_as_float(hw[k] & 0xFFFF0000u);
                    }
                    uint4 ol;
                    ol.x = pack_bf16(l[0], l[1]);
                    ol.y = pack_bf16(l[2], l[3]);
                    ol.z = pack_bf16(l[4], l[5]);
                    ol.w = pack_bf16(l[6], l[7]);
                    *reinterpret_cast<uint4*>(sS + sw128_offset(r, 4 * h + c)) = o;
                    *reinterpret_cast<uint4*>(sSl + sw128_offset(r, 4 * h + c)) = ol;
                }
                if (h == 0) sZ[b1 * 128 + r] = feat0 + r < p.m ? __uint_as_float(z0) : 0.f;
                tc_fence_before();
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_snap);
            }
            // ---- A~ = scores masked by j <= i, as bf16 hi + lo, in place: the 16 columns of keys
            // [16 s, 16 s + 16) become 8 columns of hi and 8 of lo
            // Whether a 16-key chunk is wholly below, wholly above or across the diagonal is the same
            // for the warp's 32 rows [32 q, 32 q + 32) unless the chunk meets them: warp-uniform branches.
            float dO = 0.f;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const int s = 4 * h + s4;
                const uint32_t ca = tbase + lane_off + kColSc + 16 * s;
                uint32_t w[16];
                if (16 * s > 32 * q + 31) {  // every key of the chunk is after every row: A~ = 0
#pragma unroll
                    for (int k = 0; k < 16; ++k) w[k] = 0u;
                } else {
                    const bool full = 16 * s + 15 <= 32 * q;  // every key at or before every row
                    uint32_t v[16];
                    tmem_ld16(ca, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 16; k += 2) {
                        const int j = 16 * s + k;
                        const float a0 = (full || j <= r) ? __uint_as_float(v[k]) : 0.f;
                        const float a1 = (full || j + 1 <= r) ? __uint_as_float(v[k + 1]) : 0.f;
                        dO += a0 + a1;
                        const uint32_t hw = pack_bf16(a0, a1);
                        w[k / 2] = hw;
                        w[8 + k / 2] = pack_bf16(a0 - __uint_as_float(hw << 16), a1 - __uint_as_float(hw & 0xFFFF0000u));
                    }
                }
                tmem_st16(ca, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_atil);
            sDenO[h * 128 + r] = dO;
            // ---- output of tile t: columns [32 h, 32 h + 32) of row r
            failed |= !mbar_wait(&bar_num, t & 1, &abort_flag);
            failed |= !mbar_wait(&bar_den[b], (t >> 1) & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            uint32_t nv[32];
            tmem_ld32(tbase + lane_off + kColNum + 64 * b + 32 * h, nv);
            tmem_ld_wait();
            named_bar(2, NO);  // both halves' score row sums are visible
            const float den = ((sDenF[(b * 2) * 128 + r] + sDenF[(b * 2 + 1) * 128 + r]) + sDenO[r]) + sDenO[128 + r];
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_dfree[b]);  // numerator buffer b and its den shares are free
            float dsum = den;
            const int owner = r / RP;
            const int i_tok = t * kTile + r;
            const bool valid = i_tok < p.n;
            if (CS > 1) {
                // Partial sums of row r go to the CTA that finalises it: slot [sender][row][kXStride
                // floats]; the odd number of 16-byte groups per row keeps a warp's float4 accesses
                // free of bank conflicts. Every output warp of this CTA is past its reads of the
                // previous tile's slots (named barrier above), so its buffer may be refilled.
                if (ow == 0 && lane == 0)
                    for (int c = 0; c < CS; ++c)
                        if (c != rank) mbar_arrive_cluster(mapa(smem_u32(&bar_xfree), c));
                if (owner != rank) {
                    failed |= !mbar_wait_cluster(&bar_xfree, t & 1, &abort_flag);
                    __syncwarp();
                    const int slot = rank < owner ? rank : rank - 1;
                    float* rowp = sX + ((size_t)slot * RP + (r - owner * RP)) * kXStride;
                    const uint32_t ca = mapa(smem_u32(rowp + 32 * h), owner);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_cluster_v4(ca + 16 * c, make_uint4(nv[4 * c], nv[4 * c + 1], nv[4 * c + 2], nv[4 * c + 3]));
                    if (h == 0) st_cluster_f32(mapa(smem_u32(rowp + 64), owner), den);
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa(smem_u32(&bar_xfull), owner));
                } else {
                    failed |= !mbar_wait_cluster(&bar_xfull, t & 1, &abort_flag);
                    __syncwarp();
                    // add the peers' contributions to this CTA's own, peers in rank order (a fixed
                    // order: the result is bitwise reproducible)
                    float dacc = den;
                    for (int slot = 0; slot < CS - 1; ++slot) {
                        const float* src = sX + ((size_t)slot * RP + (r - rank * RP)) * kXStride;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 x4 = *reinterpret_cast<const float4*>(src + 32 * h + i);
                            nv[i] = __float_as_uint(__uint_as_float(nv[i]) + x4.x);
                            nv[i + 1] = __float_as_uint(__uint_as_float(nv[i + 1]) + x4.y);
                            nv[i + 2] = __float_as_uint(__uint_as_float(nv[i + 2]) + x4.z);
                            nv[i + 3] = __float_as_uint(__uint_as_float(nv[i + 3]) + x4.w);
                        }
                        dacc += src[64];
                    }
                    dsum = dacc;
                }
            }
            if (valid && owner == rank) {
                const float inv = 1.f / dsum;
                uint4* dst = reinterpret_cast<uint4*>(p.Y + ((size_t)bh * p.n + i_tok) * kD + 32 * h);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
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
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
    cluster_sync();  // no CTA leaves while a peer may still write into its shared memory
}

}  // namespace tcc
}  // namespace favor
