// Tensor-core (tcgen05 + TMA + TMEM) causal FAVOR+ scan for wide heads (m > 256), bf16 in / fp32
// accumulate, d = 64: up to two 128-feature groups per CTA, one tile at a time.
//
// One CTA walks the 128-token tiles of one head in order. Per tile t (rows i, keys j of the tile):
//   num_i = phi(q_i) S_<t + sum_{j <= i} (phi(q_i) . phi(k_j)) v_j
//   den_i = phi(q_i) z_<t + sum_{j <= i}  phi(q_i) . phi(k_j)
//   y_i   = num_i / den_i;   then S_<t+1 = S_<t + Phi(K_t)^T V_t,  z_<t+1 = z_<t + Phi(K_t)^T 1.
// The prefix state is carried at every tile boundary (128 tokens); within a tile the keys are
// masked by j <= i, which for two 64-token chunks is exactly their chunked prefix-sum result.
//
// Features are processed in 128-feature groups g; a head's groups are split over the CTAs of a
// thread-block cluster (1, 2 or 4 CTAs, at most two groups each), which add their partial
// numerators and denominators through distributed shared memory once per tile. Per group:
//   U = Q_t Omega_g^T -> phi_g(Q) (tokens on TMEM lanes) -> shared memory (K-major);
//   U = K_t Omega_g^T -> phi_g(K) -> shared memory;
//   scores D_sc += phi_g(Q) phi_g(K)^T, inter D_num += phi_g(Q) S_g (the state as taken at the tile
//   start, split into hi + lo bf16 images so that it keeps about 16 significant bits), state S_g += phi_g(K)^T V_t and z_g += phi_g(K)^T 1 (MMA with a block
//   of ones), all on the tensor cores with fp32 accumulation in TMEM.
// After the groups: the masked scores A~ are split into two bf16 operands (hi + lo, about 16
// significant bits) for D_num += A~ V_t; den takes phi(q) . z_<t on the CUDA cores plus the fp32
// row sums of the masked scores.
//
// Stabilisers: a query row uses c_i = W |q^_i| (W = largest row norm of Omega; Cauchy-Schwarz bounds
// every w_r . q^_i by it), the same in every feature group; keys use one running per-head constant
// raised (with a rescale of S and z) when a tile's bound W |k^| - |k^|^2/2 exceeds it by more than
// kStabSlackHi. Both cancel in num / den; the common 1/sqrt(m) is dropped.
#pragma once

#include "tc.cuh"
#include "tc_noncausal.cuh"  // shared helpers: ex2, tile_row_sqnorm, slack constants

namespace favor {
namespace tccw {

using namespace favor::tc;
using tcnc::ex2;
using tcnc::kStabSlackHi;
using tcnc::kStabSlackLo;
using tcnc::tile_row_sqnorm;

constexpr int kTile = 128;
constexpr int kD = 64;                 // head dimension handled by this kernel
constexpr int kEpiWarps = 16;  // four column groups x four TMEM lane quarters
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTileBytes = kTile * kD * 2;  // 16 KB: one [128 x 64] bf16 tile
constexpr int kPhiBytes = kTile * 128 * 2;  // 32 KB: [128 tokens x 128 features] bf16, two K atoms
constexpr int kXStride = 84;                // floats per row of the cluster exchange buffer (64 + den + pad)

// TMEM columns
constexpr uint32_t kColS = 0;      // S_g at g * 80: 64 columns of S, 16 of z (all equal)
constexpr uint32_t kColU = 160;    // projection output, 128 columns
constexpr uint32_t kColSc = 288;   // scores, 128 columns
constexpr uint32_t kColNum = 416;  // numerator, 64 columns

struct CausalParams {
    int n;
    int m;
    int m_pad;   // features handled by one CTA, a multiple of 128 (at most 256)
    int kind;
    float relu_eps_s;
    float scale;
    __nv_bfloat16* Y;
};

struct CausalSmem {
    // Omega (m_pad x 64, K-major), Q, K and V tiles, phi(Q) / A~lo, phi(K) / A~hi, the state snapshot
    // as hi and lo bf16 images (m_pad x 64 each, MN-major), ones block (16 x 128 bf16, K-major), z
    // snapshot (m_pad fp32).
    static size_t bytes(int m_pad) {
        return 1024 + (size_t)m_pad * 128 + 3 * kTileBytes + 2 * kPhiBytes + 2 * (size_t)m_pad * 128 + 4096 +
               (size_t)m_pad * 4;
    }
};

__global__ void __launch_bounds__(kThreads, 1)
    causal_tc_wide(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
              const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mOm, CausalParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 by hand below
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int MP = p.m_pad;  // this CTA's features
    const int G = MP / 128;
    // A head's features are split over the CS CTAs of a cluster: CTA `rank` owns features
    // [rank * MP, (rank + 1) * MP). Partial numerators and denominators are summed across the
    // cluster once per tile; CTA `rank` finalises the rows [rank * RP, (rank + 1) * RP).
    const int CS = (int)cluster_size();
    const int rank = (int)cluster_rank();
    const int RP = kTile / CS;
    const int feat0 = rank * MP;
    uint8_t* sOm = smem;                          // G regions of 128 rows x 128 B
    uint8_t* sQ = sOm + (size_t)MP * 128;
    uint8_t* sK = sQ + kTileBytes;
    uint8_t* sV = sK + kTileBytes;
    uint8_t* sPQ = sV + kTileBytes;               // phi(Q): 2 K-atom regions of 128 rows x 128 B; later A~lo
    uint8_t* sPK = sPQ + kPhiBytes;               // phi(K); later A~hi
    uint8_t* sS = sPK + kPhiBytes;                // S snapshot hi: MP rows x 128 B (MN-major, d contiguous)
    uint8_t* sSl = sS + (size_t)MP * 128;         // S snapshot lo (S - hi, rounded)
    uint8_t* sOnes = sSl + (size_t)MP * 128;      // 2 K-atom regions of 16 rows x 128 B
    float* sZ = reinterpret_cast<float*>(sOnes + 4096);  // [MP] z snapshot
    __shared__ uint64_t bar_om, bar_qfull, bar_kfull, bar_qkempty, bar_vfull, bar_vempty;
    __shared__ uint64_t bar_snap, bar_ufull, bar_ufree, bar_phq, bar_phk, bar_grp, bar_atil, bar_num, bar_dfree;
    __shared__ uint64_t bar_xfree, bar_xfull;  // cluster exchange of the partial sums
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float red[2][kEpiWarps];
    __shared__ float sW[4];  // per-rank largest squared row norm of Omega
    __shared__ float sWred[kThreads / 32];
    __shared__ float sDen[4 * 128];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x / CS;
    const int T = (p.n + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_om, 1);
        mbar_init(&bar_qfull, 1);
        mbar_init(&bar_kfull, 1);
        mbar_init(&bar_qkempty, 1);
        mbar_init(&bar_vfull, 1);
        mbar_init(&bar_vempty, 1);
        mbar_init(&bar_snap, kEpiWarps);
        mbar_init(&bar_ufull, 1);
        mbar_init(&bar_ufree, kEpiWarps);
        mbar_init(&bar_phq, kEpiWarps);
        mbar_init(&bar_phk, kEpiWarps);
        mbar_init(&bar_grp, 1);
        mbar_init(&bar_atil, kEpiWarps);
        mbar_init(&bar_num, 1);
        mbar_init(&bar_dfree, kEpiWarps);
        mbar_init(&bar_xfree, CS > 1 ? CS - 1 : 1);
        mbar_init(&bar_xfull, CS > 1 ? (CS - 1) * (RP / 32) * 4 : 1);
        fence_mbar_init();
    }
    // ones block (K-major, every element 1.0): z_g = phi_g(K)^T 1 via the tensor cores
    for (int i = threadIdx.x; i < 4096 / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(sOnes)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
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
        mbar_arrive_expect_tx(&bar_om, (uint32_t)MP * 128);
        for (int r0 = 0; r0 < MP; r0 += 128) tma_load_2d(sOm + (size_t)r0 * 128, &mOm, &bar_om, 0, feat0 + r0);
    }
    bool om_ok = mbar_wait(&bar_om, 0, &abort_flag);
    {
        float w2 = 0.f;
        if (p.kind == kKindExp)
            for (int row = threadIdx.x; row < MP; row += blockDim.x)
                w2 = fmaxf(w2, tile_row_sqnorm<64>(sOm + (size_t)(row >> 7) * 16384, row & 127));
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
    float W_all = 0.f;
    for (int c = 0; c < CS; ++c) W_all = fmaxf(W_all, sW[c]);
    W_all = sqrtf(W_all);
    (void)om_ok;

    if (warp == 0) {
        // ---------------- TMA producer (lane 0) ----------------
        if (lane == 0) {
            tma_prefetch_desc(&mQ);
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mV);
            bool ok = true;
            for (int t = 0; t < T && ok; ++t) {
                // Q and K of tile t once tile t-1 is projected; V of tile t once tile t-1's intra MMA is done.
                if (!(ok = mbar_wait(&bar_qkempty, (t & 1) ^ 1, &abort_flag))) break;
                mbar_arrive_expect_tx(&bar_qfull, kTileBytes);
                tma_load_3d(sQ, &mQ, &bar_qfull, 0, t * kTile, bh);
                mbar_arrive_expect_tx(&bar_kfull, kTileBytes);
                tma_load_3d(sK, &mK, &bar_kfull, 0, t * kTile, bh);
                if (!(ok = mbar_wait(&bar_vempty, (t & 1) ^ 1, &abort_flag))) break;
                mbar_arrive_expect_tx(&bar_vfull, kTileBytes);
                tma_load_3d(sV, &mV, &bar_vfull, 0, t * kTile, bh);
            }
            // Drain the loads in flight before the CTA may exit.
            volatile int never = 0;
            if (T > 0) {
                mbar_wait(&bar_qfull, (T - 1) & 1, &never);
                mbar_wait(&bar_kfull, (T - 1) & 1, &never);
                mbar_wait(&bar_vfull, (T - 1) & 1, &never);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (lane 0) ----------------
        if (lane == 0) {
            constexpr uint32_t id_proj = idesc_bf16(128, 128, false, false);  // U = X Om_g^T
            constexpr uint32_t id_sc = idesc_bf16(128, 128, false, false);    // phi(Q) phi(K)^T
            constexpr uint32_t id_num = idesc_bf16(128, kD, false, true);     // phi(Q) S_g, A~ V
            constexpr uint32_t id_st = idesc_bf16(128, kD, true, true);       // phi(K)^T V
            constexpr uint32_t id_z = idesc_bf16(128, 16, true, false);       // phi(K)^T 1
            bool ok = mbar_wait(&bar_om, 0, &abort_flag);
            tc_fence_after();
            int uuse = 0;  // uses of the U slot so far
            auto proj = [&](const uint8_t* x, int g) {
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    uint64_t ad = sdesc_sw128(smem_u32(x + ks * 32), 16, 1024);
                    uint64_t bd = sdesc_sw128(smem_u32(sOm + (size_t)g * 16384 + ks * 32), 16, 1024);
                    mma_ss(tbase + kColU, ad, bd, id_proj, ks > 0);
                }
                mma_commit(&bar_ufull);
            };
            for (int t = 0; t < T && ok; ++t) {
                ok = ok && mbar_wait(&bar_qfull, t & 1, &abort_flag) && mbar_wait(&bar_kfull, t & 1, &abort_flag);
                ok = ok && mbar_wait(&bar_snap, t & 1, &abort_flag);
                ok = ok && mbar_wait(&bar_dfree, (t & 1) ^ 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint8_t* vt = sV;
                bool have_v = false;
                for (int g = 0; g < G && ok; ++g) {
                    // projections: Q then K into the one U slot
                    ok = mbar_wait(&bar_ufree, (uuse & 1) ^ 1, &abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    proj(sQ, g);
                    ++uuse;
                    ok = mbar_wait(&bar_ufree, (uuse & 1) ^ 1, &abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    proj(sK, g);
                    ++uuse;
                    if (g == G - 1) mma_commit(&bar_qkempty);
                    const int gu = t * G + g;  // group use count
                    ok = mbar_wait(&bar_phq, gu & 1, &abort_flag) && mbar_wait(&bar_phk, gu & 1, &abort_flag);
                    if (ok && !have_v) ok = have_v = mbar_wait(&bar_vfull, t & 1, &abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    // scores and inter numerator (K = 128 features of group g, two K atoms)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int a = ks / 4, w = ks % 4;
                        uint64_t ad = sdesc_sw128(smem_u32(sPQ + a * 16384 + w * 32), 16, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(sPK + a * 16384 + w * 32), 16, 1024);
                        mma_ss(tbase + kColSc, ad, bd, id_sc, (g > 0 || ks > 0));
                    }
                    for (int part = 0; part < 2; ++part) {  // state snapshot hi, then lo
                        const uint8_t* sp = part == 0 ? sS : sSl;
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const int a = ks / 4, w = ks % 4;
                            uint64_t ad = sdesc_sw128(smem_u32(sPQ + a * 16384 + w * 32), 16, 1024);
                            uint64_t bd = sdesc_sw128(smem_u32(sp + (size_t)(g * 128 + ks * 16) * 128), 16, 1024);
                            mma_ss(tbase + kColNum, ad, bd, id_num, (g > 0 || part > 0 || ks > 0));
                        }
                    }
                    // state update: S_g += phi_g(K)^T V_t, z_g += phi_g(K)^T 1 (K = 128 tokens)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        uint64_t ad = sdesc_sw128(smem_u32(sPK + ks * 2048), 16384, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(vt + ks * 2048), 16, 1024);
                        mma_ss(tbase + kColS + g * 80, ad, bd, id_st, (t > 0 || ks > 0));
                    }
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int a = ks / 4, w = ks % 4;
                        uint64_t ad = sdesc_sw128(smem_u32(sPK + ks * 2048), 16384, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(sOnes + a * 2048 + w * 32), 16, 1024);
                        mma_ss(tbase + kColS + g * 80 + 64, ad, bd, id_z, (t > 0 || ks > 0));
                    }
                    mma_commit(&bar_grp);
                }
                if (!ok) break;
                // intra-tile numerator: D_num += (A~hi + A~lo) V_t (hi in the phi(K) buffer, lo in the
                // phi(Q) buffer; K = 128 tokens)
                ok = mbar_wait(&bar_atil, t & 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                for (int part = 0; part < 2; ++part) {
                    const uint8_t* at = part == 0 ? sPK : sPQ;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int a = ks / 4, w = ks % 4;
                        uint64_t ad = sdesc_sw128(smem_u32(at + a * 16384 + w * 32), 16, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(vt + ks * 2048), 16, 1024);
                        mma_ss(tbase + kColNum, ad, bd, id_num, 1);
                    }
                }
                mma_commit(&bar_num);
                mma_commit(&bar_vempty);
            }
        }
    } else {
        // ---------------- epilogue: 16 warps ----------------
        // Warp ew = warp - 2 reads TMEM lane quarter q = warp % 4 (a hardware rule) and takes column
        // group cg = ew / 4 of every row it handles. Its lane is a token row for the projections,
        // the scores and the numerator, and a feature row for the state.
        constexpr int NT = 32 * kEpiWarps;
        const int ew = warp - 2;
        const int q = warp & 3, cg = ew >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const float A2 = p.scale * kLog2e;
        const bool exp_kind = p.kind == kKindExp;
        bool failed = !mbar_wait(&bar_om, 0, &abort_flag);
        __syncwarp();
        const float W = W_all;
        float stab = 0.f;
        int guse = 0;    // feature groups whose MMAs have been committed (bar_grp phases)
        int uuse_e = 0;  // projections consumed (bar_ufull phases)
        for (int t = 0; t < T; ++t) {
            const int i_tok = t * kTile + r;  // this thread's token (query row / key row)
            const bool valid = i_tok < p.n;
            failed |= !mbar_wait(&bar_qfull, t & 1, &abort_flag);
            failed |= !mbar_wait(&bar_kfull, t & 1, &abort_flag);
            __syncwarp();
            // norms of this row's query and key (each column group recomputes them: 64 elements)
            const float qn2 = exp_kind ? p.scale * p.scale * tile_row_sqnorm<64>(sQ, r) : 0.f;
            const float kn2 = exp_kind ? p.scale * p.scale * tile_row_sqnorm<64>(sK, r) : 0.f;
            const float cq = exp_kind ? W * sqrtf(qn2) * kLog2e : 0.f;
            float f = 1.f;
            if (exp_kind) {
                const float b = valid ? W * sqrtf(kn2) - 0.5f * kn2 : -INFINITY;
                const float bm = warp_max(b);
                if (lane == 0) red[t & 1][ew] = bm;
                named_bar(1, NT);
                float Bt = -INFINITY;
#pragma unroll
                for (int i = 0; i < kEpiWarps; ++i) Bt = fmaxf(Bt, red[t & 1][i]);
                if (t == 0) {
                    stab = Bt - kStabSlackLo;
                } else if (Bt > stab + kStabSlackHi) {
                    const float nst = Bt - kStabSlackLo;
                    f = ex2((stab - nst) * kLog2e);
                    stab = nst;
                }
            }
            const float ck = valid ? (exp_kind ? (0.5f * kn2 + stab) * kLog2e : 0.f) : INFINITY;
            // ---- state snapshot for this tile (lane = feature r of each group; 16 columns per warp) ----
            if (t > 0) {
                // every state MMA of the previous tile has completed once its last group committed
                failed |= !mbar_wait(&bar_grp, (guse - 1) & 1, &abort_flag);
                __syncwarp();
                tc_fence_after();
            }
            for (int g = 0; g < G; ++g) {
                const int feat = g * 128 + r;
                uint32_t v[16];
                const uint32_t sa = tbase + lane_off + kColS + g * 80;
                if (t > 0) {
                    tmem_ld16(sa + 16 * cg, v);
                    uint32_t zz[16];
                    if (cg == 0) tmem_ld16(sa + 64, zz);
                    tmem_ld_wait();
                    if (f != 1.f) {  // the key stabiliser moved: rescale the accumulated state
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tmem_st16(sa + 16 * cg, v);
                        if (cg == 0) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) zz[i] = __float_as_uint(__uint_as_float(zz[i]) * f);
                            tmem_st16(sa + 64, zz);
                        }
                        tmem_st_wait();
                    }
                    if (cg == 0) sZ[feat] = feat0 + feat < p.m ? __uint_as_float(zz[0]) : 0.f;
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0u;
                    if (cg == 0) sZ[feat] = 0.f;
                }
                // bf16 snapshot of S row `feat`, columns [16 cg, 16 cg + 16), as hi + lo
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float x[8], l[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) x[k] = __uint_as_float(v[8 * c + k]);
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
                    *reinterpret_cast<uint4*>(sS + sw128_offset(feat, 2 * cg + c)) = o;
                    *reinterpret_cast<uint4*>(sSl + sw128_offset(feat, 2 * cg + c)) = ol;
                }
            }
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_snap);
            named_bar(1, NT);  // z snapshot visible to every epilogue thread
            // ---- per feature group: phi(Q), phi(K) into shared memory (32 features per warp) ----
            float den = 0.f;  // this warp's share of the row's denominator
            for (int g = 0; g < G; ++g) {
                if (g > 0) {  // the previous group's MMAs have read the phi buffers
                    failed |= !mbar_wait(&bar_grp, (guse - 1) & 1, &abort_flag);
                    __syncwarp();
                }
                for (int which = 0; which < 2; ++which) {  // 0: queries, 1: keys
                    failed |= !mbar_wait(&bar_ufull, uuse_e & 1, &abort_flag);
                    __syncwarp();
                    tc_fence_after();
                    ++uuse_e;
                    uint32_t v[32];
                    tmem_ld32(tbase + lane_off + kColU + 32 * cg, v);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_ufree);  // U has been read: the next projection may overwrite it
                    uint8_t* dst = which == 0 ? sPQ : sPK;
                    const float cst = which == 0 ? cq : ck;
                    const bool zero_row = which == 1 && !valid;
                    const int f0 = g * 128 + 32 * cg;  // this CTA's feature index
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float ph[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float a = __uint_as_float(v[8 * c + k]);
                            float x = exp_kind ? ex2(fmaf(a, A2, -cst)) : fmaxf(a * p.scale, 0.f) + p.relu_eps_s;
                            if (zero_row || feat0 + f0 + 8 * c + k >= p.m) x = 0.f;
                            ph[k] = x;
                        }
                        uint4 o;
                        o.x = pack_bf16(ph[0], ph[1]);
                        o.y = pack_bf16(ph[2], ph[3]);
                        o.z = pack_bf16(ph[4], ph[5]);
                        o.w = pack_bf16(ph[6], ph[7]);
                        *reinterpret_cast<uint4*>(dst + (cg >> 1) * 16384 + sw128_offset(r, (cg & 1) * 4 + c)) = o;
                        if (which == 0) {  // den: phi(q) . z_<t with the bf16-rounded features
                            const float4 za = *reinterpret_cast<const float4*>(sZ + f0 + 8 * c);
                            const float4 zb = *reinterpret_cast<const float4*>(sZ + f0 + 8 * c + 4);
                            den = fmaf(__uint_as_float(o.x << 16), za.x, den);
                            den = fmaf(__uint_as_float(o.x & 0xFFFF0000u), za.y, den);
                            den = fmaf(__uint_as_float(o.y << 16), za.z, den);
                            den = fmaf(__uint_as_float(o.y & 0xFFFF0000u), za.w, den);
                            den = fmaf(__uint_as_float(o.z << 16), zb.x, den);
                            den = fmaf(__uint_as_float(o.z & 0xFFFF0000u), zb.y, den);
                            den = fmaf(__uint_as_float(o.w << 16), zb.z, den);
                            den = fmaf(__uint_as_float(o.w & 0xFFFF0000u), zb.w, den);
                        }
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(which == 0 ? &bar_phq : &bar_phk);
                }
                ++guse;
            }
            // ---- masked scores (keys [32 cg, 32 cg + 32) of row r) -> A~ hi (phi(K) buffer), lo (phi(Q) buffer) ----
            failed |= !mbar_wait(&bar_grp, (guse - 1) & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            {
                uint32_t v[32];
                tmem_ld32(tbase + lane_off + kColSc + 32 * cg, v);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float a[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        a[k] = (32 * cg + 8 * c + k <= r) ? __uint_as_float(v[8 * c + k]) : 0.f;
                        den += a[k];
                    }
                    // A~ = hi + lo, both bf16: the intra-tile weights keep about 16 significant bits.
                    uint4 o, ol;
                    o.x = pack_bf16(a[0], a[1]);
                    o.y = pack_bf16(a[2], a[3]);
                    o.z = pack_bf16(a[4], a[5]);
                    o.w = pack_bf16(a[6], a[7]);
                    ol.x = pack_bf16(a[0] - __uint_as_float(o.x << 16), a[1] - __uint_as_float(o.x & 0xFFFF0000u));
                    ol.y = pack_bf16(a[2] - __uint_as_float(o.y << 16), a[3] - __uint_as_float(o.y & 0xFFFF0000u));
                    ol.z = pack_bf16(a[4] - __uint_as_float(o.z << 16), a[5] - __uint_as_float(o.z & 0xFFFF0000u));
                    ol.w = pack_bf16(a[6] - __uint_as_float(o.w << 16), a[7] - __uint_as_float(o.w & 0xFFFF0000u));
                    const uint32_t off = (cg >> 1) * 16384 + sw128_offset(r, (cg & 1) * 4 + c);
                    *reinterpret_cast<uint4*>(sPK + off) = o;
                    *reinterpret_cast<uint4*>(sPQ + off) = ol;
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_atil);
            sDen[cg * 128 + r] = den;
            named_bar(1, NT);  // denominator shares visible
            const float den_row = ((sDen[r] + sDen[128 + r]) + sDen[256 + r]) + sDen[384 + r];
            // ---- y = num / den, output columns [16 cg, 16 cg + 16) ----
            failed |= !mbar_wait(&bar_num, t & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(tbase + lane_off + kColNum + 16 * cg, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_dfree);
            float num[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) num[i] = __uint_as_float(v[i]);
            float dsum = den_row;
            const int owner = r / RP;
            if (CS > 1) {
                // Partial sums of row r go to the CTA that finalises it, through its phi(Q) buffer
                // (idle once this tile's intra MMA is done): slot [sender][row][kXStride floats]; the odd
                // number of 16-byte groups per row keeps a warp's float4 accesses free of bank conflicts.
                if (ew == 0 && lane == 0)
                    for (int c = 0; c < CS; ++c)
                        if (c != rank) mbar_arrive_cluster(mapa(smem_u32(&bar_xfree), c));
                if (owner != rank) {
                    failed |= !mbar_wait_cluster(&bar_xfree, t & 1, &abort_flag);
                    __syncwarp();
                    const int slot = rank < owner ? rank : rank - 1;
                    float* dstp = reinterpret_cast<float*>(sPQ) + ((size_t)slot * RP + (r - owner * RP)) * kXStride + 16 * cg;
                    const uint32_t ca = mapa(smem_u32(dstp), owner);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_cluster_v4(ca + 16 * c, make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]));
                    if (cg == 0) st_cluster_f32(mapa(smem_u32(reinterpret_cast<float*>(sPQ) + ((size_t)slot * RP + (r - owner * RP)) * kXStride + 64), owner), den_row);
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa(smem_u32(&bar_xfull), owner));
                } else {
                    failed |= !mbar_wait_cluster(&bar_xfull, t & 1, &abort_flag);
                    __syncwarp();
                    // sum the cluster's contributions in rank order (deterministic)
                    float acc[16];
                    float dacc = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                    for (int c = 0; c < CS; ++c) {
                        if (c == rank) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[i] += num[i];
                            dacc += den_row;
                        } else {
                            const int slot = c < rank ? c : c - 1;
                            const float* src = reinterpret_cast<const float*>(sPQ) + ((size_t)slot * RP + (r - rank * RP)) * kXStride;
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[i] += src[16 * cg + i];
                            dacc += src[64];
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) num[i] = acc[i];
                    dsum = dacc;
                }
            }
            if (valid && owner == rank) {
                const float inv = 1.f / dsum;
                uint4* dst = reinterpret_cast<uint4*>(p.Y + ((size_t)bh * p.n + i_tok) * kD + 16 * cg);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint4 o;
                    o.x = pack_bf16(num[8 * c + 0] * inv, num[8 * c + 1] * inv);
                    o.y = pack_bf16(num[8 * c + 2] * inv, num[8 * c + 3] * inv);
                    o.z = pack_bf16(num[8 * c + 4] * inv, num[8 * c + 5] * inv);
                    o.w = pack_bf16(num[8 * c + 6] * inv, num[8 * c + 7] * inv);
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

}  // namespace tccw
}  // namespace favor
