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
//                 cores, num = phi(Q) S on the tensor cores, Y = num / den stored in whole sectors.
//
// Stabilisers. A query row may use any constant of its own and a head's keys any one constant:
// both cancel between numerator and denominator. Queries use their exact row maximum. Keys use a
// running constant per CTA that follows the exact largest key exponent of the tiles already
// reduced (known two tiles late), and is never less than the bound
// u_r(k) <= W |k^| - |k^|^2 / 2 (Cauchy-Schwarz, W = largest row norm of Omega) of the current
// tile minus kStabGuard, so that no feature can overflow before its tile's maximum is known; each
// move rescales the accumulated S and z. The common factor 1/sqrt(m) is dropped on both sides for
// the same reason.
#pragma once

#include "tc.cuh"

namespace favor {
namespace tcnc {

using namespace favor::tc;

constexpr int kTile = 128;            // tokens per tile (the MMA M or N extent)
constexpr int kEpiWarps = 16;         // four column groups x four TMEM lane quarters
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;  // warp 0: TMA, warp 1: MMA, then the epilogue warps
constexpr float kStabSlackHi = 24.f;  // the key constant is raised once a key exponent exceeds it by this much
constexpr float kStabGuard = 60.f;    // ... and never lies further than this below the current tile's bound
constexpr float kStabSlackDown = 40.f;  // ... lowered once the keys seen so far all lie this far below it
constexpr float kStabStepDown = 20.f;   // ... by at most this much per tile

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// TMEM column of the packed phi^T for state-MMA K step ks (16 tokens): each epilogue warp packs its
// 64 tokens into the first 32 columns of its own 64-column range.
__host__ __device__ constexpr uint32_t phi_col(int ks) { return 64u * (uint32_t)(ks / 4) + 8u * (uint32_t)(ks % 4); }

// a0 += lo^2, a1 += hi^2 for the two bf16 values of w, with one packed fp32x2 FMA.
__device__ __forceinline__ void sq_acc_bf16x2(uint32_t w, float& a0, float& a1) {
    asm("{\n\t.reg .b64 x, acc;\n\t.reg .b32 lo, hi;\n\t"
        "shl.b32 lo, %2, 16;\n\tand.b32 hi, %2, 0xffff0000;\n\t"
        "mov.b64 x, {lo, hi};\n\tmov.b64 acc, {%0, %1};\n\t"
        "fma.rn.f32x2 acc, x, x, acc;\n\t"
        "mov.b64 {%0, %1}, acc;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w));
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
            for (int i = 0; i < 4; ++i) sq_acc_bf16x2(w[i], s0, s1);
        }
    }
    return s0 + s1;
}

// =============================================================================================
// Key-side state kernel
// =============================================================================================
struct StateParams {
    int n;              // tokens per head
    int m;              // features
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
    // K tile t is needed by the first projection of tile t and V tile t by the first state MMA of
    // tile t, which comes three MMA groups later; a K tile is refilled after its tile's last
    // projection, a V tile after its tile's last state MMA. The K ring is the deeper one so that
    // a refill has about as many MMA groups of lead time as the V refill.
    static constexpr int kKStages = (D == 64) ? 5 : 3;
    static constexpr int kVStages = (D == 64) ? 5 : 2;
    static constexpr int kTileBytes = kTile * D * 2;  // one [128 x D] bf16 tile
    // Omega region: D/64 swizzled regions of (groups * 128) rows, each row 128 B.
    __host__ __device__ static size_t omega_bytes(int groups) { return (size_t)groups * 128 * D * 2; }
    static size_t bytes(int groups) {
        return 1024 + omega_bytes(groups) + (size_t)(kKStages + kVStages) * kTileBytes + 2 * 128 * 4 /*sC*/ + 64;
    }
};

// Key-side kernel roles: warp 0 TMA (lane 0 K tiles, lane 1 V tiles), warp 1 MMA issue, warps 2-3
// norms and the key stabiliser, warps 4.. two epilogue teams of 8 warps. A unit is one 128-token
// tile for one 128-feature group; unit u = tile * groups + group sits in TMEM slot u % 2 and is
// handled by team u % 2.
constexpr int kStateUnitTok = 128;
constexpr int kStateSlots = 2;
constexpr int kStateTeamWarps = 8;
constexpr int kStateEpiWarps = 2 * kStateTeamWarps;
constexpr int kStateNormWarps = 2;
constexpr int kStateEpiWarp0 = 2 + kStateNormWarps;
constexpr int kStateThreads = 32 * (kStateEpiWarp0 + kStateEpiWarps);

template <int D, int KIND>
__global__ void __launch_bounds__(kStateThreads, 1)
    nc_state_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                const __grid_constant__ CUtensorMap mOm, StateParams p) {
    using SM = StateSmem<D>;
    constexpr int NK = SM::kKStages, NV = SM::kVStages;
    constexpr int kAtoms = D / 64;
    extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 by hand below
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int G = p.groups;
    uint8_t* sOm = smem;                                   // kAtoms regions of G*128 rows
    uint8_t* sK = sOm + SM::omega_bytes(G);                // NK K tiles
    uint8_t* sV = sK + (size_t)NK * SM::kTileBytes;        // NV V tiles
    float* sC = reinterpret_cast<float*>(sV + (size_t)NV * SM::kTileBytes);  // [2][128] per-token constants
    __shared__ uint64_t bar_kfull[NK], bar_kempty[NK], bar_vfull[NV], bar_vempty[NV], bar_om;
    __shared__ uint64_t bar_ufull[kStateSlots], bar_ufree[kStateSlots], bar_phi[kStateSlots];
    __shared__ uint64_t bar_nfull[2], bar_nempty[2];
    // bar_rs: one completion per tile whose stabiliser moved, once every state MMA of the tiles
    // before it has completed; bar_sdone: once, after the last state MMA. Every epilogue warp waits
    // on every completion of both, so no wait can mistake an old phase for the one it wants (a wait
    // on a slot barrier could: a team that does not use a slot may be two of its phases behind).
    __shared__ uint64_t bar_rs, bar_sdone;
    __shared__ float sF[2];  // per-tile rescale factor of the accumulated state (1 = none)
    __shared__ float sStabT[2];                       // the key stabiliser of tile t (slot t & 1), nats
    __shared__ float sUnitMax[4][kStateEpiWarps];     // per epilogue warp: exact largest key exponent of tile t (slot t & 3)
    __shared__ float sRed[2][kStateNormWarps];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int split = blockIdx.x, splits = gridDim.x;
    const int bh = blockIdx.y;
    const int fslice = blockIdx.z, fslices = gridDim.z;
    const int f0 = fslice * G * 128;  // first feature of this CTA
    const int j0 = split * p.tokens_per_split;
    const int j1 = min(p.n, j0 + p.tokens_per_split);
    const int T = (j1 - j0 + kTile - 1) / kTile;
    const int UPT = G;        // units per tile
    const int U = T * UPT;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < NK; ++i) {
            mbar_init(&bar_kfull[i], 1);
            mbar_init(&bar_kempty[i], 1 + kStateNormWarps);  // MMA commit after the tile's last projection + norm warps
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&bar_vfull[i], 1);
            mbar_init(&bar_vempty[i], 1);
        }
        mbar_init(&bar_om, 1);
        for (int i = 0; i < kStateSlots; ++i) {
            mbar_init(&bar_ufull[i], 1);
            mbar_init(&bar_ufree[i], 1);
            mbar_init(&bar_phi[i], kStateTeamWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_nfull[i], kStateNormWarps);
            mbar_init(&bar_nempty[i], kStateEpiWarps);
            if (i == 0) {
                mbar_init(&bar_rs, 1);
                mbar_init(&bar_sdone, 1);
            }
        }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) griddep_launch();  // the combine may be scheduled now; it waits for this grid
    const uint32_t tbase = tmem_base;
    // TMEM: S_g at columns [g*D, (g+1)*D); two 128-column U slots from column 256.
    auto u_col = [](int s) { return 256u + 128u * (uint32_t)s; };

    if (warp == 0) {
        // ---------------- TMA producers: lane 0 streams K tiles, lane 1 V tiles ----------------
        if (lane == 0) {
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mOm);
            mbar_arrive_expect_tx(&bar_om, (uint32_t)SM::omega_bytes(G));
            for (int g = 0; g < G; ++g)
                for (int a = 0; a < kAtoms; ++a)
                    tma_load_2d(sOm + (size_t)a * G * 16384 + g * 16384, &mOm, &bar_om, a * 64, f0 + g * 128);
        } else if (lane == 1) {
            tma_prefetch_desc(&mV);
        }
        if (lane < 2) {
            const int NR = lane == 0 ? NK : NV;
            uint64_t* full = lane == 0 ? bar_kfull : bar_vfull;
            uint64_t* empty = lane == 0 ? bar_kempty : bar_vempty;
            uint8_t* ring = lane == 0 ? sK : sV;
            const CUtensorMap* map = lane == 0 ? &mK : &mV;
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int st = t % NR;
                if (!mbar_wait(&empty[st], ((t / NR) & 1) ^ 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&full[st], SM::kTileBytes);
                for (int a = 0; a < kAtoms; ++a)
                    tma_load_3d(ring + (size_t)st * SM::kTileBytes + a * 16384, map, &full[st], a * 64, j0 + t * kTile, bh);
                issued = t + 1;
            }
            // Drain: every issued load must land before the CTA may exit.
            for (int t = max(0, issued - NR); t < issued; ++t) {
                volatile int never = 0;
                mbar_wait(&full[t % NR], (t / NR) & 1, &never);
            }
            if (lane == 0) {
                volatile int never = 0;
                mbar_wait(&bar_om, 0, &never);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_p = idesc_bf16(128, kStateUnitTok, false, false);  // U^T = Om_g K_half^T
            constexpr uint32_t idesc_s = idesc_bf16(128, D, false, true);               // S_g += phi^T V_half
            bool ok = mbar_wait(&bar_om, 0, &abort_flag);
            tc_fence_after();
            // unit u: tile u / G, group u % G, slot u % 2
            auto issue_proj = [&](int u) -> bool {
                const int t = u / UPT, g = u % UPT, s = u % kStateSlots, st = t % NK;
                if (u % UPT == 0 && !mbar_wait(&bar_kfull[st], (t / NK) & 1, &abort_flag)) return false;
                if (!mbar_wait(&bar_ufree[s], ((u / kStateSlots) & 1) ^ 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* kt = sK + (size_t)st * SM::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int a = ks / 4, w = ks % 4;
                    uint64_t ad = sdesc_sw128(smem_u32(sOm + (size_t)a * G * 16384 + g * 16384 + w * 32), 16, 1024);
                    uint64_t bd = sdesc_sw128(smem_u32(kt + a * 16384 + w * 32), 16, 1024);
                    mma_ss(tbase + u_col(s), ad, bd, idesc_p, ks > 0);
                }
                mma_commit(&bar_ufull[s]);
                if (u % UPT == UPT - 1) mma_commit(&bar_kempty[st]);
                return true;
            };
            auto issue_state = [&](int u) -> bool {
                const int t = u / UPT, g = u % UPT, s = u % kStateSlots, st = t % NV;
                if (u % UPT == 0 && !mbar_wait(&bar_vfull[st], (t / NV) & 1, &abort_flag)) return false;
                if (!mbar_wait(&bar_phi[s], (u / kStateSlots) & 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* vt = sV + (size_t)st * SM::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < kStateUnitTok / 16; ++ks) {
                    uint64_t bd = sdesc_sw128(smem_u32(vt + ks * 2048), 16384, 1024);
                    mma_ts(tbase + (uint32_t)(g * D), tbase + u_col(s) + phi_col(ks), bd, idesc_s, (t > 0 || ks > 0));
                }
                mma_commit(&bar_ufree[s]);
                if (u % UPT == UPT - 1) {
                    mma_commit(&bar_vempty[st]);
                    // the next tile's rescale factor (the norm warps publish it with bar_nfull); if the
                    // stabiliser moved, signal the epilogue once this tile's state MMAs have completed
                    const int tn = t + 1;
                    if (tn < T) {
                        if (!mbar_wait(&bar_nfull[tn & 1], (tn >> 1) & 1, &abort_flag)) return false;
                        if (sF[tn & 1] != 1.f) mma_commit(&bar_rs);
                    }
                }
                return true;
            };
            // Order P(0), P(1), S(0), P(2), S(1), ...: the projection into a slot waits for the state
            // MMA that last read it, which was issued one step earlier.
            if (ok) {
                for (int u = 0; u < U; ++u) {
                    if (!issue_proj(u)) break;
                    if (u >= 1 && !issue_state(u - 1)) break;
                }
                if (!abort_flag && U > 0) issue_state(U - 1);
            }
            mma_commit(&bar_sdone);  // every state MMA issued has completed
        }
    } else if (warp < kStateEpiWarp0) {
        // ---------------- norms and the key stabiliser (two warps) ----------------
        // Norm warp nw owns tokens [64 nw, 64 nw + 64) of every tile, two per lane. Per tile:
        // sC[t & 1][j] = (|k^_j|^2 / 2 + stab) log2 e (+inf for tokens outside the split) and
        // sF[t & 1] = the factor by which the state accumulated so far must be rescaled before this
        // tile (1 when the stabiliser did not move). Both warps run the same stabiliser logic.
        const int nw = warp - 2;
        const int nt = 32 * kStateNormWarps;
        bool ok = mbar_wait(&bar_om, 0, &abort_flag);
        float W = 0.f;
        if (KIND == kKindExp) {
            float w2 = 0.f;
            for (int row = nw * 32 + lane; row < G * 128; row += nt) {
                const int g = row >> 7, rr = row & 127;
                float s2 = 0.f;
                for (int a = 0; a < kAtoms; ++a) s2 += tile_row_sqnorm<64>(sOm + (size_t)a * G * 16384 + g * 16384, rr);
                w2 = fmaxf(w2, s2);
            }
            w2 = warp_max(w2);
            if (lane == 0) sRed[1][nw] = w2;
            named_bar(2, nt);
            float m2 = 0.f;
#pragma unroll
            for (int i = 0; i < kStateNormWarps; ++i) m2 = fmaxf(m2, sRed[1][i]);
            W = sqrtf(m2);
        }
        float stab = 0.f, run = -INFINITY;  // run: exact largest key exponent of the tiles reported so far
        for (int t = 0; t < T; ++t) {
            const int st = t % NK, b2 = t & 1;
            ok &= mbar_wait(&bar_nempty[b2], ((t >> 1) & 1) ^ 1, &abort_flag);
            ok &= mbar_wait(&bar_kfull[st], (t / NK) & 1, &abort_flag);
            __syncwarp();
            const uint8_t* kt = sK + (size_t)st * SM::kTileBytes;
            float h2[2], bmax = -INFINITY;
            bool v2[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int tok = nw * 64 + lane + 32 * i;
                v2[i] = j0 + t * kTile + tok < j1;
                const float xn2 = KIND == kKindExp ? p.scale * p.scale * tile_row_sqnorm<D>(kt, tok) : 0.f;
                h2[i] = 0.5f * xn2;
                if (v2[i]) bmax = fmaxf(bmax, W * sqrtf(xn2) - h2[i]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_kempty[st]);
            float f = 1.f;
            if (KIND == kKindExp) {
                const float wm = warp_max(bmax);
                if (lane == 0) sRed[b2][nw] = wm;
                named_bar(2, nt);
                float Bt = -INFINITY;
#pragma unroll
                for (int i = 0; i < kStateNormWarps; ++i) Bt = fmaxf(Bt, sRed[b2][i]);
                // The constant follows the exact largest key exponent of the tiles seen so far (from
                // the epilogue, two tiles behind): raised to it once it is exceeded by kStabSlackHi,
                // lowered towards it by at most kStabStepDown per tile once it lies kStabSlackDown
                // below (the unreported tile t-1 sits below e^kStabGuard before that step, so it
                // stays finite after it). The bound keeps every feature of tile t below
                // e^kStabGuard at all times.
                if (t >= 2) {
#pragma unroll
                    for (int i = 0; i < kStateEpiWarps; ++i) run = fmaxf(run, sUnitMax[(t - 2) & 3][i]);
                }
                const float guard = Bt - kStabGuard;
                float nst = stab;
                if (t == 0) {
                    nst = guard;
                } else {
                    if (run > nst + kStabSlackHi) nst = run;
                    else if (run > -INFINITY && run < nst - kStabSlackDown) nst = fmaxf(run, nst - kStabStepDown);
                    if (guard > nst) nst = guard;
                    if (nst != stab) f = ex2((stab - nst) * kLog2e);
                }
                stab = nst;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
                sC[b2 * 128 + nw * 64 + lane + 32 * i] =
                    v2[i] ? (KIND == kKindExp ? (h2[i] + stab) * kLog2e : 0.f) : INFINITY;
            if (nw == 0 && lane == 0) {
                sF[b2] = f;
                sStabT[b2] = stab;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_nfull[b2]);
        }
        if (nw == 0 && lane == 0)
            p.pstab[((size_t)bh * splits + split) * fslices + fslice] = (KIND == kKindExp && ok) ? stab : 0.f;
    } else {
        // ---------------- epilogue: two teams of 8 warps ----------------
        // Team tm handles the units u = tm (mod 2). Within a team, warp (cg, q) reads TMEM lane
        // quarter q = warp % 4 (a hardware rule) and the 32 tokens [32 cg, 32 cg + 32) of the unit.
        const int ew = warp - kStateEpiWarp0;
        const int tm = ew / kStateTeamWarps, cg = (ew % kStateTeamWarps) >> 2, q = warp & 3;
        const int r = q * 32 + lane;  // feature lane within a group
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const float A2 = p.scale * kLog2e;
        float zacc[4] = {0.f, 0.f, 0.f, 0.f};
        bool failed = false;
        int nrs = 0;  // rescale events waited for (bar_rs completions)
        for (int t = 0; t < T; ++t) {
            const int b2 = t & 1;
            failed |= !mbar_wait(&bar_nfull[b2], (t >> 1) & 1, &abort_flag);
            __syncwarp();
            const float f = sF[b2];
            if (f != 1.f) {
                // The key stabiliser moved: once every state MMA so far has completed, scale S and z.
                failed |= !mbar_wait(&bar_rs, nrs & 1, &abort_flag);
                ++nrs;
                __syncwarp();
                tc_fence_after();
                const int part = tm * 2 + cg;  // this warp's quarter of the S columns
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if (g >= G) break;
                    constexpr int kC = D / 4;
                    const uint32_t sa = tbase + lane_off + g * D + part * kC;
                    if constexpr (kC == 32) {
                        uint32_t v[32];
                        tmem_ld32(sa, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tmem_st32(sa, v);
                    } else {
                        uint32_t v[16];
                        tmem_ld16(sa, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tmem_st16(sa, v);
                    }
                    zacc[g] *= f;
                }
                tmem_st_wait();
                tc_fence_before();
                named_bar(1, 32 * kStateEpiWarps);  // both teams' parts are rescaled before any phi of tile t
            }
            const float* cj = sC + b2 * 128 + 64 * cg;
            const float stab_t = sStabT[b2];
            float umax = -INFINITY;  // exact largest key exponent of the units this warp handles (log2, relative)
            for (int g = 0; g < G; ++g) {
                const int u = t * UPT + g;
                if ((u & 1) != tm) continue;
                const bool real_feat = f0 + g * 128 + r < p.m;
                float umu = -INFINITY;  // the unit's largest exponent (counted for real features only)
                const int s = u % kStateSlots;
                failed |= !mbar_wait(&bar_ufull[s], (u / kStateSlots) & 1, &abort_flag);
                __syncwarp();
                tc_fence_after();
                const uint32_t ua = tbase + lane_off + u_col(s) + 64 * cg;
                float zs0 = 0.f, zs1 = 0.f;
                // Two halves of 32 tokens: load, map, pack, store. The packed phi of half hh goes to
                // columns [16 hh, 16 hh + 16) of this warp's own 64, which the loads of half 0 have
                // already consumed: no other warp reads them.
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t vv[32];
                    tmem_ld32(ua + 32 * hh, vv);
                    tmem_ld_wait();
                    const float* cc = cj + 32 * hh;
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 c4 = *reinterpret_cast<const float4*>(cc + i);
                        float f[4];
                        if (KIND == kKindExp) {
                            const float e0 = fmaf(__uint_as_float(vv[i + 0]), A2, -c4.x);
                            const float e1 = fmaf(__uint_as_float(vv[i + 1]), A2, -c4.y);
                            const float e2 = fmaf(__uint_as_float(vv[i + 2]), A2, -c4.z);
                            const float e3 = fmaf(__uint_as_float(vv[i + 3]), A2, -c4.w);
                            f[0] = ex2(e0);
                            f[1] = ex2(e1);
                            f[2] = ex2(e2);
                            f[3] = ex2(e3);
                            umu = fmaxf(umu, fmaxf(fmaxf(e0, e1), fmaxf(e2, e3)));
                        } else {
                            f[0] = c4.x == 0.f ? phi_plain(__uint_as_float(vv[i + 0]) * p.scale, KIND, 1.f, p.relu_eps_s) : 0.f;
                            f[1] = c4.y == 0.f ? phi_plain(__uint_as_float(vv[i + 1]) * p.scale, KIND, 1.f, p.relu_eps_s) : 0.f;
                            f[2] = c4.z == 0.f ? phi_plain(__uint_as_float(vv[i + 2]) * p.scale, KIND, 1.f, p.relu_eps_s) : 0.f;
                            f[3] = c4.w == 0.f ? phi_plain(__uint_as_float(vv[i + 3]) * p.scale, KIND, 1.f, p.relu_eps_s) : 0.f;
                        }
                        pk[i / 2] = pack_bf16(f[0], f[1]);
                        pk[i / 2 + 1] = pack_bf16(f[2], f[3]);
                        zs0 += f[0] + f[2];
                        zs1 += f[1] + f[3];
                    }
                    tmem_st16(ua + 16 * hh, pk);
                }
                if (g == 0) zacc[0] += zs0 + zs1;
                else if (g == 1) zacc[1] += zs0 + zs1;
                else if (g == 2) zacc[2] += zs0 + zs1;
                else zacc[3] += zs0 + zs1;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_phi[s]);
                if (real_feat) umax = fmaxf(umax, umu);
            }
            if (KIND == kKindExp) {  // for the key constant two tiles on (nats, absolute)
                umax = warp_max(umax);
                if (lane == 0) sUnitMax[t & 3][ew] = umax == -INFINITY ? -INFINITY : umax / kLog2e + stab_t;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_nempty[b2]);
        }
        // Final state: wait for the last state MMA, then write this CTA's partial S and z.
        const bool done = __all_sync(0xffffffffu, U > 0 && mbar_wait(&bar_sdone, 0, &abort_flag));
        tc_fence_after();
        const size_t part_idx = (size_t)bh * splits + split;
        // z partials of the two teams and two column groups meet in shared memory (the V ring is idle now).
        float* sZ = reinterpret_cast<float*>(sV);
        const int zpart = tm * 2 + cg;
#pragma unroll
        for (int g = 0; g < 4; ++g)
            if (g < G) sZ[(zpart * 4 + g) * 128 + r] = zacc[g];
        named_bar(1, 32 * kStateEpiWarps);
        if (__all_sync(0xffffffffu, done && !failed)) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                if (g >= G) break;
                const int feat = f0 + g * 128 + r;
                constexpr int kC = D / 4;
                float* out = p.pS + (part_idx * p.m_pad + feat) * D + zpart * kC;
                const uint32_t sa = tbase + lane_off + g * D + zpart * kC;
                if constexpr (kC == 32) {
                    uint32_t v[32];
                    tmem_ld32(sa, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(out + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                                          __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                } else {
                    uint32_t v[16];
                    tmem_ld16(sa, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4*>(out + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                                          __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                }
                if (zpart == 0)
                    p.pz[part_idx * p.m_pad + feat] =
                        ((sZ[(0 * 4 + g) * 128 + r] + sZ[(1 * 4 + g) * 128 + r]) + sZ[(2 * 4 + g) * 128 + r]) +
                        sZ[(3 * 4 + g) * 128 + r];
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
    __shared__ float red[4];
    griddep_launch();  // the readout may start its prologue; it waits for this grid before reading S
    griddep_wait();    // the key-side partial states are complete
    const int bh = blockIdx.y;
    const int nst = splits * fslices;
    const float* st = pstab + (size_t)bh * nst;
    // stabilisers: loaded in parallel, reduced, turned into weights exp(stab_s - max)
    float M = -INFINITY;
    for (int i = threadIdx.x; i < nst; i += blockDim.x) {
        wts[i] = st[i];
        M = fmaxf(M, wts[i]);
    }
    M = warp_max(M);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    for (int i = threadIdx.x; i < nst; i += blockDim.x) wts[i] = ex2((wts[i] - M) * kLog2e);
    __syncthreads();
    const int rows_per_block = 128 / kChunks;  // D=64: 16 rows, D=128: 8 rows
    const int row = blockIdx.x * rows_per_block + threadIdx.x / kChunks;
    const int ch = threadIdx.x % kChunks;
    if (row >= m_pad) return;
    const int fs = row / feats_per_slice;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float zs = 0.f;
    // Splits in a fixed order, eight at a time with their loads issued together.
    for (int s0 = 0; s0 < splits; s0 += 8) {
        float4 a[8], b[8];
        float zp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (s0 + k < splits) {
                const float* src = pS + (((size_t)bh * splits + s0 + k) * m_pad + row) * D + ch * 8;
                a[k] = *reinterpret_cast<const float4*>(src);
                b[k] = *reinterpret_cast<const float4*>(src + 4);
                zp[k] = ch == 0 ? pz[((size_t)bh * splits + s0 + k) * m_pad + row] : 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (s0 + k < splits) {
                const float w = wts[(s0 + k) * fslices + fs];
                acc[0] = fmaf(w, a[k].x, acc[0]); acc[1] = fmaf(w, a[k].y, acc[1]);
                acc[2] = fmaf(w, a[k].z, acc[2]); acc[3] = fmaf(w, a[k].w, acc[3]);
                acc[4] = fmaf(w, b[k].x, acc[4]); acc[5] = fmaf(w, b[k].y, acc[5]);
                acc[6] = fmaf(w, b[k].z, acc[6]); acc[7] = fmaf(w, b[k].w, acc[7]);
                zs = fmaf(w, zp[k], zs);
            }
        }
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
    if (!FAVOR_IN_BOUNDS(bh < (int)gridDim.y && row < m_pad && a < D / 64)) return;
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
    __nv_bfloat16* Y;     // [BH][n][D] output
};

template <int D>
struct ReadoutSmem {
    static constexpr int kStages = (D == 64) ? 4 : 2;
    static constexpr int kTileBytes = kTile * D * 2;
    static size_t bytes(int m_pad) {
        return 1024 + (size_t)m_pad * D * 2 /*Omega*/ + (size_t)m_pad * D * 2 /*S image*/ + (size_t)m_pad * 4 /*z*/ +
               (size_t)kStages * kTileBytes + 2 * 2 * 4 * 128 * 4 /*max, den partials*/;
    }
};

template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    nc_readout_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mOm, ReadoutParams p) {
    using SM = ReadoutSmem<D>;
    constexpr int NS = SM::kStages;
    constexpr int kAtoms = D / 64;
    extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 by hand below
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int MP = p.m_pad;
    uint8_t* sOm = smem;                                   // kAtoms regions of MP rows x 128 B
    uint8_t* sS = sOm + (size_t)MP * D * 2;                // S image: kAtoms regions of MP rows x 128 B
    uint8_t* sQ = sS + (size_t)MP * D * 2;                 // NS stages
    float* sz = reinterpret_cast<float*>(sQ + (size_t)NS * SM::kTileBytes);  // [MP]
    float* sMax = sz + MP;                                 // [2][4][128] row-max partials
    float* sDen = sMax + 2 * 4 * 128;                      // [2][4][128] denominator partials
    __shared__ uint64_t bar_full[NS], bar_empty[NS], bar_const, bar_sz, bar_ufull[2], bar_ufree[2], bar_phi[2], bar_num[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y;
    const int tiles_head = (p.n + kTile - 1) / kTile;
    const int t0 = blockIdx.x * p.tiles_per_cta;
    const int T = max(0, min(tiles_head, t0 + p.tiles_per_cta) - t0);
    // Two TMEM slots of 256 columns when m_pad <= 256, else one slot of 512.
    const bool two = MP <= 256;
    const int nslot = two ? 2 : 1;
    const uint32_t slot_cols = two ? 256u : 512u;
    const int Wf = MP / 4;  // features per column group of epilogue warps
    // Packed phi: compact [0, MP/2) when m_pad <= 256 (all U values are in registers before any
    // warp overwrites U); otherwise each warp packs into the first half of its own column range.
    auto phi_col_r = [&](int ks) -> uint32_t {
        if (two) return (uint32_t)ks * 8u;
        const int f = ks * 16;
        return (uint32_t)((f / Wf) * Wf + (f % Wf) / 2);
    };
    const uint32_t num_off = two ? 128u : (MP < 512 ? (uint32_t)MP : 64u);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_const, 1);
        mbar_init(&bar_sz, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_ufull[i], 1);
            mbar_init(&bar_ufree[i], kEpiWarps);
            mbar_init(&bar_phi[i], kEpiWarps);
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
            const uint32_t sbytes = (uint32_t)MP * D * 2;
            mbar_arrive_expect_tx(&bar_const, sbytes);
            for (int a = 0; a < kAtoms; ++a)
                for (int r0 = 0; r0 < MP; r0 += 128)
                    tma_load_2d(sOm + (size_t)a * MP * 128 + r0 * 128, &mOm, &bar_const, a * 64, r0);
            // The first query tiles do not depend on the preceding kernels: load them before waiting.
            int issued = 0;
            for (int t = 0; t < min(T, NS); ++t) {
                mbar_arrive_expect_tx(&bar_full[t], SM::kTileBytes);
                for (int a = 0; a < kAtoms; ++a)
                    tma_load_3d(sQ + (size_t)t * SM::kTileBytes + a * 16384, &mQ, &bar_full[t], a * 64,
                                (t0 + t) * kTile, bh);
                issued = t + 1;
            }
            griddep_wait();  // the combined state image and z are complete
            mbar_arrive_expect_tx(&bar_sz, sbytes + (uint32_t)MP * 4);
            bulk_load(sS, p.Simg + (size_t)bh * sbytes, sbytes, &bar_sz);
            bulk_load(sz, p.z + (size_t)bh * MP, (uint32_t)MP * 4, &bar_sz);
            for (int t = issued; t < T; ++t) {
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
            mbar_wait(&bar_sz, 0, &never);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const int nN = two ? 1 : 2;    // N blocks of the projection
            const int Nb = two ? MP : MP / 2;
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
            bool have_sz = false;
            auto issue_out = [&](int t) -> bool {
                const int s = t % nslot, k = t / nslot;
                if (!have_sz && !(have_sz = mbar_wait(&bar_sz, 0, &abort_flag))) return false;
                if (!mbar_wait(&bar_phi[s], k & 1, &abort_flag)) return false;
                tc_fence_after();
                for (int ks = 0; ks < MP / 16; ++ks) {
                    uint64_t bd = sdesc_sw128(smem_u32(sS + ks * 2048), (uint32_t)MP * 128, 1024);
                    mma_ts(tbase + s * slot_cols + num_off, tbase + s * slot_cols + phi_col_r(ks), bd, idesc_o, ks > 0);
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
        // Warp ew reads TMEM lane quarter q = warp % 4 (tokens 32q..32q+31 of the tile) and column
        // group cg = ew / 4: features [cg Wf, (cg+1) Wf) in the first pass, output columns
        // [cg D/4, (cg+1) D/4) in the second.
        const int ew = warp - 2;
        const int q = warp & 3, cg = ew >> 2;
        const int r = q * 32 + lane;  // token row of the tile
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const float A2 = p.scale * kLog2e;
        const bool exp_kind = KIND == kKindExp;
        bool failed = !mbar_wait(&bar_const, 0, &abort_flag);
        __syncwarp();
        bool have_sz = false;

        // phi for 32 raw projections, row constant cst; den accumulates bf16(phi) * z.
        auto features32 = [&](uint32_t (&v)[32], const float* zr, float cst, uint32_t (&pk)[16], float& dsum) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 z4 = *reinterpret_cast<const float4*>(zr + i);
                float f[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    f[k] = exp_kind ? ex2(fmaf(__uint_as_float(v[i + k]), A2, -cst))
                                    : phi_plain(__uint_as_float(v[i + k]) * p.scale, KIND, 1.f, p.relu_eps_s);
                const uint32_t w0 = pack_bf16(f[0], f[1]), w1 = pack_bf16(f[2], f[3]);
                pk[i / 2] = w0;
                pk[i / 2 + 1] = w1;
                dsum = fmaf(__uint_as_float(w0 << 16), z4.x, dsum);
                dsum = fmaf(__uint_as_float(w0 & 0xFFFF0000u), z4.y, dsum);
                dsum = fmaf(__uint_as_float(w1 << 16), z4.z, dsum);
                dsum = fmaf(__uint_as_float(w1 & 0xFFFF0000u), z4.w, dsum);
            }
        };

        auto epi1 = [&](int t) -> bool {
            const int s = t % nslot, k = t / nslot;
            const bool ok = mbar_wait(&bar_ufull[s], k & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            const uint32_t ua = tbase + lane_off + s * slot_cols;
            float* mx = sMax + (t & 1) * 512;
            float* dn = sDen + (t & 1) * 512;
            float dsum = 0.f;
            if (two) {
                // Wf <= 64: hold this warp's projections in registers across the row-max exchange.
                uint32_t v0[32], v1[32];
                float rmax = -INFINITY;
                tmem_ld32(ua + cg * Wf, v0);
                if (Wf == 64) tmem_ld32(ua + cg * Wf + 32, v1);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) rmax = fmaxf(rmax, __uint_as_float(v0[i]));
                if (Wf == 64) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) rmax = fmaxf(rmax, __uint_as_float(v1[i]));
                }
                mx[cg * 128 + r] = rmax;
                named_bar(1, kEpiThreads);  // every warp has its U values: U may now be overwritten
                rmax = fmaxf(fmaxf(mx[r], mx[128 + r]), fmaxf(mx[256 + r], mx[384 + r]));
                if (!have_sz) {  // z (from the preceding kernels) is needed from here on
                    have_sz = mbar_wait(&bar_sz, 0, &abort_flag);
                    __syncwarp();
                }
                const float cst = exp_kind ? A2 * rmax : 0.f;
                uint32_t pk[16];
                features32(v0, sz + cg * Wf, cst, pk, dsum);
                tmem_st16(ua + cg * (Wf / 2), pk);
                if (Wf == 64) {
                    features32(v1, sz + cg * Wf + 32, cst, pk, dsum);
                    tmem_st16(ua + cg * (Wf / 2) + 16, pk);
                }
            } else {
                // Wf = 96 or 128: max pass, exchange, then reload and pack into the own range.
                float rmax = -INFINITY;
                for (int c0 = 0; c0 < Wf; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(ua + cg * Wf + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) rmax = fmaxf(rmax, __uint_as_float(v[i]));
                }
                mx[cg * 128 + r] = rmax;
                named_bar(1, kEpiThreads);
                rmax = fmaxf(fmaxf(mx[r], mx[128 + r]), fmaxf(mx[256 + r], mx[384 + r]));
                if (!have_sz) {
                    have_sz = mbar_wait(&bar_sz, 0, &abort_flag);
                    __syncwarp();
                }
                const float cst = exp_kind ? A2 * rmax : 0.f;
                for (int c0 = 0; c0 < Wf; c0 += 32) {
                    uint32_t v[32], pk[16];
                    tmem_ld32(ua + cg * Wf + c0, v);
                    tmem_ld_wait();
                    features32(v, sz + cg * Wf + c0, cst, pk, dsum);
                    tmem_st16(ua + cg * Wf + c0 / 2, pk);
                }
            }
            dn[cg * 128 + r] = dsum;
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
            const float* dn = sDen + (t & 1) * 512;
            const float inv = 1.f / (((dn[r] + dn[128 + r]) + dn[256 + r]) + dn[384 + r]);
            constexpr int kC = D / 4;  // output columns per column group
            const uint32_t na = tbase + lane_off + s * slot_cols + num_off + cg * kC;
            uint32_t v[32];
            if constexpr (kC == 32) {
                tmem_ld32(na, v);
            } else {
                uint32_t v16[16];
                tmem_ld16(na, v16);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = v16[i];
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_ufree[s]);
            // Each thread stores whole 32-byte sectors of its own row (rows past n are not written).
            const int row = (t0 + t) * kTile + r;
            if (row < p.n && FAVOR_IN_BOUNDS(bh < (int)gridDim.y && (cg + 1) * kC <= D)) {
                uint4* dst = reinterpret_cast<uint4*>(p.Y + ((size_t)bh * p.n + row) * D + cg * kC);
#pragma unroll
                for (int cc = 0; cc < kC / 8; ++cc) {
                    uint4 o;
                    o.x = pack_bf16(__uint_as_float(v[8 * cc + 0]) * inv, __uint_as_float(v[8 * cc + 1]) * inv);
                    o.y = pack_bf16(__uint_as_float(v[8 * cc + 2]) * inv, __uint_as_float(v[8 * cc + 3]) * inv);
                    o.z = pack_bf16(__uint_as_float(v[8 * cc + 4]) * inv, __uint_as_float(v[8 * cc + 5]) * inv);
                    o.w = pack_bf16(__uint_as_float(v[8 * cc + 6]) * inv, __uint_as_float(v[8 * cc + 7]) * inv);
                    dst[cc] = o;
                }
            }
            return ok;
        };
        // Every epilogue thread runs the whole schedule (failed waits return at once), so the named
        // barriers always see all epilogue threads.
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
