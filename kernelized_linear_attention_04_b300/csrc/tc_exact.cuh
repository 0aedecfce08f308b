// Exact softmax attention Y = softmax(Q K^T / sqrt(d)) V (optionally causal), bf16 in / fp32
// accumulate, d = 64, on the tensor cores: the quadratic operator FAVOR+ approximates ("Performer"
// paper note, *Standard Attention Cost*), the comparator of the speed and divergence sweep
// ("Linear Attention and the Performer", *Exercise*).
//
// One CTA handles 128 query rows of one head and walks the key tiles of 128 with an online softmax:
//   S_j  = Q K_j^T                      (tcgen05, A and B from shared memory)   -> TMEM
//   m    = max(m, rowmax S_j); P_j = 2^((S_j - m) log2 e / sqrt(d)) as bf16, in place in TMEM
//   PV_j = P_j V_j                      (tcgen05, A = P_j from TMEM)            -> TMEM
//   O    = 2^((m_old - m) ...) O + PV_j, l likewise (in registers)
// S and PV have two TMEM buffers each, so S_{j+1} and PV_j run while P_j / O are formed.
// Warp 0: TMA (Q once, K and V in a ring of three stages); warp 1: MMA issuer; warps 2-9: softmax
// team, two warps per TMEM lane quarter (64 keys of S and 32 columns of O each), which exchange
// their row maxima through shared memory once per tile.
#pragma once

#include "tc.cuh"
#include "tc_noncausal.cuh"  // ex2

namespace favor {
namespace tce {

using namespace favor::tc;
using tcnc::ex2;

constexpr int kTile = 128;
constexpr int kD = 64;
constexpr int kStages = 3;
constexpr int kSoftWarps = 8;
constexpr int kThreads = 64 + 32 * kSoftWarps;
constexpr int kTileBytes = kTile * kD * 2;
constexpr uint32_t kColS = 0;    // two S / P buffers of 128 columns
constexpr uint32_t kColO = 256;  // two PV buffers of 64 columns

struct ExactParams {
    int n;
    int causal;
    float c;  // log2 e / sqrt(d)
    __nv_bfloat16* Y;
};

struct ExactSmem {
    static size_t bytes() { return 1024 + (size_t)(1 + 2 * kStages) * kTileBytes + 2 * 2 * 128 * 4; }
};

__global__ void __launch_bounds__(kThreads, 1)
    exact_attn(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, ExactParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + kTileBytes;                 // kStages tiles
    uint8_t* sV = sK + (size_t)kStages * kTileBytes;  // kStages tiles
    float* sMx = reinterpret_cast<float*>(sV + (size_t)kStages * kTileBytes);  // [2][2][128]
    __shared__ uint64_t bar_q, bar_kfull[kStages], bar_vfull[kStages], bar_kvfree[kStages];
    __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2], bar_ofree[2], bar_drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y;
    const int qt = blockIdx.x;  // query tile
    const int tiles = (p.n + kTile - 1) / kTile;
    const int J = p.causal ? qt + 1 : tiles;  // key tiles this CTA reads

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_q, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bar_kfull[i], 1);
            mbar_init(&bar_vfull[i], 1);
            mbar_init(&bar_kvfree[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar_s[b], 1);
            mbar_init(&bar_p[b], kSoftWarps);
            mbar_init(&bar_o[b], 1);
            mbar_init(&bar_ofree[b], kSoftWarps);
        }
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&mQ);
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mV);
            mbar_arrive_expect_tx(&bar_q, kTileBytes);
            tma_load_3d(sQ, &mQ, &bar_q, 0, qt * kTile, bh);
            int issued = 0;
            for (int j = 0; j < J; ++j) {
                const int st = j % kStages;
                if (j >= kStages && !mbar_wait(&bar_kvfree[st], ((j / kStages) & 1) ^ 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&bar_kfull[st], kTileBytes);
                tma_load_3d(sK + (size_t)st * kTileBytes, &mK, &bar_kfull[st], 0, j * kTile, bh);
                mbar_arrive_expect_tx(&bar_vfull[st], kTileBytes);
                tma_load_3d(sV + (size_t)st * kTileBytes, &mV, &bar_vfull[st], 0, j * kTile, bh);
                issued = j + 1;
            }
            volatile int never = 0;
            mbar_wait(&bar_q, 0, &never);
            for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j) {
                mbar_wait(&bar_kfull[j % kStages], (j / kStages) & 1, &never);
                mbar_wait(&bar_vfull[j % kStages], (j / kStages) & 1, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S = Q K^T
            constexpr uint32_t id_o = idesc_bf16(128, kD, false, true);    // PV = P V (V MN-major)
            bool ok = mbar_wait(&bar_q, 0, &abort_flag);
            auto issue_s = [&](int j) -> bool {
                const int st = j % kStages, b = j & 1;
                if (!mbar_wait(&bar_kfull[st], (j / kStages) & 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* kt = sK + (size_t)st * kTileBytes;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint64_t ad = sdesc_sw128(smem_u32(sQ + ks * 32), 16, 1024);
                    const uint64_t bd = sdesc_sw128(smem_u32(kt + ks * 32), 16, 1024);
                    mma_ss(tbase + kColS + 128u * b, ad, bd, id_s, ks > 0);
                }
                mma_commit(&bar_s[b]);
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int st = j % kStages, b = j & 1, u = j >> 1;
                if (!mbar_wait(&bar_p[b], u & 1, &abort_flag)) return false;
                if (!mbar_wait(&bar_vfull[st], (j / kStages) & 1, &abort_flag)) return false;
                if (!mbar_wait(&bar_ofree[b], (u & 1) ^ 1, &abort_flag)) return false;
                tc_fence_after();
                const uint8_t* vt = sV + (size_t)st * kTileBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    // P packed per half: keys [64 h, 64 h + 64) in columns [64 h, 64 h + 32)
                    const uint32_t pcol = kColS + 128u * b + 64u * (uint32_t)(ks >> 2) + 8u * (uint32_t)(ks & 3);
                    const uint64_t bd = sdesc_sw128(smem_u32(vt + ks * 2048), 16, 1024);
                    mma_ts(tbase + kColO + 64u * b, tbase + pcol, bd, id_o, ks > 0);
                }
                mma_commit(&bar_o[b]);
                mma_commit(&bar_kvfree[st]);
                return true;
            };
            if (ok && J > 0) ok = issue_s(0);
            for (int j = 0; j < J && ok; ++j) {
                if (j + 1 < J && !(ok = issue_s(j + 1))) break;
                ok = issue_pv(j);
            }
            mma_commit(&bar_drain);
            volatile int never = 0;
            mbar_wait(&bar_drain, 0, &never);
        }
    } else {
        // ---------------- softmax team ----------------
        const int sw = warp - 2;
        const int q = warp & 3, h = sw >> 2;
        const int r = q * 32 + lane;
        const int i_tok = qt * kTile + r;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        bool failed = false;
        float mrow = -INFINITY, l = 0.f, alpha_prev = 1.f;
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
        // O = alpha O + PV_j (columns [32 h, 32 h + 32)), then PV buffer j & 1 is free
        auto fold = [&](int j, float alpha) {
            const int b = j & 1;
            failed |= !mbar_wait(&bar_o[b], (j >> 1) & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tbase + lane_off + kColO + 64u * b + 32u * h, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_ofree[b]);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = fmaf(o[i], alpha, __uint_as_float(v[i]));
        };
        for (int j = 0; j < J; ++j) {
            const int b = j & 1;
            failed |= !mbar_wait(&bar_s[b], (j >> 1) & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            const uint32_t sa = tbase + lane_off + kColS + 128u * b + 64u * h;
            // keys [128 j + 64 h, ... + 64): masked past n, and past the query in the diagonal tile
            const int key0 = j * kTile + 64 * h;
            const int lim = p.causal ? min(i_tok, p.n - 1) : p.n - 1;  // last key this row may see
            float mx = -INFINITY;
            uint32_t v0[32], v1[32];
            tmem_ld32(sa, v0);
            tmem_ld32(sa + 32, v1);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                if (key0 + k <= lim) mx = fmaxf(mx, __uint_as_float(v0[k]));
                if (key0 + 32 + k <= lim) mx = fmaxf(mx, __uint_as_float(v1[k]));
            }
            float* mxb = sMx + (j & 1) * 256;
            mxb[h * 128 + r] = mx;
            named_bar(1, 32 * kSoftWarps);
            const float mnew = fmaxf(mrow, fmaxf(mxb[r], mxb[128 + r]));
            const float alpha = mrow == -INFINITY ? 0.f : ex2((mrow - mnew) * p.c);
            mrow = mnew;
            const float off = mnew * p.c;
            float sum = 0.f;
            // P_j packed in place: keys [64 h, 64 h + 64) -> columns [64 h, 64 h + 32) of the buffer,
            // which only this warp has read
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t(&v)[32] = hh == 0 ? v0 : v1;
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const int kk = key0 + 32 * hh + k;
                    const float a0 = kk <= lim ? ex2(fmaf(__uint_as_float(v[k]), p.c, -off)) : 0.f;
                    const float a1 = kk + 1 <= lim ? ex2(fmaf(__uint_as_float(v[k + 1]), p.c, -off)) : 0.f;
                    w[k / 2] = pack_bf16(a0, a1);
                    sum += __uint_as_float(w[k / 2] << 16) + __uint_as_float(w[k / 2] & 0xFFFF0000u);
                }
                tmem_st16(sa + 16u * hh, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_p[b]);
            l = fmaf(l, alpha, sum);
            if (j > 0) fold(j - 1, alpha_prev);
            alpha_prev = alpha;
        }
        if (J > 0) fold(J - 1, alpha_prev);
        // both halves' sums of the bf16-rounded probabilities make the row's denominator
        float* lb = sMx + (J & 1) * 256;
        lb[h * 128 + r] = l;
        named_bar(1, 32 * kSoftWarps);
        const float inv = 1.f / (lb[r] + lb[128 + r]);
        if (i_tok < p.n && FAVOR_IN_BOUNDS(bh < (int)gridDim.y && 32 * h + 32 <= kD)) {
            uint4* dst = reinterpret_cast<uint4*>(p.Y + ((size_t)bh * p.n + i_tok) * kD + 32 * h);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 ov;
                ov.x = pack_bf16(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
                ov.y = pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
                ov.z = pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
                ov.w = pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
                dst[c] = ov;
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

}  // namespace tce
}  // namespace favor
