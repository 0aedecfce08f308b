// Tensor-core (tcgen05 + TMA + TMEM) feature map phi(X) for bf16 inputs, fp32 output.
//
// Per 128-token tile of one head: U = X_tile Omega^T on the tensor cores (tokens on TMEM lanes,
// fp32 accumulate), then the epilogue applies the feature map of the "Performer" paper note's FAVOR+
// section exactly, per element,
//     phi_r(x) = exp(w_r . x^ - |x^|^2 / 2 - stab) / sqrt(m)        (exp family)
//     phi_r(x) = max(0, w_r . x^) / sqrt(m) + eps                   (ReLU family)
// with |x^|^2 from the tile in shared memory, and stores the rows in fp32.
// Stabilisers: NONE (0), ROW (the row's largest exponent, exchanged between the four warps that
// share a row), HEAD (the head's largest exponent, from a first launch of the same kernel in
// max-only mode that atomically raises an order-preserving encoding of it per head).
#pragma once

#include "tc.cuh"
#include "tc_noncausal.cuh"  // ex2, sq_acc helpers

namespace favor {
namespace tcf {

using namespace favor::tc;
using tcnc::ex2;

constexpr int kTile = 128;
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + 32 * kEpiWarps;

struct FeatParams {
    int n, m, m_pad;
    int tiles_per_cta;
    int kind, stab;
    int max_only;          // 1: only raise head_max (stab HEAD, first launch)
    float relu_eps;
    float scale;           // d^(-1/4)
    float* Phi;            // [BH][n][m] fp32
    unsigned* head_max;    // [BH], ordered encoding (stab HEAD)
};

template <int D>
struct FeatSmem {
    static constexpr int kStages = D == 64 ? 3 : 2;
    static constexpr int kTileBytes = kTile * D * 2;
    static size_t bytes(int m_pad) { return 1024 + (size_t)m_pad * D * 2 + (size_t)kStages * kTileBytes + 4096; }
};

// Squared norm of row `row` of a [128 x D] bf16 tile (D/64 swizzled regions of 16 KB).
template <int D>
__device__ __forceinline__ float row_sqnorm(const uint8_t* tile, int row) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int a = 0; a < D / 64; ++a) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(tile + a * 16384 + sw128_offset(row, c));
            tcnc::sq_acc_bf16x2(v.x, s0, s1);
            tcnc::sq_acc_bf16x2(v.y, s0, s1);
            tcnc::sq_acc_bf16x2(v.z, s0, s1);
            tcnc::sq_acc_bf16x2(v.w, s0, s1);
        }
    }
    return s0 + s1;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    features_tc(const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mOm, FeatParams p) {
    using SM = FeatSmem<D>;
    constexpr int NS = SM::kStages;
    constexpr int kAtoms = D / 64;
    extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 by hand below
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int MP = p.m_pad;
    uint8_t* sOm = smem;                        // kAtoms regions of MP rows x 128 B
    uint8_t* sX = sOm + (size_t)MP * D * 2;     // NS stages
    float* sMax = reinterpret_cast<float*>(sX + (size_t)NS * SM::kTileBytes);  // [2][4][128]
    __shared__ uint64_t bar_full[NS], bar_empty[NS], bar_om, bar_ufull[2], bar_ufree[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y;
    const int tiles_head = (p.n + kTile - 1) / kTile;
    const int t0 = blockIdx.x * p.tiles_per_cta;
    const int T = max(0, min(tiles_head, t0 + p.tiles_per_cta) - t0);
    const bool two = MP <= 256;
    const int nslot = two ? 2 : 1;
    const uint32_t slot_cols = two ? 256u : 512u;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1 + kEpiWarps);  // MMA commit + every epilogue warp (norms read)
        }
        mbar_init(&bar_om, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_ufull[i], 1);
            mbar_init(&bar_ufree[i], kEpiWarps);
        }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&mX);
            tma_prefetch_desc(&mOm);
            mbar_arrive_expect_tx(&bar_om, (uint32_t)MP * D * 2);
            for (int a = 0; a < kAtoms; ++a)
                for (int r0 = 0; r0 < MP; r0 += 128)
                    tma_load_2d(sOm + (size_t)a * MP * 128 + r0 * 128, &mOm, &bar_om, a * 64, r0);
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int st = t % NS;
                if (!mbar_wait(&bar_empty[st], ((t / NS) & 1) ^ 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&bar_full[st], SM::kTileBytes);
                for (int a = 0; a < kAtoms; ++a)
                    tma_load_3d(sX + (size_t)st * SM::kTileBytes + a * 16384, &mX, &bar_full[st], a * 64,
                                (t0 + t) * kTile, bh);
                issued = t + 1;
            }
            for (int t = max(0, issued - NS); t < issued; ++t) {
                volatile int never = 0;
                mbar_wait(&bar_full[t % NS], (t / NS) & 1, &never);
            }
            volatile int never = 0;
            mbar_wait(&bar_om, 0, &never);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const int nN = two ? 1 : 2;
            const int Nb = two ? MP : MP / 2;
            const uint32_t idesc = idesc_bf16(128, Nb, false, false);
            bool ok = mbar_wait(&bar_om, 0, &abort_flag);
            tc_fence_after();
            for (int t = 0; t < T && ok; ++t) {
                const int s = t % nslot, st = t % NS, k = t / nslot;
                ok = mbar_wait(&bar_full[st], (t / NS) & 1, &abort_flag) &&
                     mbar_wait(&bar_ufree[s], (k & 1) ^ 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint8_t* xt = sX + (size_t)st * SM::kTileBytes;
                for (int nb = 0; nb < nN; ++nb) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const int a = ks / 4, w = ks % 4;
                        uint64_t ad = sdesc_sw128(smem_u32(xt + a * 16384 + w * 32), 16, 1024);
                        uint64_t bd = sdesc_sw128(smem_u32(sOm + (size_t)a * MP * 128 + (size_t)nb * Nb * 128 + w * 32), 16, 1024);
                        mma_ss(tbase + s * slot_cols + nb * Nb, ad, bd, idesc, ks > 0);
                    }
                }
                mma_commit(&bar_ufull[s]);
                mma_commit(&bar_empty[st]);
            }
        }
    } else {
        // ---------------- epilogue: warp (q, cg): token rows 32q..32q+31, features [cg Wf, (cg+1) Wf) ----------------
        const int ew = warp - 2;
        const int q = warp & 3, cg = ew >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int Wf = MP / 4;
        const bool exp_kind = p.kind == kKindExp;
        const float A2 = p.scale * kLog2e;
        const float lsm = 0.5f * log2f((float)p.m);  // log2 sqrt(m)
        const float inv_sqrt_m = rsqrtf((float)p.m);
        float head_st = 0.f;
        if (exp_kind && p.stab == kStabHead && !p.max_only) head_st = ordered_decode(p.head_max[bh]);
        float run_max = -INFINITY;  // max-only mode: this thread's largest exponent
        bool failed = !mbar_wait(&bar_om, 0, &abort_flag);
        __syncwarp();
        for (int t = 0; t < T; ++t) {
            const int s = t % nslot, st = t % NS, k = t / nslot;
            failed |= !mbar_wait(&bar_full[st], (t / NS) & 1, &abort_flag);
            __syncwarp();
            const float h = exp_kind ? 0.5f * p.scale * p.scale * row_sqnorm<D>(sX + (size_t)st * SM::kTileBytes, r) : 0.f;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_empty[st]);
            failed |= !mbar_wait(&bar_ufull[s], k & 1, &abort_flag);
            __syncwarp();
            tc_fence_after();
            const uint32_t ua = tbase + lane_off + s * slot_cols + cg * Wf;
            const int row = (t0 + t) * kTile + r;
            const bool valid = row < p.n;
            // row maximum of the raw projections (ROW stabiliser, or the max-only pass)
            float rmax = -INFINITY;
            const bool need_max = exp_kind && (p.stab == kStabRow || p.max_only);
            if (need_max) {
                for (int c0 = 0; c0 < Wf; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(ua + c0, v);
                    tmem_ld_wait();
                    for (int i = 0; i < 32; ++i)
                        if (cg * Wf + c0 + i < p.m) rmax = fmaxf(rmax, __uint_as_float(v[i]));
                }
            }
            if (p.max_only) {
                if (valid && rmax > -INFINITY) run_max = fmaxf(run_max, A2 * rmax / kLog2e - h);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_ufree[s]);
                continue;
            }
            float stab_r = 0.f;  // in log2 units, h included
            if (exp_kind) {
                if (p.stab == kStabRow) {
                    float* mx = sMax + (t & 1) * 512;
                    mx[cg * 128 + r] = rmax;
                    named_bar(1, 32 * kEpiWarps);
                    rmax = fmaxf(fmaxf(mx[r], mx[128 + r]), fmaxf(mx[256 + r], mx[384 + r]));
                    stab_r = A2 * rmax;  // u_max = sc * rmax - h: the h terms cancel
                } else {
                    stab_r = (h + head_st) * kLog2e;
                }
            }
            for (int c0 = 0; c0 < Wf; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(ua + c0, v);
                tmem_ld_wait();
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float a = __uint_as_float(v[i]);
                    o[i] = exp_kind ? ex2(fmaf(a, A2, -stab_r - lsm)) : phi_plain(a * p.scale, p.kind, inv_sqrt_m, p.relu_eps);
                }
                const int f0 = cg * Wf + c0;
                // (features past m, in the padding of the last group, are skipped by the guards below)
                if (valid && FAVOR_IN_BOUNDS(bh < (int)gridDim.y && row < p.n)) {
                    float* dst = p.Phi + ((size_t)bh * p.n + row) * p.m + f0;
                    if (f0 + 32 <= p.m && (p.m & 3) == 0) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
                    } else {
                        for (int i = 0; i < 32; ++i)
                            if (f0 + i < p.m) dst[i] = o[i];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_ufree[s]);
        }
        if (p.max_only) {
            const float wm = warp_max(run_max);
            if (lane == 0 && wm > -INFINITY) atomicMax(p.head_max + bh, ordered_encode(wm));
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

}  // namespace tcf
}  // namespace favor
