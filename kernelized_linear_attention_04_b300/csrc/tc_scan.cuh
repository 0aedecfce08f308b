// Tensor-core (tcgen05 + TMA + TMEM) causal FAVOR+ scan, bf16 in / fp32 accumulate, d = 64,
// m <= 512.
//
// A group of CS = ceil(m / 128) CTAs walks the 128-token tiles of one head in order; CTA `rank`
// of the group owns the features [128 rank, 128 rank + 128). Per tile t (query rows i, keys j of
// the tile) each CTA forms, over its own features,
//   num_i = phi(q_i) S_<t + sum_{j <= i} (phi(q_i) . phi(k_j)) v_j
//   den_i = phi(q_i) z_<t + sum_{j <= i}  phi(q_i) . phi(k_j)
// and then S_<t+1 = S_<t + Phi(K_t)^T V_t, z_<t+1 = z_<t + Phi(K_t)^T 1 ("Performer for vision",
// *How It Works*, Step 2: prefix sums; the state is carried every 128 tokens and keys are masked
// by j <= i inside the tile, which for two 64-token chunks is exactly their chunked prefix sum).
// The CTAs of a group then combine their partial results row by row: each writes its partial rows
// of tile t into a ring of kRing tiles in global memory (L2-resident) and counts them into the
// group's counters; a separate warp team of each CTA combines the rows it finalises once every
// CTA's rows are counted in, so that neither the tensor-core pipeline nor the NUM drain waits on
// a peer.
//
// The grid is persistent: G groups (at most one CTA per SM, all resident together, launched
// cooperatively when CS > 1), group g taking the heads g, g + G, g + 2G, ... one after another.
// The groups need no common GPC, as thread-block clusters would (four-CTA clusters leave SMs of
// every GPC idle). Within a CTA the tiles of all its heads form one sequence (index gt) that
// drives every buffer and barrier phase; at a head's first tile the state restarts from zero.
//
// Every contraction runs on the tensor cores, with the A operand in TMEM wherever it is produced
// there:
//   P_K   = K_t Omega_g^T        (A, B from shared memory)           -> TMEM, tokens on lanes
//   P_Q   = Q_t Omega_g^T        (same)                              -> TMEM, tokens on lanes
//   SC    = phi(Q) phi(K)^T      (A: phi(Q) packed bf16 in TMEM, B: phi(K) in shared memory)
//   NUM   = phi(Q) [S | z]_<t    (A: phi(Q) in TMEM, B: bf16 image of the state; for the exp family
//                                 a second MMA adds phi(Q) S_lo, the rounding remainder of S)
//   [S|z] += phi(K)^T [V | 1]    (A: phi(K) in shared memory, read transposed)
//   NUM  += A~ [V | 1]           (A: masked scores A~ packed bf16 in TMEM, in place of SC)
// Columns 64 and 65 of NUM add up to the denominator (the ones column of [V | 1]; z and its
// rounding remainder in the state image), so no row sum is formed on the CUDA cores. MMA issue
// order per tile: scores(t), inter(t), proj Q(t+1), state(t), intra(t), proj K(t+2); each warp
// team below works on one stage while the tensor cores run the others.
//
// Warp roles:
//   warp 0       TMA producer (lane 0): Omega_g once; K and Q single-buffered, V double-buffered.
//   warp 1       MMA issuer (the warp waits, one elected lane issues).
//   warps 2-9    Q team: phi(Q_t) from P_Q (two warps per TMEM lane quarter, 64 features each) into
//                the packed phi(Q) columns; for exp features the exact row maximum over the CTA's
//                features is exchanged between the two halves of the row.
//   warps 10-13  K team: phi(K_t) from P_K into shared memory (K-major rows, the scores' B operand
//                and, read transposed, the state's A operand); the running key stabiliser.
//   warps 14-17  A team: SC -> A~ (masked by j <= i, bf16) in place; then the bf16 image of
//                [S | z] after the state update (rescaled first if the key stabiliser rose).
//   warps 18-21  O team: NUM -> y (alone: the output; in a group: the partial rows, to the ring).
//   warps 22-25  X team (CS > 1 only): the rows this CTA finalises, from the ring's partials.
//   warps 26-27  signal warps (CS > 1 only): release a tile's stored partial rows to the group,
//                and report the slots the X team has read.
//
// Stabilisers (exp family; Y does not depend on them, both cancel between num and den):
//   queries: c_i = the exact largest w_r . q^_i over the CTA's features (the row's largest feature
//   is 1); the common -|q^_i|^2/2 is dropped;
//   keys: a running constant per CTA, the exact largest exponent w_r . k^_j - |k^_j|^2/2 seen so
//   far over the CTA's features and the head's keys, raised (and the state rescaled) only when a
//   tile exceeds it by more than kSlackHi binary orders of magnitude;
//   across the group, each CTA's partial row y_g = num_g / den_g carries the log-weight
//   l_g = log2(den_g) + c_i + beta; the owner of the row weights the partials by 2^(l_g - max l).
// The common factor 1/sqrt(m) is dropped. The generalized-ReLU and elu + 1 families have no
// stabiliser.
#pragma once

#include <cuda_fp16.h>

#include "tc.cuh"
#include "tc_noncausal.cuh"  // shared helpers: ex2, tile_row_sqnorm

namespace favor {
namespace tcs {

using namespace favor::tc;
using tcnc::ex2;
using tcnc::tile_row_sqnorm;

constexpr int kTile = 128;
constexpr int kD = 64;
constexpr int kMaxCluster = 4;                    // m <= 512: CTAs per group
constexpr int kQWarp0 = 2, kQWarps = 8;
constexpr int kKWarp0 = kQWarp0 + kQWarps, kKWarps = 4;
constexpr int kAWarp0 = kKWarp0 + kKWarps, kAWarps = 4;
constexpr int kOWarp0 = kAWarp0 + kAWarps, kOWarps = 4;
constexpr int kXWarp0 = kOWarp0 + kOWarps, kXWarps = 4;
constexpr int kSWarp0 = kXWarp0 + kXWarps, kSWarps = 2;  // ring signalling: full, free
constexpr int kThreads = 32 * (kSWarp0 + kSWarps);  // 896
constexpr int kTileBytes = kTile * kD * 2;          // 16 KB: [128 x 64] bf16
constexpr int kPhiBytes = kTile * 128 * 2;          // 32 KB: [128 tokens x 128 features] bf16
constexpr int kPrefetch = 3;                        // tiles of K, Q, V prefetched into L2 ahead of their loads
constexpr int kRing = 4;                            // tiles of partial rows in flight per head
constexpr int kXChunks = 9;                         // 16-byte chunks of a partial row: 8 of y (fp16), log-weight and scales
constexpr float kSlackHi = 16.f;                    // key stabiliser rises once exceeded by 2^16
constexpr int kMaxCtas = 160;                       // persistent grid bound (at least a device's SMs)
constexpr int kFlagWords = 16;                      // per group: kRing full and kRing free counters, padded

// Timeline of one CTA for profiling builds (compiled with -DFAVOR_SCAN_TRACE): the SM clock at
// named points of each role, for the first kTraceTiles tiles of CTA 0. Off in the library.
#ifdef FAVOR_SCAN_TRACE
constexpr int kTraceTiles = 16, kTraceEvents = 32;
__device__ unsigned long long g_scan_trace[kTraceTiles][kTraceEvents];
__device__ unsigned long long g_scan_cta_time[2048][6];  // per CTA: clock and globaltimer at start and end, SM id
__device__ unsigned long long g_scan_cta_wait[2048][10];  // per CTA: cycles the MMA warp spent in each kind of wait
#define TIMED_WAIT(i, call) ([&]() { const unsigned long long s_ = clock64(); const bool r_ = (call); wacc[i] += clock64() - s_; return r_; }())
#ifndef FAVOR_SCAN_TRACE_FROM
#define FAVOR_SCAN_TRACE_FROM 0
#endif
#define SCAN_TRACE(t, ev)                                                                            \
    do {                                                                                             \
        const int tr_t_ = (t) - FAVOR_SCAN_TRACE_FROM;                                               \
        if (blockIdx.x == 0 && tr_t_ >= 0 && tr_t_ < kTraceTiles) g_scan_trace[tr_t_][(ev)] = clock64(); \
    } while (0)
#else
#define SCAN_TRACE(t, ev) ((void)0)
#define TIMED_WAIT(i, call) (call)
#endif

// TMEM columns (512 allocated)
constexpr uint32_t kColS = 0;      // [S | z]: 64 columns of S, z in column 64, 65..79 zero
constexpr uint32_t kColPQ = 80;    // phi(Q) packed bf16: 128 features in 64 columns
constexpr uint32_t kColNum = 144;  // NUM: 64 numerator columns, denominator parts in columns 64, 65
constexpr uint32_t kColR0 = 224;   // two 128-column regions: P_K(t), then P_Q(t), then SC(t) / A~(t)

// Shared memory offsets from the 1024-aligned base.
constexpr uint32_t kOffOm = 0;
constexpr uint32_t kOffQ = kOffOm + kTileBytes;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kTileBytes;          // two buffers
constexpr uint32_t kOffPK = kOffV + 2 * kTileBytes;     // two phi(K) buffers
constexpr uint32_t kOffSnap = kOffPK + 2 * kPhiBytes;   // S image (bf16 hi), MN-major [128 features x 64]
constexpr uint32_t kOffZb = kOffSnap + kTileBytes;      // z image: elements 0 (hi) and 1 (lo) of each feature row
constexpr uint32_t kOffSlo = kOffZb + kTileBytes;       // S rounding remainder (bf16 lo), exp family
constexpr uint32_t kOffOnes = kOffSlo + kTileBytes;     // element 0 of each token row = 1
constexpr uint32_t kOffCq = kOffOnes + kTileBytes;      // [2][128] f32 query row constants
constexpr uint32_t kOffMx = kOffCq + 2 * 128 * 4;       // [2][2][128] f32 row-max halves
constexpr uint32_t kOffEnd = kOffMx + 2 * 2 * 128 * 4;

struct ScanParams {
    int n;
    int m;
    int kind;
    float relu_eps_s;  // relu_eps * sqrt(m): the features are scaled by sqrt(m) (a common factor)
    float scale;       // d^-1/4 (1 for elu + 1)
    __nv_bfloat16* Y;
    int bh;            // heads (B * H)
    int cs;            // CTAs per group, ceil(m / 128)
    uint8_t* ring;     // cs > 1: per group kRing x cs x kXChunks x 128 rows x 16 bytes (ScanWs)
    uint32_t* flags;   // cs > 1: per group kFlagWords counters, zero at launch (ScanWs)
};

struct ScanSmem {
    static size_t bytes() { return 1024 + kOffEnd; }
};

// Workspace of the scan (only for cs > 1): the groups' counters, then their rings of partial rows.
// Sized for the largest grid any device may get, min(BH, kMaxCtas / cs) groups.
struct ScanWs {
    static int max_groups(size_t BH, int cs) { return (int)(BH < (size_t)(kMaxCtas / cs) ? BH : (size_t)(kMaxCtas / cs)); }
    static size_t flag_bytes(size_t BH, int cs) { return ((size_t)max_groups(BH, cs) * kFlagWords * 4 + 255) & ~size_t(255); }
    __host__ __device__ static size_t ring_bytes(int cs) { return (size_t)kRing * cs * kXChunks * kTile * 16; }
    static size_t bytes(size_t BH, int cs) { return cs > 1 ? flag_bytes(BH, cs) + max_groups(BH, cs) * ring_bytes(cs) : 0; }
};

// bf16 image of 8 fp32 values as one 16-byte chunk, and (lo) the bf16 rounding of what the first
// image leaves out.
__device__ __forceinline__ uint4 pack8_hi(const uint32_t* v) {
    return make_uint4(pack_bf16(__uint_as_float(v[0]), __uint_as_float(v[1])),
                      pack_bf16(__uint_as_float(v[2]), __uint_as_float(v[3])),
                      pack_bf16(__uint_as_float(v[4]), __uint_as_float(v[5])),
                      pack_bf16(__uint_as_float(v[6]), __uint_as_float(v[7])));
}
__device__ __forceinline__ uint32_t lo_pair(uint32_t x0, uint32_t x1, uint32_t hw) {
    return pack_bf16(__uint_as_float(x0) - __uint_as_float(hw << 16), __uint_as_float(x1) - __uint_as_float(hw & 0xFFFF0000u));
}

// The CTA's abort word. The scan's waits spin inline on their phase and give up once it is set:
// the kernel's instruction footprint sets its speed, and a call to a bounded slow path at each
// wait site costs more code than the wait. The bound comes from the CTA's watchdog lane instead,
// which sets the word (and the timeout error) once no role has made progress for the wait limit;
// the waits that run after a role's last beat (the drains, the group counters) keep a bound of
// their own.
__shared__ int s_abort;
__shared__ uint32_t s_beat[3];  // progress: the MMA warp's, the O team's and the X team's tiles
__shared__ uint32_t s_done;     // warps (but the watchdog's) past the end of their role
__device__ __forceinline__ bool scan_wait(uint64_t* bar, uint32_t parity) {
    while (!mbar_try_wait(bar, parity))
        if (*reinterpret_cast<volatile int*>(&s_abort)) return false;
    return true;
}

// KIND: the feature family (kKindExp, kKindRelu, kKindElu), fixed per instance so that each
// instance carries only its own feature map and stabiliser code. CSX: the CTAs of a group, CS =
// ceil(m / 128), fixed per instance (1, 2, 3: the combine unrolled over exactly CS partials), or
// 0 for CS read from the parameters (used for CS = 4, where it measured faster than a fixed CS);
// with CS > 1 the ring, the X team and the signal warps, with CS = 1 the O team writes the output.
template <int KIND, int CSX>
__global__ void __launch_bounds__(kThreads, 1)
    causal_scan(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mOm, ScanParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 by hand below
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr bool GROUPED = CSX != 1;
    const int CS = CSX > 0 ? CSX : p.cs;
    const int G = (int)gridDim.x / CS;  // groups
    const int grp = (int)blockIdx.x / CS, rank = (int)blockIdx.x % CS;
    const int RP = (kTile + CS - 1) / CS;  // rows finalised by each CTA of the group
    const int feat0 = rank * 128;
    uint8_t* sOm = smem + kOffOm;
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sK = smem + kOffK;
    uint8_t* sV = smem + kOffV;
    uint8_t* sPK = smem + kOffPK;
    uint8_t* sSnap = smem + kOffSnap;
    uint8_t* sZb = smem + kOffZb;
    uint8_t* sSlo = smem + kOffSlo;
    uint8_t* sOnes = smem + kOffOnes;
    float* sCq = reinterpret_cast<float*>(smem + kOffCq);
    float* sMx = reinterpret_cast<float*>(smem + kOffMx);
    __shared__ uint64_t bar_om, bar_kfull, bar_kfree, bar_qfull, bar_qfree, bar_vfull[2], bar_vfree[2];
    __shared__ uint64_t bar_pk[2], bar_pkfree[2], bar_pq[2], bar_scr[2], bar_phkfree[2];
    __shared__ uint64_t bar_sc, bar_atil, bar_st, bar_inter, bar_num, bar_beta[4], bar_cq[2];
    __shared__ uint64_t bar_drain, bar_rfull[kRing], bar_rfree[kRing], bar_ostore[kRing], bar_xread[kRing];
    __shared__ uint32_t tmem_base;
    __shared__ float sBeta[4], sF[4], sKmx[4];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // extents for the debug build's bounds checks: output rows, one group's ring
    [[maybe_unused]] const size_t y_rows = (size_t)p.bh * p.n;
    [[maybe_unused]] const size_t ring_head = ScanWs::ring_bytes(CS);
    const int T = (p.n + kTile - 1) / kTile;
    // This CTA's tiles: those of its group's heads grp, grp + G, ..., one sequence gt in [0, GT).
    // Roles that need a tile's head and place in it follow them with seq_next.
    const int GT = (p.bh - grp + G - 1) / G * T;
    auto seq_next = [&](int& hd, int& tl) {
        if (++tl == T) {
            tl = 0;
            hd += G;
        }
    };
    // the group's ring and counters (full: [0, kRing), free: [kRing, 2 kRing))
    uint8_t* const ring_grp = GROUPED ? p.ring + (size_t)grp * ScanWs::ring_bytes(CS) : nullptr;
    uint32_t* const flags = GROUPED ? p.flags + (size_t)grp * kFlagWords : nullptr;
    constexpr bool exp_kind = KIND == kKindExp;
    constexpr bool hilo = exp_kind;     // state image with its rounding remainder
    const float A2 = p.scale * kLog2e;  // projections -> exponents in binary orders of magnitude
    uint32_t eps2;                      // bf16x2 {eps, eps} of the ReLU family's floor
    {
        const __nv_bfloat162 e2 = __floats2bfloat162_rn(p.relu_eps_s, p.relu_eps_s);
        eps2 = *reinterpret_cast<const uint32_t*>(&e2);
    }
    // 32 raw projections -> 16 bf16x2 words of features (zero when `real` is false: padding
    // features of the last 128-feature group); c is the row or key constant of the exp family.
    auto features16 = [&](const uint32_t (&v)[32], uint32_t (&w)[16], bool real, float c) {
        if (!real) {
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = 0u;
        } else if constexpr (KIND == kKindExp) {
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = exp_pair(v[2 * k], v[2 * k + 1], A2, c);
        } else if constexpr (KIND == kKindRelu) {
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = relu_pair(v[2 * k], v[2 * k + 1], p.scale, p.relu_eps_s, eps2);
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                w[k] = pack_bf16(phi_plain(__uint_as_float(v[2 * k]), KIND, 1.f, 0.f),
                                 phi_plain(__uint_as_float(v[2 * k + 1]), KIND, 1.f, 0.f));
        }
    };

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_done = 0;
        s_beat[0] = s_beat[1] = s_beat[2] = 0;
        mbar_init(&bar_om, 1);
        mbar_init(&bar_kfull, 1);
        mbar_init(&bar_kfree, kKWarps);
        mbar_init(&bar_qfull, 1);
        mbar_init(&bar_qfree, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar_vfull[b], 1);
            mbar_init(&bar_vfree[b], 1);
            mbar_init(&bar_pk[b], 1);
            mbar_init(&bar_pkfree[b], kKWarps);
            mbar_init(&bar_pq[b], 1);
            // the scores of tile t may start: phi(Q_t) packed (Q team) and phi(K_t) stored (K team)
            mbar_init(&bar_scr[b], kQWarps + kKWarps);
            mbar_init(&bar_phkfree[b], 1);
            mbar_init(&bar_cq[b], kQWarps / 2);
        }
        for (int b = 0; b < 4; ++b) mbar_init(&bar_beta[b], 1);
        mbar_init(&bar_sc, 1);
        mbar_init(&bar_atil, kAWarps);
        mbar_init(&bar_st, 1);
        // the inter MMA of tile t may start: the state image of S_<t (A team) and NUM drained (O team)
        mbar_init(&bar_inter, kAWarps + kOWarps);
        mbar_init(&bar_num, 1);
        mbar_init(&bar_drain, 1);
        for (int i = 0; i < kRing; ++i) {
            // every CTA of the group has stored its partial rows of the slot's tile / read them
            mbar_init(&bar_rfull[i], 1);
            mbar_init(&bar_rfree[i], 1);
            // this CTA's partial rows of a slot are stored / its X team has read a slot
            mbar_init(&bar_ostore[i], kOWarps);
            mbar_init(&bar_xread[i], kXWarps);
        }
        fence_mbar_init();
    }
    // Constant operands: the ones column of [V | 1] (element 0 of every token row), and the initial
    // state image S_<0 = 0, z_<0 = 0. In the 128-byte swizzle, element 0 of row k sits in 16-byte
    // chunk (k mod 8) of the row.
    for (int i = threadIdx.x; i < kTileBytes / 16; i += blockDim.x) {
        const int row = i >> 3, chunk = i & 7;
        reinterpret_cast<uint4*>(sOnes)[i] = make_uint4(chunk == (row & 7) ? 0x00003F80u : 0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(sSnap)[i] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(sSlo)[i] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(sZb)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    if (warp == 1) tmem_alloc(&tmem_base, 512);
    __syncthreads();
    tc_fence_after();
#ifdef FAVOR_SCAN_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 2048) {
        g_scan_cta_time[blockIdx.x][0] = clock64();
        g_scan_cta_time[blockIdx.x][1] = globaltimer();
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_scan_cta_time[blockIdx.x][4] = smid;
    }
#endif
    const uint32_t tbase = tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer (lane 0) ----------------
        if (lane == 0) {
            tma_prefetch_desc(&mOm);
            tma_prefetch_desc(&mQ);
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mV);
            mbar_arrive_expect_tx(&bar_om, (uint32_t)kTileBytes);
            tma_load_2d(sOm, &mOm, &bar_om, 0, feat0);
            int kl = 0, ql = 0, vl = 0;  // tiles loaded
            // K, Q and V of the tiles kPrefetch ahead go to L2 first: the loads below have only
            // about one tile of lead (single K and Q buffers), less than a device-memory round
            // trip under load
            int pf = 1, ph = grp, pt = 0;  // the next tile to prefetch (tile 0 is loaded at once)
            seq_next(ph, pt);
            for (int gt = 0, hb = grp, tl = 0; gt < GT; ++gt, seq_next(hb, tl)) {
                const int b = gt & 1, u = gt >> 1;
                const int row = tl * kTile;
                for (; pf <= gt + kPrefetch && pf < GT; ++pf, seq_next(ph, pt)) {  // up to tile gt + kPrefetch
                    tma_prefetch_3d(&mK, 0, pt * kTile, ph);
                    tma_prefetch_3d(&mQ, 0, pt * kTile, ph);
                    tma_prefetch_3d(&mV, 0, pt * kTile, ph);
                }
                // K(gt) once the K team has taken the norms of K(gt-1) and P_K(gt-1) has read it
                if (gt > 0 && !scan_wait(&bar_kfree, (gt - 1) & 1)) break;
                mbar_arrive_expect_tx(&bar_kfull, kTileBytes);
                tma_load_3d(sK, &mK, &bar_kfull, 0, row, hb);
                kl = gt + 1;
                // Q(gt) once P_Q(gt-1) has read Q(gt-1)
                if (gt > 0 && !scan_wait(&bar_qfree, (gt - 1) & 1)) break;
                mbar_arrive_expect_tx(&bar_qfull, kTileBytes);
                tma_load_3d(sQ, &mQ, &bar_qfull, 0, row, hb);
                ql = gt + 1;
                // V(gt) once the intra MMA of tile gt-2 (the last reader of buffer b) is done
                if (gt > 1 && !scan_wait(&bar_vfree[b], (u & 1) ^ 1)) break;
                mbar_arrive_expect_tx(&bar_vfull[b], kTileBytes);
                tma_load_3d(sV + b * kTileBytes, &mV, &bar_vfull[b], 0, row, hb);
                vl = gt + 1;
            }
            // Drain the loads in flight before the CTA may exit (whether or not it gave up): Omega,
            // the last K and Q, the last two V (one wait site, cold code).
            volatile int never = 0;
#pragma unroll 1
            for (int i = 0; i < 5; ++i) {
                const int t = i == 1 ? kl - 1 : i == 2 ? ql - 1 : vl - 5 + i;
                if (i > 0 && t < 0) continue;
                uint64_t* bar = i == 0 ? &bar_om : i == 1 ? &bar_kfull : i == 2 ? &bar_qfull : &bar_vfull[t & 1];
                mbar_wait_lean(bar, i == 0 ? 0u : i <= 2 ? (uint32_t)(t & 1) : (uint32_t)((t >> 1) & 1), &never);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: the whole warp waits, one elected lane issues ----------------
        constexpr uint32_t id_p = idesc_bf16(128, 128, false, false);      // P = X Omega_g^T
        constexpr uint32_t id_sc = idesc_bf16(128, 128, false, false);     // SC = phi(Q) phi(K)^T
        constexpr uint32_t id_o = idesc_bf16(128, kD + 16, false, true);   // NUM += {phi(Q), A~} [.. | ..]
        constexpr uint32_t id_lo = idesc_bf16(128, kD, false, true);       // NUM += phi(Q) S_lo
        constexpr uint32_t id_st = idesc_bf16(128, kD + 16, true, true);   // [S|z] += phi(K)^T [V | 1]
        // Base descriptors; each MMA moves one on by a constant offset.
        const uint64_t d_om = sdesc_sw128(smem_u32(sOm), 16, 1024);
        const uint64_t d_q = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t d_k = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t d_snap = sdesc_sw128(smem_u32(sSnap), kOffZb - kOffSnap, 1024);
        const uint64_t d_slo = sdesc_sw128(smem_u32(sSlo), 16, 1024);
        uint64_t d_pk_sc[2], d_pk_st[2], d_v[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            d_pk_sc[b] = sdesc_sw128(smem_u32(sPK + b * kPhiBytes), 16, 1024);
            d_pk_st[b] = sdesc_sw128(smem_u32(sPK + b * kPhiBytes), 16384, 1024);
            d_v[b] = sdesc_sw128(smem_u32(sV + b * kTileBytes), (uint32_t)(sOnes - (sV + b * kTileBytes)), 1024);
        }
        const bool leader = elect_one();
#ifdef FAVOR_SCAN_TRACE
        unsigned long long wacc[10] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
#endif
        bool ok = scan_wait(&bar_om, 0);
        tc_fence_after();
        // P_K(t) into region t & 1 (once K(t) is loaded)
        auto issue_pk = [&](int t) -> bool {
            if (!TIMED_WAIT(0, scan_wait(&bar_kfull, t & 1))) return false;
            tc_fence_after();
            if (leader) {
                const uint32_t dcol = tbase + kColR0 + 128u * (uint32_t)(t & 1);
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_ss(dcol, sdesc_add(d_k, 32u * ks), sdesc_add(d_om, 32u * ks), id_p, ks > 0);
                mma_commit(&bar_pk[t & 1]);
            }
            __syncwarp();
            return true;
        };
        // P_Q(t) into region t & 1, once Q(t) is loaded and the K team has read P_K(t)
        auto issue_pq = [&](int t) -> bool {
            const int b = t & 1;
            if (!TIMED_WAIT(1, scan_wait(&bar_qfull, t & 1))) return false;
            if (!TIMED_WAIT(2, scan_wait(&bar_pkfree[b], (t >> 1) & 1))) return false;
            tc_fence_after();
            if (leader) {
                const uint32_t dcol = tbase + kColR0 + 128u * (uint32_t)b;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_ss(dcol, sdesc_add(d_q, 32u * ks), sdesc_add(d_om, 32u * ks), id_p, ks > 0);
                mma_commit(&bar_pq[b]);
                mma_commit(&bar_qfree);
            }
            __syncwarp();
            return true;
        };
        // t: this CTA's tile sequence over its heads (phases and buffers); the state restarts at
        // each head's first tile. Iterations -2 and -1 issue only the first projections (P_K(0);
        // P_Q(0), P_K(1)), so that each stage has one copy of its code.
        for (int t = -2, tl = 0; t < GT && ok; ++t) {
            const int b = t & 1, u = t >> 1;
            const bool head_start = tl == 0;
            const uint32_t R = tbase + kColR0 + 128u * (uint32_t)b;
            const uint32_t pq = tbase + kColPQ;
            const uint32_t num = tbase + kColNum;
            if (t >= 0) {
                // scores: SC = phi(Q_t) phi(K_t)^T (K = 128 features, two K atoms of phi(K))
                SCAN_TRACE(t, 20);
                ok = TIMED_WAIT(3, scan_wait(&bar_scr[b], u & 1));
                if (!ok) break;
                SCAN_TRACE(t, 0);
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts(R, pq + 8u * ks, sdesc_add(d_pk_sc[b], (ks >> 2) * 16384u + (ks & 3) * 32u), id_sc, ks > 0);
                    mma_commit(&bar_sc);
                }
                __syncwarp();
                // inter: NUM = phi(Q_t) [S_<t | z_<t] (K = 128 features), plus phi(Q_t) S_lo; none at
                // a head's first tile (S_<0 = 0), whose intra MMA starts NUM. Waited for all the
                // same: NUM must have been drained.
                SCAN_TRACE(t, 21);
                ok = TIMED_WAIT(5, scan_wait(&bar_inter, t & 1));
                if (!ok) break;
                SCAN_TRACE(t, 1);
                tc_fence_after();
                if (leader && !head_start) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) mma_ts(num, pq + 8u * ks, sdesc_add(d_snap, 2048u * ks), id_o, ks > 0);
                    if (hilo) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) mma_ts(num, pq + 8u * ks, sdesc_add(d_slo, 2048u * ks), id_lo, 1u);
                    }
                }
                __syncwarp();
            }
            // the next tile's query projection (phi(Q_t) has been read by now, in MMA order), so
            // that phi(Q_{t+1}) is formed while this tile's state and intra MMAs run
            if (t >= -1 && t + 1 < GT && !(ok = issue_pq(t + 1))) break;
            if (t >= 0) {
                SCAN_TRACE(t, 2);
                // state: [S | z] += phi(K_t)^T [V_t | 1] (K = 128 tokens; phi(K) read MN-major, its
                // second 64-feature region LBO bytes on; the ones are the second N region of B)
                if (!(ok = TIMED_WAIT(7, scan_wait(&bar_vfull[b], u & 1)))) break;
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss(tbase + kColS, sdesc_add(d_pk_st[b], 2048u * ks), sdesc_add(d_v[b], 2048u * ks), id_st,
                               (!head_start || ks > 0) ? 1u : 0u);
                    mma_commit(&bar_st);
                    mma_commit(&bar_phkfree[b]);
                }
                __syncwarp();
                SCAN_TRACE(t, 3);
                // intra: NUM += A~ [V_t | 1] (K = 128 keys, A~ packed in place of the scores)
                SCAN_TRACE(t, 22);
                if (!(ok = TIMED_WAIT(8, scan_wait(&bar_atil, t & 1)))) break;
                SCAN_TRACE(t, 4);
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts(num, R + 8u * ks, sdesc_add(d_v[b], 2048u * ks), id_o, (!head_start || ks > 0) ? 1u : 0u);
                    mma_commit(&bar_num);
                    mma_commit(&bar_vfree[b]);
                }
                __syncwarp();
                if (++tl == T) tl = 0;
                if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&s_beat[0]) = (uint32_t)t + 1u;
            }
            if (t + 2 < GT && !(ok = issue_pk(t + 2))) break;
            if (t >= 0) SCAN_TRACE(t, 5);
        }
#ifdef FAVOR_SCAN_TRACE
        if (lane == 0 && blockIdx.x < 2048)
            for (int i = 0; i < 10; ++i) g_scan_cta_wait[blockIdx.x][i] = wacc[i];
#endif
        // Every MMA issued (all of them, or those before a wait gave up) completes before TMEM is
        // released.
        if (leader) mma_commit(&bar_drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait_lean(&bar_drain, 0, &never);
    } else if (warp < kKWarp0) {
        // ---------------- Q team: 8 warps ----------------
        const int qw = warp - kQWarp0;
        const int q = warp & 3, h = qw >> 2;  // TMEM lane quarter, feature half
        const int r = q * 32 + lane;          // token row of the tile
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int fv = min(64, max(0, p.m - feat0 - 64 * h));  // real features among this warp's 64
        bool failed = false;
        for (int t = 0; t < GT; ++t) {  // the CTA's tile sequence
            const int b = t & 1, u = t >> 1;
            failed |= !scan_wait(&bar_pq[b], u & 1);
            if (warp == kQWarp0 && lane == 0) SCAN_TRACE(t, 6);
            __syncwarp();
            tc_fence_after();
            const uint32_t pa = tbase + lane_off + kColR0 + 128u * (uint32_t)b + 64u * (uint32_t)h;
            float c = 0.f;
            if (exp_kind) {
                float mx = -INFINITY;
#pragma unroll 1
                for (int cc = 0; cc < 2; ++cc) {
                    if (32 * cc < fv) {
                        uint32_t v[32];
                        tmem_ld32(pa + 32u * cc, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(v[i]));
                    }
                }
                float* mxb = sMx + (t & 1) * 256;
                mxb[h * 128 + r] = mx;
                named_bar(1, 32 * kQWarps);
                c = A2 * fmaxf(mxb[r], mxb[128 + r]);
                if (h == 0) {
                    sCq[(t & 1) * 128 + r] = c;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_cq[t & 1]);
                }
            }
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32], w[16];
                tmem_ld32(pa + 32u * cc, v);
                tmem_ld_wait();
                features16(v, w, 32 * cc < fv, c);
                tmem_st16(tbase + lane_off + kColPQ + 32u * h + 16u * cc, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_scr[b]);
            if (warp == kQWarp0 && lane == 0) SCAN_TRACE(t, 7);
        }
        (void)failed;
    } else if (warp < kAWarp0) {
        // ---------------- K team: 4 warps ----------------
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int fv = min(128, p.m - feat0);  // real features of this CTA (64 or 128)
        const float s2 = p.scale * p.scale;
        float beta = -INFINITY;  // running key stabiliser, binary orders of magnitude
        bool failed = false;
        for (int t = 0, hd = grp, tl = 0; t < GT; ++t, seq_next(hd, tl)) {  // the CTA's tile sequence
            const int b = t & 1, u = t >> 1;
            const bool valid = tl * kTile + r < p.n;
            if (tl == 0) beta = -INFINITY;  // a new head
            float kn = 0.f;  // |k^_r|^2 / 2 in binary orders of magnitude
            if (exp_kind) {
                failed |= !scan_wait(&bar_kfull, t & 1);
                __syncwarp();
                float sa = 0.f, sb = 0.f;  // |k_r|^2 over the 8 chunks of the row, one chunk per step
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    const uint4 kv = *reinterpret_cast<const uint4*>(sK + sw128_offset(r, c));
                    tcnc::sq_acc_bf16x2(kv.x, sa, sb);
                    tcnc::sq_acc_bf16x2(kv.y, sa, sb);
                    tcnc::sq_acc_bf16x2(kv.z, sa, sb);
                    tcnc::sq_acc_bf16x2(kv.w, sa, sb);
                }
                kn = 0.5f * s2 * (sa + sb) * kLog2e;
            }
            failed |= !scan_wait(&bar_pk[b], u & 1);
            if (warp == kKWarp0 && lane == 0) SCAN_TRACE(t, 8);
            __syncwarp();
            tc_fence_after();
            if (lane == 0) mbar_arrive(&bar_kfree);  // K(t) has been read by P_K(t) and for the norms
            const uint32_t pa = tbase + lane_off + kColR0 + 128u * (uint32_t)b;
            float f = 1.f;
            if (exp_kind) {
                float mx = -INFINITY;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    if (32 * cc < fv) {
                        uint32_t v[32];
                        tmem_ld32(pa + 32u * cc, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(v[i]));
                    }
                }
                const float mj = valid ? fmaf(A2, mx, -kn) : -INFINITY;
                if (named_bar_or(2, 32 * kKWarps, mj > beta + kSlackHi)) {
                    const float wm = warp_max(mj);
                    if (lane == 0) sKmx[q] = wm;
                    named_bar(2, 32 * kKWarps);
                    const float M = fmaxf(fmaxf(sKmx[0], sKmx[1]), fmaxf(sKmx[2], sKmx[3]));
                    f = ex2(beta - M);  // 0 on the first tile (beta = -inf), when the state is still empty
                    beta = M;
                }
            } else {
                beta = 0.f;
            }
            if (exp_kind && r == 0) {  // the other families keep no stabiliser
                sBeta[t & 3] = beta;
                sF[t & 3] = f;
                mbar_arrive(&bar_beta[t & 3]);
                SCAN_TRACE(t, 9);
            }
            // phi(K_t) into buffer b once the MMAs of tile t-2 have read it
            if (t >= 2) {
                failed |= !scan_wait(&bar_phkfree[b], (u & 1) ^ 1);
                __syncwarp();
            }
            uint8_t* dst = sPK + b * kPhiBytes;
            const float ck = kn + beta;
            const uint32_t keep = valid ? 0xFFFFFFFFu : 0u;  // keys past n contribute nothing
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32], w[16];
                tmem_ld32(pa + 32u * cc, v);
                tmem_ld_wait();
                if (cc == 3) {  // P_K(t) fully read: the region may take P_Q(t)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_pkfree[b]);
                }
                features16(v, w, 32 * cc < fv, ck);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    if (FAVOR_IN_BOUNDS(dst - sPK + (cc >> 1) * 16384 + sw128_offset(r, (cc & 1) * 4 + k4) + 16 <= 2 * kPhiBytes))
                    *reinterpret_cast<uint4*>(dst + (cc >> 1) * 16384 + sw128_offset(r, (cc & 1) * 4 + k4)) =
                        make_uint4(w[4 * k4] & keep, w[4 * k4 + 1] & keep, w[4 * k4 + 2] & keep, w[4 * k4 + 3] & keep);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_scr[b]);
            if (warp == kKWarp0 && lane == 0) SCAN_TRACE(t, 10);
        }
        (void)failed;
    } else if (warp < kOWarp0) {
        // ---------------- A team: 4 warps ----------------
        const int q = warp & 3;
        const int r = q * 32 + lane;  // query row of SC; feature row of the state
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        bool failed = false;
        const bool withhold = g_favor_test_wait_ns != 0;  // test hook: never publish the first state image
        // the state image before tile 0 (zero) is in place
        __syncwarp();
        if (lane == 0 && !withhold) mbar_arrive(&bar_inter);
        for (int t = 0; t < GT; ++t) {  // the CTA's tile sequence
            failed |= !scan_wait(&bar_sc, t & 1);
            if (warp == kAWarp0 && lane == 0) SCAN_TRACE(t, 11);
            __syncwarp();
            tc_fence_after();
            const uint32_t ra = tbase + lane_off + kColR0 + 128u * (uint32_t)(t & 1);
            // keys [32 cc, 32 cc + 32) of row 32 q + lane: all after the warp's rows (cc > q), all at
            // or before them (cc < q), or across the diagonal (cc == q). Packed key j -> column j / 2;
            // chunk cc writes columns the chunks up to cc have already been read from.
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t w[16];
                if (cc > q) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) w[k] = 0u;
                } else {
                    uint32_t v[32];
                    tmem_ld32(ra + 32u * (uint32_t)cc, v);
                    tmem_ld_wait();
                    const int lim = cc < q ? 31 : lane;  // keys j <= i of the chunk
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float a0 = 2 * k <= lim ? __uint_as_float(v[2 * k]) : 0.f;
                        const float a1 = 2 * k + 1 <= lim ? __uint_as_float(v[2 * k + 1]) : 0.f;
                        w[k] = pack_bf16(a0, a1);
                    }
                }
                tmem_st16(ra + 16u * (uint32_t)cc, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_atil);
            if (warp == kAWarp0 && lane == 0) SCAN_TRACE(t, 12);
            // ---- the state image S_<t+1 once state(t) is done (rescaled if the key stabiliser rose;
            // unused if tile t + 1 starts a head, whose inter MMA is skipped)
            if (t + 1 < GT) {
                const int t1 = t + 1;
                failed |= !scan_wait(&bar_st, t & 1);
                if (exp_kind) failed |= !scan_wait(&bar_beta[t1 & 3], (t1 >> 2) & 1);
                if (warp == kAWarp0 && lane == 0) SCAN_TRACE(t, 13);
                __syncwarp();
                tc_fence_after();
                const float f = exp_kind ? sF[t1 & 3] : 1.f;
                const uint32_t sa = tbase + lane_off + kColS;
                uint32_t zr;
                tmem_ld1(sa + 64, zr);
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t v[32];
                    tmem_ld32(sa + 32u * (uint32_t)hh, v);
                    tmem_ld_wait();
                    if (f != 1.f) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tmem_st32(sa + 32u * (uint32_t)hh, v);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 o = pack8_hi(v + 8 * c);
                        if (FAVOR_IN_BOUNDS(sw128_offset(r, 4 * hh + c) + 16 <= kTileBytes))
                            *reinterpret_cast<uint4*>(sSnap + sw128_offset(r, 4 * hh + c)) = o;
                        if (hilo) {
                            const uint4 ol = make_uint4(lo_pair(v[8 * c + 0], v[8 * c + 1], o.x), lo_pair(v[8 * c + 2], v[8 * c + 3], o.y),
                                                        lo_pair(v[8 * c + 4], v[8 * c + 5], o.z), lo_pair(v[8 * c + 6], v[8 * c + 7], o.w));
                            if (FAVOR_IN_BOUNDS(sw128_offset(r, 4 * hh + c) + 16 <= kTileBytes))
                                *reinterpret_cast<uint4*>(sSlo + sw128_offset(r, 4 * hh + c)) = ol;
                        }
                    }
                }
                if (f != 1.f) {
                    zr = __float_as_uint(__uint_as_float(zr) * f);
                    tmem_st1(sa + 64, zr);
                    tmem_st_wait();
                }
                // z as bf16 hi (element 0) and lo (element 1): the two denominator columns of NUM
                const float zf = __uint_as_float(zr);
                const uint32_t zh = pack_bf16(zf, 0.f);
                *reinterpret_cast<uint32_t*>(sZb + sw128_offset(r, 0)) =
                    (zh & 0xFFFFu) | (pack_bf16(zf - __uint_as_float(zh << 16), 0.f) << 16);
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_inter);
                if (warp == kAWarp0 && lane == 0) SCAN_TRACE(t, 14);
            }
        }
        (void)failed;
    } else if (warp < kXWarp0) {
        // ---------------- O team: 4 warps ----------------
        const int q = warp & 3;
        const int r = q * 32 + lane;  // query row of NUM
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        bool failed = false;
        // The group's ring: [slot][rank][chunk][row] x 16 bytes.
        uint8_t* ring = ring_grp;
        // NUM is free for the first tile's inter MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_inter);
        for (int tt = 0, bh = grp, tl = 0; tt < GT; ++tt, seq_next(bh, tl)) {  // the CTA's tile sequence
            const int slot = tt % kRing, use = tt / kRing;
            const int i_tok = tl * kTile + r;
            // where this row's results go: the output row (alone), or its partial record in the ring
            uint8_t* rec = GROUPED ? ring + ((size_t)(slot * CS + rank) * kXChunks) * kTile * 16 + r * 16 : nullptr;
            uint4* yrow = reinterpret_cast<uint4*>(p.Y + ((size_t)bh * p.n + i_tok) * kD);
            const bool store = GROUPED || i_tok < p.n;
            // the slot's previous tile has been read by every CTA of the group
            if (GROUPED && use > 0) failed |= !scan_wait(&bar_rfree[slot], (use - 1) & 1);
            if (warp == kOWarp0 && lane == 0) SCAN_TRACE(tt, 23);
            failed |= !scan_wait(&bar_num, tt & 1);
            if (warp == kOWarp0 && lane == 0) SCAN_TRACE(tt, 15);
            __syncwarp();
            tc_fence_after();
            // NUM in two halves (the second with the denominator first); y = num / den of this CTA's
            // features. Alone, the bf16 output row; in a group, fp16 times a power-of-two scale per
            // half row (so that any bf16 value range survives), the partial row for its owner.
            const uint32_t na = tbase + lane_off + kColNum;
            float den_own = 0.f, inv_own = 0.f, big = 1.f, e_own = 0.f, sc0 = 1.f, sc1 = 1.f;
#pragma unroll 1
            for (int h = 1; h >= 0; --h) {
                uint32_t v[32];
                tmem_ld32(na + 32u * (uint32_t)h, v);
                if (h == 1) {
                    uint32_t d0, d1;
                    tmem_ld1(na + 64, d0);
                    tmem_ld1(na + 65, d1);
                    tmem_ld_wait();
                    den_own = __uint_as_float(d0) + __uint_as_float(d1);
                    // y = num / den; a den below 2^-64 (keys far below the stabiliser) is scaled by
                    // 2^64 first (num with it), so that 1 / den stays finite
                    big = den_own < 0x1p-64f ? 0x1p64f : 1.f;
                    inv_own = den_own > 0.f ? 1.f / (den_own * big) : 0.f;
                } else {
                    // the row's exponent offset: read before NUM is released, which lets the Q and
                    // K teams move on to the tiles that reuse these slots
                    if (exp_kind && GROUPED) {
                        failed |= !scan_wait(&bar_cq[tt & 1], (tt >> 1) & 1);
                        failed |= !scan_wait(&bar_beta[tt & 3], (tt >> 2) & 1);
                        e_own = sCq[(tt & 1) * 128 + r] + sBeta[tt & 3];
                    }
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_inter);  // NUM may take the next tile's inter MMA
                    if (warp == kOWarp0 && lane == 0) SCAN_TRACE(tt, 16);
                }
                // half row h: alone, the bf16 output; in a group, fp16 times a power-of-two scale 2^ex
                // with max |y| 2^-ex in [2^14, 2^15) (from the IEEE exponent field, clamped so that
                // all factors stay finite), so that fp16 keeps 11 bits of any bf16 value range
                float pw = 1.f;
                if (GROUPED) {
                    float mx = 0.f;
#pragma unroll
                    for (int k = 0; k < 32; ++k) mx = fmaxf(mx, fabsf(__uint_as_float(v[k])));
                    mx = mx * big * inv_own;
                    const int ex = mx > 0.f ? max(-60, min(113, (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127 - 14)) : 0;
                    const float scl = __uint_as_float((uint32_t)(ex + 127) << 23);
                    pw = __uint_as_float((uint32_t)(127 - ex) << 23);
                    if (h) sc1 = scl;
                    else sc0 = scl;
                }
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float y0 = __uint_as_float(v[2 * k]) * big * inv_own * pw;
                    const float y1 = __uint_as_float(v[2 * k + 1]) * big * inv_own * pw;
                    if (!GROUPED) {
                        w[k] = pack_bf16(y0, y1);
                    } else {
                        __half2 h2 = __floats2half2_rn(y0, y1);
                        w[k] = *reinterpret_cast<uint32_t*>(&h2);
                    }
                }
                if (store) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 o = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                        if (!GROUPED) {
                            if (FAVOR_IN_BOUNDS((size_t)bh * p.n + i_tok < y_rows)) yrow[4 * h + c] = o;
                        } else if (FAVOR_IN_BOUNDS((size_t)(rec - ring) + (4 * h + c) * kTile * 16 + 16 <= ring_head)) {
                            __stcg(reinterpret_cast<uint4*>(rec + (4 * h + c) * kTile * 16), o);
                        }
                    }
                }
            }
            if (GROUPED) {
                // the row's log-weight: log2(den) plus its exponent offset (-inf: no weight)
                const float l_own = den_own > 0.f ? log2_pos(den_own) + e_own : -INFINITY;
                if (FAVOR_IN_BOUNDS((size_t)(rec - ring) + 8 * kTile * 16 + 16 <= ring_head))
                __stcg(reinterpret_cast<uint4*>(rec + 8 * kTile * 16),
                       make_uint4(__float_as_uint(l_own), __float_as_uint(sc0), __float_as_uint(sc1), 0u));
                // the warp's partial rows of this tile are stored (released at CTA scope; the
                // full-signal warp releases them to the group)
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_ostore[slot]);
            }
            if (warp == kOWarp0 && lane == 0) {
                *reinterpret_cast<volatile uint32_t*>(&s_beat[1]) = (uint32_t)tt + 1u;
                SCAN_TRACE(tt, 18);
            }
        }
        (void)failed;
    } else if (warp < kSWarp0) {
        // ---------------- X team: 4 warps (groups of CS > 1 only) ----------------
        // The rows [rank RP, rank RP + rows) of each tile from the CS partial rows in the ring: a
        // row's result is sum_g w_g y_g / sum_g w_g with w_g = 2^(l_g - max l), l_g = log2(den_g) + e_g
        // (y_g = num_g / den_g as stored, times its power-of-two scale). TPR threads per row, each
        // taking 8 / TPR consecutive 16-byte chunks of it.
        if (GROUPED) {
            const int xt = threadIdx.x - 32 * kXWarp0;
            const uint8_t* ring = ring_grp;
            const int row0 = rank * RP, rows = min(RP, kTile - row0);
            bool failed = false;
            // One tile: passes of 32 rows, four threads per row with two 16-byte chunks each.
            auto combine = [&](int tc, int bh, int t) {  // tile t of head bh, the sequence's tile tc
                constexpr int NC = CSX > 0 ? CSX : kMaxCluster;  // partials past CS carry no weight
                const int slot = tc % kRing;
#pragma unroll 1
                for (int item = xt; item < rows * 4; item += 32 * kXWarps) {
                    const int row = row0 + item / 4, c0 = (item % 4) * 2;
                    const int tok = t * kTile + row;
                    if (tok >= p.n) continue;
                    uint4 meta[NC], yv[NC][2];
#pragma unroll
                    for (int g = 0; g < NC; ++g) {
                        if (g >= CS) {  // log-weight -inf
                            meta[g] = make_uint4(0xFF800000u, 0u, 0u, 0u);
                            yv[g][0] = yv[g][1] = make_uint4(0u, 0u, 0u, 0u);
                            continue;
                        }
                        const uint8_t* rec = ring + ((size_t)(slot * CS + g) * kXChunks) * kTile * 16 + row * 16;
                        if (!FAVOR_IN_BOUNDS((size_t)(rec - ring) + 8 * kTile * 16 + 16 <= ring_head)) {
                            meta[g] = make_uint4(0xFF800000u, 0u, 0u, 0u);
                            yv[g][0] = yv[g][1] = make_uint4(0u, 0u, 0u, 0u);
                            continue;
                        }
                        meta[g] = __ldcg(reinterpret_cast<const uint4*>(rec + 8 * kTile * 16));
#pragma unroll
                        for (int k = 0; k < 2; ++k) yv[g][k] = __ldcg(reinterpret_cast<const uint4*>(rec + (c0 + k) * kTile * 16));
                    }
                    float L = -INFINITY;
#pragma unroll
                    for (int g = 0; g < NC; ++g) L = fmaxf(L, __uint_as_float(meta[g].x));
                    float ws[NC], wsum = 0.f;
#pragma unroll
                    for (int g = 0; g < NC; ++g) {
                        const float w = L > -INFINITY ? ex2(__uint_as_float(meta[g].x) - L) : 0.f;  // the largest is 1
                        wsum += w;
                        ws[g] = w * __uint_as_float(c0 < 4 ? meta[g].y : meta[g].z);
                    }
                    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
                    uint4* dst = reinterpret_cast<uint4*>(p.Y + ((size_t)bh * p.n + tok) * kD + 8 * c0);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int g = 0; g < NC; ++g) {
                            const uint32_t hw[4] = {yv[g][k].x, yv[g][k].y, yv[g][k].z, yv[g][k].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 y2 = __half22float2(*reinterpret_cast<const __half2*>(&hw[e]));
                                acc[2 * e] = fmaf(ws[g], y2.x, acc[2 * e]);
                                acc[2 * e + 1] = fmaf(ws[g], y2.y, acc[2 * e + 1]);
                            }
                        }
                        if (FAVOR_IN_BOUNDS((size_t)bh * p.n + tok < y_rows && c0 + k < 8))
                        dst[k] = make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                                            pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
                    }
                }
                // the warp has consumed its loads of the slot (the free-signal warp passes that on)
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_xread[slot]);
            };
            for (int tc = 0, hd = grp, tl = 0; tc < GT; ++tc, seq_next(hd, tl)) {  // the CTA's tile sequence
                // every CTA of the group has stored its partial rows of tile tc
                failed |= !scan_wait(&bar_rfull[tc % kRing], (tc / kRing) & 1);
                if (warp == kXWarp0 && lane == 0) SCAN_TRACE(tc, 17);
                combine(tc, hd, tl);
                if (warp == kXWarp0 && lane == 0) *reinterpret_cast<volatile uint32_t*>(&s_beat[2]) = (uint32_t)tc + 1u;
                if (warp == kXWarp0 && lane == 0) SCAN_TRACE(tc, 25);
            }
            (void)failed;
        }
    } else {
        // ---------------- signal warps (groups of CS > 1 only) ----------------
        // The group's counters, kept off the teams' paths (a load from L2 per tile would sit in the
        // O team's loop). Warp kSWarp0, per tile: once the O team has stored this CTA's partial
        // rows, counts them into the slot's full counter; once the counter shows every CTA's rows,
        // lets the X team combine them. Warp kSWarp0 + 1, per tile: once the X team has read the
        // slot, counts that into its free counter; once every CTA has read it, lets the O team
        // store the tile kRing later into it. Each holds the one GPU-scope fence of its tile (the
        // teams only arrive on local barriers), and the adds are relaxed.
        if (GROUPED && lane == 0) {
            const bool full_side = warp == kSWarp0;
            uint64_t* local = full_side ? bar_ostore : bar_xread;
            uint64_t* ready = full_side ? bar_rfull : bar_rfree;
            uint32_t* counter = flags + (full_side ? 0 : kRing);
            bool failed = false;
            for (int t = 0; t < GT && !failed; ++t) {
                const int slot = t % kRing, use = t / kRing;
                failed |= !scan_wait(&local[slot], use & 1);
                fence_acq_rel_gpu();
                counter_add_relaxed(&counter[slot], 1u);
                if (!full_side && t + kRing >= GT) continue;  // no later tile takes the slot
                failed |= !counter_wait(&counter[slot], (uint32_t)(CS * (use + 1)), &s_abort);
                mbar_arrive(&ready[slot]);
            }
        } else if (warp == kSWarp0 + 1 && lane == 31) {
            // ---- the watchdog: until every other warp has left its role, watch the progress beats;
            // if none moves for the wait limit, set the abort word (all spinning waits give up)
            const uint64_t tlim = g_favor_test_wait_ns;
            const uint64_t limit = tlim ? tlim : kWaitLimitNs;
            volatile uint32_t* beat = s_beat;
            volatile uint32_t* done = &s_done;
            volatile int* abort_word = &s_abort;
            uint32_t last = beat[0] + beat[1] + beat[2];
            uint64_t t0 = globaltimer();
            while (*done < (uint32_t)(kThreads / 32 - 1)) {
                __nanosleep(1000);
                const uint32_t now_beat = beat[0] + beat[1] + beat[2];
                const uint64_t now = globaltimer();
                if (now_beat != last) {
                    last = now_beat;
                    t0 = now;
                } else if (now - t0 > limit && !*abort_word) {
                    atomicOr(&g_favor_error, kDevErrTimeout);
                    *abort_word = 1;
                }
            }
        }
    }
    // this warp's role has ended (the watchdog's warp is not counted: it waits for the others)
    if (lane == 0 && warp != kSWarp0 + 1) atomicAdd(&s_done, 1u);
    tc_fence_before();
    __syncthreads();
#ifdef FAVOR_SCAN_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 2048) {
        g_scan_cta_time[blockIdx.x][2] = clock64();
        g_scan_cta_time[blockIdx.x][3] = globaltimer();
    }
#endif
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace tcs
}  // namespace favor
