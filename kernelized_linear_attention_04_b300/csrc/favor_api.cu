// C ABI of libfavor.so (declared in include/favor.h): argument checks, workspace layout, kernel
// dispatch, launch tracing and the device error word. One translation unit holds every kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/favor.h"
#include "common.cuh"
#include "simt_kernels.cuh"
#include "tc_noncausal.cuh"
#include "tc_scan.cuh"
#include "tc_exact.cuh"
#include "tc_features.cuh"
#include "tc_fused.cuh"
#include "decode.cuh"
#include "omega.cuh"
#include "tma_host.h"

namespace favor {
namespace {

// ------------------------------------------------------------------------------------------------
// Tracing: two events around every launch while enabled.
// ------------------------------------------------------------------------------------------------
struct TraceRec {
    int kid;
    cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_recs;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pool_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void release_records() {
    for (auto& r : g_recs) {
        g_event_pool.push_back(r.a);
        g_event_pool.push_back(r.b);
    }
    g_recs.clear();
}

// Runs `launch` (which enqueues one kernel on `s`) and reports launch errors.
template <class F>
favor_status_t traced(int kid, cudaStream_t s, F&& launch) {
    bool on;
    {
        std::lock_guard<std::mutex> g(g_trace_mu);
        on = g_trace_on;
    }
    cudaEvent_t a = nullptr, b = nullptr;
    if (on) {
        std::lock_guard<std::mutex> g(g_trace_mu);
        a = pool_event();
        b = pool_event();
        if (a) cudaEventRecord(a, s);
    }
    launch();
    cudaError_t err = cudaGetLastError();
    if (on && a && b) {
        cudaEventRecord(b, s);
        std::lock_guard<std::mutex> g(g_trace_mu);
        g_recs.push_back({kid, a, b});
    }
    return err == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

#define FAVOR_TRY(expr)                       \
    do {                                      \
        favor_status_t _st = (expr);          \
        if (_st != FAVOR_OK) return _st;      \
    } while (0)

// ------------------------------------------------------------------------------------------------
// Argument checks and workspace layout
// ------------------------------------------------------------------------------------------------
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

favor_status_t check_shape(int B, int H, int n, int d, int m, favor_dtype_t dt, favor_kind_t kind) {
    if (B < 0 || H < 0 || n < 0) return FAVOR_ERR_INVALID_ARG;
    if (dt != FAVOR_F32 && dt != FAVOR_BF16) return FAVOR_ERR_INVALID_ARG;
    if (kind != FAVOR_EXP && kind != FAVOR_RELU && kind != FAVOR_ELU) return FAVOR_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FAVOR_ERR_UNSUPPORTED;
    if (m < 64 || m > 512 || m % 64 != 0) return FAVOR_ERR_UNSUPPORTED;
    if (kind == FAVOR_ELU && m != d) return FAVOR_ERR_UNSUPPORTED;  // elu + 1: feature dimension d
    return FAVOR_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Head-count limits of the launches: B*H heads index gridDim.y of the feature-map and non-causal
// kernels (at most 65535), and gridDim.x (with up to 4 CTAs per head) everywhere else.
constexpr int64_t kMaxHeadsGridY = 65535;
constexpr int64_t kMaxHeads = int64_t(1) << 24;
bool heads_ok(int B, int H, int64_t limit) { return (int64_t)B * H <= limit; }

constexpr int kMaxSplits = 64;

// Token splits of the non-causal state pass: enough CTAs to fill the GPU about twice, at least
// 64 tokens per split.
int noncausal_splits(int B, int H, int n, int m) {
    int64_t heads = (int64_t)B * H * (m / simt::kSlice);
    int64_t want = (2 * 148 + heads - 1) / (heads > 0 ? heads : 1);
    int64_t cap = (n + 63) / 64;
    int64_t s = want < cap ? want : cap;
    if (s < 1) s = 1;
    if (s > kMaxSplits) s = kMaxSplits;
    return (int)s;
}

struct NoncausalWs {
    int splits;
    size_t off_pS, off_pz, off_pst, off_S, off_z, total;
};

NoncausalWs noncausal_ws(int B, int H, int n, int d, int m) {
    NoncausalWs w{};
    const size_t BH = (size_t)B * H;
    w.splits = noncausal_splits(B, H, n, m);
    size_t o = 0;
    w.off_pS = o; o = align_up(o + BH * w.splits * m * d * sizeof(float), 256);
    w.off_pz = o; o = align_up(o + BH * w.splits * m * sizeof(float), 256);
    w.off_pst = o; o = align_up(o + BH * w.splits * (m / simt::kSlice) * sizeof(float), 256);
    w.off_S = o; o = align_up(o + BH * m * d * sizeof(float), 256);
    w.off_z = o; o = align_up(o + BH * m * sizeof(float), 256);
    w.total = o;
    return w;
}

// ---- tensor-core non-causal path (bf16) ----------------------------------------------------------
constexpr int kNumSMs = 148;

int m_padded(int m) { return (m + 127) / 128 * 128; }

// The tensor-core kernels take bf16 with d = 64 (m up to 512) or d = 128 (m up to 256); the
// readout's shared memory holds Omega and the S image, which bounds m at d = 128.
bool tc_noncausal_ok(int d, int m, favor_dtype_t dt) {
    return dt == FAVOR_BF16 && (d == 64 || m_padded(m) <= 256);
}

struct TcNcWs {
    int splits, tokens_per_split, chunks, tiles_per_cta, m_pad;
    size_t off_pS, off_pz, off_pst, off_img, off_z, total;
};

// One CTA per SM (each holds all 512 TMEM columns): about one wave of (head, split) CTAs.
TcNcWs tc_noncausal_ws(int B, int H, int n, int d, int m) {
    TcNcWs w{};
    const int64_t BH = (int64_t)B * H;
    const int tiles = (n + tcnc::kTile - 1) / tcnc::kTile;
    int64_t want = std::max<int64_t>(1, kNumSMs / std::max<int64_t>(BH, 1));
    w.splits = (int)std::max<int64_t>(1, std::min<int64_t>(want, tiles));
    const int tps = (tiles + w.splits - 1) / w.splits;
    w.tokens_per_split = tps * tcnc::kTile;
    w.splits = (tiles + tps - 1) / tps;  // every split owns at least one token
    w.chunks = w.splits;
    w.tiles_per_cta = tps;
    w.m_pad = m_padded(m);
    size_t o = 0;
    w.off_pS = o; o = align_up(o + (size_t)BH * w.splits * w.m_pad * d * sizeof(float), 256);
    w.off_pz = o; o = align_up(o + (size_t)BH * w.splits * w.m_pad * sizeof(float), 256);
    w.off_pst = o; o = align_up(o + (size_t)BH * w.splits * sizeof(float), 256);
    w.off_img = o; o = align_up(o + (size_t)BH * w.m_pad * d * 2, 256);
    w.off_z = o; o = align_up(o + (size_t)BH * w.m_pad * sizeof(float), 256);
    w.total = o;
    return w;
}

// Short sequences (one cluster of at most 8 tiles per head) run as a single fused launch.
bool tc_fused_ok(int n, int d, int m, favor_dtype_t dt) {
    return dt == FAVOR_BF16 && d == 64 && m_padded(m) <= 256 && n >= 1 && n <= tcfu::kMaxCluster * tcfu::kTile;
}

size_t noncausal_ws_bytes(int B, int H, int n, int d, int m, favor_dtype_t dt) {
    if (tc_fused_ok(n, d, m, dt))
        return tcfu::fused_ws_bytes(B * H, (n + tcfu::kTile - 1) / tcfu::kTile, m_padded(m));
    return tc_noncausal_ok(d, m, dt) ? tc_noncausal_ws(B, H, n, d, m).total : noncausal_ws(B, H, n, d, m).total;
}

// The tensor-core causal scan takes bf16 with d = 64 and m <= 512: one 128-feature group per CTA, a
// cluster of ceil(m / 128) CTAs per head.
bool tc_causal_ok(int d, int m, favor_dtype_t dt) { return dt == FAVOR_BF16 && d == 64 && m_padded(m) <= 512; }
// With a cluster, the ring of partial rows the CTAs of a head combine through (L2-resident).
size_t tc_causal_ws_bytes(int B, int H, int m) { return tcs::ScanWs::bytes((size_t)B * H, m_padded(m) / 128); }

size_t causal_ws_bytes(int B, int H, int d, int m) {
    const size_t BH = (size_t)B * H;
    return align_up(BH * m * d * sizeof(float), 256) + align_up(BH * m * sizeof(float), 256);
}

size_t features_ws_bytes(int B, int H, favor_kind_t kind, favor_stab_t stab) {
    if (kind != FAVOR_EXP || stab != FAVOR_STAB_HEAD) return 0;
    return align_up((size_t)B * H * sizeof(unsigned), 256);
}

float qk_scale(int d) { return (float)std::pow((double)d, -0.25); }
// Scale applied to the projections: d^-1/4 for the random-feature families; the elu + 1 family
// works on the raw q and k.
float feat_scale(int d, int kind) { return kind == kKindElu ? 1.f : qk_scale(d); }

template <class Kern>
favor_status_t set_smem(Kern k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess
               ? FAVOR_OK
               : FAVOR_ERR_CUDA;
}

// ------------------------------------------------------------------------------------------------
// SIMT launchers
// ------------------------------------------------------------------------------------------------
template <typename T, int D>
favor_status_t simt_features(const void* X, const void* Om, float* Phi, int B, int H, int n, int m, int kind,
                             float eps, int stab, void* ws, cudaStream_t s) {
    using namespace simt;
    const int BH = B * H;
    unsigned* head_max = static_cast<unsigned*>(ws);
    if (kind == kKindExp && stab == kStabHead) {
        if (cudaMemsetAsync(head_max, 0, sizeof(unsigned) * BH, s) != cudaSuccess) return FAVOR_ERR_CUDA;
    }
    size_t smem = sizeof(float) * (kTok * D + kOmChunk * (D + 1) + kTok * m + kTok);
    auto kern = features_kernel<T, D>;
    FAVOR_TRY(set_smem(kern, smem));
    dim3 grid((n + kTok - 1) / kTok, BH);
    FAVOR_TRY(traced(FAVOR_KERNEL_FEATURES, s, [&] {
        kern<<<grid, kThreads, smem, s>>>(static_cast<const T*>(X), static_cast<const T*>(Om), Phi, n, m, kind, eps,
                                          stab, feat_scale(D, kind), head_max);
    }));
    if (kind == kKindExp && stab == kStabHead) {
        int64_t per_head = (int64_t)n * m;
        int bx = (int)std::min<int64_t>((per_head + 255) / 256, 1024);
        FAVOR_TRY(traced(FAVOR_KERNEL_FEATURES_HEAD, s, [&] {
            features_head_apply_kernel<<<dim3(bx, BH), 256, 0, s>>>(Phi, per_head, m, head_max);
        }));
    }
    return FAVOR_OK;
}

template <typename T, int D>
favor_status_t simt_noncausal(const void* Q, const void* K, const void* V, const void* Om, void* Y, int B, int H,
                              int n, int m, int kind, float eps, void* ws, cudaStream_t s) {
    using namespace simt;
    const int BH = B * H;
    NoncausalWs w = noncausal_ws(B, H, n, D, m);
    char* base = static_cast<char*>(ws);
    float* pS = reinterpret_cast<float*>(base + w.off_pS);
    float* pz = reinterpret_cast<float*>(base + w.off_pz);
    float* pst = reinterpret_cast<float*>(base + w.off_pst);
    float* S = reinterpret_cast<float*>(base + w.off_S);
    float* z = reinterpret_cast<float*>(base + w.off_z);
    int64_t tps = ((int64_t)n + w.splits - 1) / w.splits;
    tps = (tps + kTok - 1) / kTok * kTok;
    int splits = (int)((n + tps - 1) / tps);  // every split owns at least one token
    const float sc = feat_scale(D, kind);

    size_t smem_state = sizeof(float) * (2 * kTok * D + kOmChunk * (D + 1) + kTok * kSlice + kTok + 8);
    auto kstate = state_kernel<T, D>;
    FAVOR_TRY(set_smem(kstate, smem_state));
    FAVOR_TRY(traced(FAVOR_KERNEL_STATE, s, [&] {
        kstate<<<dim3(splits, BH, m / kSlice), kThreads, smem_state, s>>>(
            static_cast<const T*>(K), static_cast<const T*>(V), static_cast<const T*>(Om), n, m, kind, eps, sc, tps,
            pS, pz, pst);
    }));
    FAVOR_TRY(traced(FAVOR_KERNEL_COMBINE, s, [&] {
        combine_kernel<D><<<dim3(BH, (m * D + kCombineChunk - 1) / kCombineChunk), kThreads, 0, s>>>(pS, pz, pst, splits,
                                                                                              m, S, z);
    }));
    size_t smem_read = sizeof(float) * (kTok * D + kOmChunk * (D + 1) + kTok * m + 2 * kTok);
    auto kread = readout_kernel<T, D>;
    FAVOR_TRY(set_smem(kread, smem_read));
    FAVOR_TRY(traced(FAVOR_KERNEL_READOUT, s, [&] {
        kread<<<dim3((n + kTok - 1) / kTok, BH), kThreads, smem_read, s>>>(
            static_cast<const T*>(Q), static_cast<const T*>(Om), S, z, static_cast<T*>(Y), n, m, kind, eps, sc);
    }));
    return FAVOR_OK;
}

template <typename T, int D>
favor_status_t simt_causal(const void* Q, const void* K, const void* V, const void* Om, void* Y, int B, int H, int n,
                           int m, int kind, float eps, void* ws, cudaStream_t s) {
    using namespace simt;
    const int BH = B * H;
    float* Sg = static_cast<float*>(ws);
    float* zg = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up((size_t)BH * m * D * sizeof(float), 256));
    size_t smem = sizeof(float) * (3 * kTok * D + 2 * kTok * m + kTok * kTok + 2 * kTok + kOmChunk * (D + 1) + 8);
    auto kern = causal_kernel<T, D>;
    FAVOR_TRY(set_smem(kern, smem));
    FAVOR_TRY(traced(FAVOR_KERNEL_CAUSAL, s, [&] {
        kern<<<BH, kThreads, smem, s>>>(static_cast<const T*>(Q), static_cast<const T*>(K), static_cast<const T*>(V),
                                        static_cast<const T*>(Om), static_cast<T*>(Y), n, m, kind, eps, feat_scale(D, kind), Sg,
                                        zg);
    }));
    return FAVOR_OK;
}

favor_status_t tc_fused(const void* Q, const void* K, const void* V, const void* Om, void* Y, int B, int H, int n, int m,
                        int kind, float eps, void* ws, cudaStream_t s) {
    const int BH = B * H;
    CUtensorMap mQ, mK, mV, mOm;
    if (!tma::encode_bf16_3d(&mQ, Q, 64, n, BH, 64, tcfu::kTile) || !tma::encode_bf16_3d(&mK, K, 64, n, BH, 64, tcfu::kTile) ||
        !tma::encode_bf16_3d(&mV, V, 64, n, BH, 64, tcfu::kTile) || !tma::encode_bf16_2d(&mOm, Om, 64, m, 64, 128))
        return FAVOR_ERR_CUDA;
    const int m_pad = m_padded(m);
    const int T = (n + tcfu::kTile - 1) / tcfu::kTile;
    char* base = static_cast<char*>(ws);
    float4* Pp = reinterpret_cast<float4*>(base);
    base += tcfu::fused_ws_part(tcfu::fused_ws_pp_bytes(BH, T, m_pad));
    float* Zp = reinterpret_cast<float*>(base);
    base += tcfu::fused_ws_part((size_t)BH * T * 2 * m_pad * 4);
    float* Stab = reinterpret_cast<float*>(base);
    tcfu::FusedParams fp{n,  m,  m_pad, kind, eps * std::sqrt((float)m), feat_scale(64, kind), static_cast<__nv_bfloat16*>(Y),
                         Pp, Zp, Stab};
    const size_t smem = tcfu::FusedSmem::bytes(m_pad);
    // one instance per feature family (each carries only its own feature map)
    auto kfused = kind == kKindExp ? tcfu::nc_fused_small<kKindExp> : kind == kKindRelu ? tcfu::nc_fused_small<kKindRelu> : tcfu::nc_fused_small<kKindElu>;
    FAVOR_TRY(set_smem(kfused, smem));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(BH * T, 1, 1);
    cfg.blockDim = dim3(tcfu::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t lerr = cudaSuccess;
    FAVOR_TRY(traced(FAVOR_KERNEL_FUSED, s, [&] { lerr = cudaLaunchKernelEx(&cfg, kfused, mQ, mK, mV, mOm, fp); }));
    return lerr == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

template <int D>
favor_status_t tc_noncausal(const void* Q, const void* K, const void* V, const void* Om, void* Y, int B, int H, int n,
                            int m, int kind, float eps, void* ws, cudaStream_t s) {
    const int BH = B * H;
    const TcNcWs w = tc_noncausal_ws(B, H, n, D, m);
    char* base = static_cast<char*>(ws);
    float* pS = reinterpret_cast<float*>(base + w.off_pS);
    float* pz = reinterpret_cast<float*>(base + w.off_pz);
    float* pst = reinterpret_cast<float*>(base + w.off_pst);
    uint8_t* img = reinterpret_cast<uint8_t*>(base + w.off_img);
    float* zf = reinterpret_cast<float*>(base + w.off_z);
    CUtensorMap mK, mV, mQ, mOm;
    if (!tma::encode_bf16_3d(&mK, K, D, n, BH, 64, tcnc::kTile) || !tma::encode_bf16_3d(&mV, V, D, n, BH, 64, tcnc::kTile) ||
        !tma::encode_bf16_3d(&mQ, Q, D, n, BH, 64, tcnc::kTile) || !tma::encode_bf16_2d(&mOm, Om, D, m, 64, 128))
        return FAVOR_ERR_CUDA;
    const float sc = feat_scale(D, kind);
    const float eps_s = eps * std::sqrt((float)m);
    const int groups = w.m_pad / 128;

    tcnc::StateParams sp{n, m, w.m_pad, groups, w.tokens_per_split, kind, eps_s, sc, pS, pz, pst};
    const size_t smem_state = tcnc::StateSmem<D>::bytes(groups);
    auto kstate = kind == kKindExp ? tcnc::nc_state_tc<D, kKindExp> : kind == kKindRelu ? tcnc::nc_state_tc<D, kKindRelu> : tcnc::nc_state_tc<D, kKindElu>;
    FAVOR_TRY(set_smem(kstate, smem_state));
    FAVOR_TRY(traced(FAVOR_KERNEL_STATE, s, [&] {
        kstate<<<dim3(w.splits, BH, 1), tcnc::kStateThreads, smem_state, s>>>(mK, mV, mOm, sp);
    }));
    // The combine and the readout are launched with programmatic stream serialisation: each may
    // start (and run its independent prologue) while its predecessor finishes, and waits for it with
    // griddepcontrol.wait before reading its output.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    const int rows_per_block = 128 / (D / 8);
    cudaLaunchConfig_t cc = {};
    cc.gridDim = dim3(w.m_pad / rows_per_block, BH, 1);
    cc.blockDim = dim3(128, 1, 1);
    cc.stream = s;
    cc.attrs = pdl;
    cc.numAttrs = 1;
    cudaError_t lerr = cudaSuccess;
    FAVOR_TRY(traced(FAVOR_KERNEL_COMBINE, s, [&] {
        lerr = cudaLaunchKernelEx(&cc, tcnc::nc_combine<D>, (const float*)pS, (const float*)pz, (const float*)pst,
                                  w.splits, 1, m, w.m_pad, w.m_pad, img, zf);
    }));
    if (lerr != cudaSuccess) return FAVOR_ERR_CUDA;
    tcnc::ReadoutParams rp{n, w.m_pad, m, w.tiles_per_cta, kind, eps_s, sc, img, zf, static_cast<__nv_bfloat16*>(Y)};
    const size_t smem_read = tcnc::ReadoutSmem<D>::bytes(w.m_pad);
    auto kread = kind == kKindExp ? tcnc::nc_readout_tc<D, kKindExp> : kind == kKindRelu ? tcnc::nc_readout_tc<D, kKindRelu> : tcnc::nc_readout_tc<D, kKindElu>;
    FAVOR_TRY(set_smem(kread, smem_read));
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3(w.chunks, BH, 1);
    rc.blockDim = dim3(tcnc::kThreads, 1, 1);
    rc.dynamicSmemBytes = smem_read;
    rc.stream = s;
    rc.attrs = pdl;
    rc.numAttrs = 1;
    FAVOR_TRY(traced(FAVOR_KERNEL_READOUT, s, [&] { lerr = cudaLaunchKernelEx(&rc, kread, mQ, mOm, rp); }));
    return lerr == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

// SMs of the current device (cached per device ordinal; 0 on failure).
int sm_count() {
    constexpr int kDevices = 64;
    static std::atomic<int> cache[kDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0 && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) cache[dev].store(v);
    return v;
}

// The causal scan as a persistent grid: G groups of cs CTAs (one per SM at most), group g taking
// the heads g, g + G, ...; with cs > 1 the groups' CTAs signal each other through counters in the
// workspace, so the launch is cooperative (all CTAs resident together) and the counters are
// cleared first.
favor_status_t tc_causal(const void* Q, const void* K, const void* V, const void* Om, void* Y, int B, int H, int n,
                         int m, int kind, float eps, void* ws, cudaStream_t s) {
    const int BH = B * H;
    const int cs = m_padded(m) / 128;
    const int sms = sm_count();
    if (sms < cs) return FAVOR_ERR_CUDA;
    const int G = std::min(tcs::ScanWs::max_groups((size_t)BH, cs), sms / cs);
    CUtensorMap mQ, mK, mV, mOm;
    if (!tma::encode_bf16_3d(&mQ, Q, 64, n, BH, 64, tcs::kTile) || !tma::encode_bf16_3d(&mK, K, 64, n, BH, 64, tcs::kTile) ||
        !tma::encode_bf16_3d(&mV, V, 64, n, BH, 64, tcs::kTile) || !tma::encode_bf16_2d(&mOm, Om, 64, m, 64, 128))
        return FAVOR_ERR_CUDA;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    uint32_t* flags = cs > 1 ? reinterpret_cast<uint32_t*>(wsb) : nullptr;
    uint8_t* ring = cs > 1 ? wsb + tcs::ScanWs::flag_bytes((size_t)BH, cs) : nullptr;
    tcs::ScanParams sp{n, m, kind, eps * std::sqrt((float)m), feat_scale(64, kind), static_cast<__nv_bfloat16*>(Y),
                       BH, cs, ring, flags};
    const size_t smem = tcs::ScanSmem::bytes();
    using ScanKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, tcs::ScanParams);
    // the instance for 4 CTAs per group reads CS from the parameters (CSX = 0)
    static const ScanKernel kScan[3][4] = {
        {tcs::causal_scan<kKindExp, 1>, tcs::causal_scan<kKindExp, 2>, tcs::causal_scan<kKindExp, 3>, tcs::causal_scan<kKindExp, 0>},
        {tcs::causal_scan<kKindRelu, 1>, tcs::causal_scan<kKindRelu, 2>, tcs::causal_scan<kKindRelu, 3>, tcs::causal_scan<kKindRelu, 0>},
        {tcs::causal_scan<kKindElu, 1>, tcs::causal_scan<kKindElu, 2>, tcs::causal_scan<kKindElu, 3>, tcs::causal_scan<kKindElu, 0>}};
    const int ki = kind == kKindExp ? 0 : kind == kKindRelu ? 1 : 2;
    if (cs < 1 || cs > tcs::kMaxCluster) return FAVOR_ERR_UNSUPPORTED;
    const ScanKernel kern = kScan[ki][cs - 1];
    FAVOR_TRY(set_smem(kern, smem));
    if (cs > 1 && cudaMemsetAsync(flags, 0, (size_t)G * tcs::kFlagWords * 4, s) != cudaSuccess) return FAVOR_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cs > 1 ? 1 : 0;
    cfg.stream = s;
    cfg.gridDim = dim3(G * cs, 1, 1);
    cfg.blockDim = dim3(tcs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaError_t lerr = cudaSuccess;
    FAVOR_TRY(traced(FAVOR_KERNEL_CAUSAL, s, [&] { lerr = cudaLaunchKernelEx(&cfg, kern, mQ, mK, mV, mOm, sp); }));
    return lerr == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

template <int D>
favor_status_t tc_features(const void* X, const void* Om, float* Phi, int B, int H, int n, int m, int kind, float eps,
                           int stab, void* ws, cudaStream_t s) {
    const int BH = B * H;
    CUtensorMap mX, mOm;
    if (!tma::encode_bf16_3d(&mX, X, D, n, BH, 64, tcf::kTile) || !tma::encode_bf16_2d(&mOm, Om, D, m, 64, 128))
        return FAVOR_ERR_CUDA;
    const int m_pad = m_padded(m);
    const int tiles = (n + tcf::kTile - 1) / tcf::kTile;
    const int chunks = std::max(1, std::min(tiles, (kNumSMs + BH - 1) / std::max(BH, 1)));
    const int tpc = (tiles + chunks - 1) / chunks;
    const int grid_x = (tiles + tpc - 1) / tpc;
    unsigned* head_max = static_cast<unsigned*>(ws);
    tcf::FeatParams fp{n, m, m_pad, tpc, kind, stab, 0, eps, feat_scale(D, kind), Phi, head_max};
    const size_t smem = tcf::FeatSmem<D>::bytes(m_pad);
    auto kern = tcf::features_tc<D>;
    FAVOR_TRY(set_smem(kern, smem));
    if (kind == kKindExp && stab == kStabHead) {
        if (cudaMemsetAsync(head_max, 0, sizeof(unsigned) * BH, s) != cudaSuccess) return FAVOR_ERR_CUDA;
        tcf::FeatParams fm = fp;
        fm.max_only = 1;
        FAVOR_TRY(traced(FAVOR_KERNEL_FEATURES_HEAD, s, [&] {
            kern<<<dim3(grid_x, BH), tcf::kThreads, smem, s>>>(mX, mOm, fm);
        }));
    }
    FAVOR_TRY(traced(FAVOR_KERNEL_FEATURES, s, [&] {
        kern<<<dim3(grid_x, BH), tcf::kThreads, smem, s>>>(mX, mOm, fp);
    }));
    return FAVOR_OK;
}

// dtype x d dispatch
#define FAVOR_DISPATCH(dt, d, FN, ...)                                                     \
    ((dt) == FAVOR_F32 ? ((d) == 64 ? FN<float, 64>(__VA_ARGS__) : FN<float, 128>(__VA_ARGS__)) \
                       : ((d) == 64 ? FN<__nv_bfloat16, 64>(__VA_ARGS__) : FN<__nv_bfloat16, 128>(__VA_ARGS__)))

favor_status_t check_attn_args(const void* Q, const void* K, const void* V, const void* Om, const void* Y, int B,
                               int H, int n, int d, int m, favor_dtype_t dt, favor_kind_t kind, float eps) {
    FAVOR_TRY(check_shape(B, H, n, d, m, dt, kind));
    if (!(eps >= 0.f) || !std::isfinite(eps)) return FAVOR_ERR_INVALID_ARG;
    if ((int64_t)B * H * n == 0) return FAVOR_OK;
    if (!Q || !K || !V || !Y || (!Om && kind != FAVOR_ELU)) return FAVOR_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(Om, 16) || !aligned(Y, 16))
        return FAVOR_ERR_MISALIGNED;
    return FAVOR_OK;
}

// The projection of the elu + 1 family is the identity (m = d): the tensor-core kernels run their
// projection MMA on it (exact: one nonzero product per output) and the CUDA-core kernels their
// dot products. One copy per dtype and head size, built at compile time.
template <typename E, int D>
struct Eye {
    E v[D * D];
};
template <typename E, int D>
constexpr Eye<E, D> make_eye(E one) {
    Eye<E, D> e{};
    for (int i = 0; i < D; ++i) e.v[i * D + i] = one;
    return e;
}
__device__ const Eye<uint16_t, 64> g_eye_bf16_64 = make_eye<uint16_t, 64>(0x3F80u);  // bf16 1.0
__device__ const Eye<uint16_t, 128> g_eye_bf16_128 = make_eye<uint16_t, 128>(0x3F80u);
__device__ const Eye<float, 64> g_eye_f32_64 = make_eye<float, 64>(1.f);
__device__ const Eye<float, 128> g_eye_f32_128 = make_eye<float, 128>(1.f);

// Device addresses of the library's __device__ arrays, cached per (device, slot) together with the
// context they were looked up in: after a device reset (or any teardown of the primary context) the
// current context differs and the address is looked up again instead of being reused stale.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CUcontext current_context() {
    static CtxGetCurrentFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<CtxGetCurrentFn>(p)
                   : nullptr;
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}
struct SymbolCache {
    CUcontext ctx;
    void* addr;
};
constexpr int kSymDevices = 64, kSymSlots = 5;  // slots 0-3: identities; 4: the no-alloc scratch
std::mutex g_sym_mu;
SymbolCache g_sym[kSymDevices][kSymSlots] = {};
template <typename Sym>
void* symbol_address(const Sym& symbol, int slot) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSymDevices) return nullptr;
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> g(g_sym_mu);
    SymbolCache& e = g_sym[dev][slot];
    if (!e.addr || e.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
        e.addr = p;
        e.ctx = ctx;
    }
    return e.addr;
}

// Device address of the identity of head size d in dtype dt on the current device (cached per device
// and context); nullptr on failure.
const void* eye_ptr(int d, favor_dtype_t dt) {
    const int k = (dt == FAVOR_BF16 ? 0 : 2) + (d == 128 ? 1 : 0);
    return k == 0   ? symbol_address(g_eye_bf16_64, 0)
           : k == 1 ? symbol_address(g_eye_bf16_128, 1)
           : k == 2 ? symbol_address(g_eye_f32_64, 2)
                    : symbol_address(g_eye_f32_128, 3);
}

favor_status_t check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (need == 0) return FAVOR_OK;
    if (!ws) return FAVOR_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return FAVOR_ERR_MISALIGNED;
    if (ws_bytes < need) return FAVOR_ERR_WORKSPACE;
    return FAVOR_OK;
}

}  // namespace
}  // namespace favor

using namespace favor;

extern "C" {

int favor_abi_version(void) { return FAVOR_ABI_VERSION; }

const char* favor_status_string(favor_status_t st) {
    switch (st) {
        case FAVOR_OK: return "FAVOR_OK";
        case FAVOR_ERR_INVALID_ARG: return "FAVOR_ERR_INVALID_ARG: null pointer, negative size or bad enum";
        case FAVOR_ERR_UNSUPPORTED: return "FAVOR_ERR_UNSUPPORTED: d must be 64 or 128, m a multiple of 64 in [64, 512]";
        case FAVOR_ERR_MISALIGNED: return "FAVOR_ERR_MISALIGNED: pointers need 16-byte (workspace 256-byte) alignment";
        case FAVOR_ERR_WORKSPACE: return "FAVOR_ERR_WORKSPACE: workspace smaller than favor_workspace_bytes()";
        case FAVOR_ERR_CUDA: return "FAVOR_ERR_CUDA: CUDA call or kernel launch failed";
        case FAVOR_ERR_TIMEOUT: return "FAVOR_ERR_TIMEOUT: a device-side bounded wait gave up";
        case FAVOR_ERR_BOUNDS: return "FAVOR_ERR_BOUNDS: a device-side index check of a debug build failed";
    }
    return "unknown favor_status_t";
}

const char* favor_kernel_name(int kid) {
    switch (kid) {
        case FAVOR_KERNEL_FEATURES: return "features";
        case FAVOR_KERNEL_FEATURES_HEAD: return "features_head_stab";
        case FAVOR_KERNEL_STATE: return "state";
        case FAVOR_KERNEL_COMBINE: return "combine";
        case FAVOR_KERNEL_READOUT: return "readout";
        case FAVOR_KERNEL_CAUSAL: return "causal";
        case FAVOR_KERNEL_DECODE: return "decode";
        case FAVOR_KERNEL_DECODE_INIT: return "decode_init";
        case FAVOR_KERNEL_OMEGA: return "omega";
        case FAVOR_KERNEL_FUSED: return "fused";
        case FAVOR_KERNEL_EXACT: return "exact";
    }
    return "unknown";
}

size_t favor_workspace_bytes(favor_op_t op, int B, int H, int n, int d, int m, favor_dtype_t dt, favor_kind_t kind,
                             favor_stab_t stab, int chunk) {
    if (check_shape(B, H, n, d, m, dt, kind) != FAVOR_OK) return (size_t)-1;
    if ((int64_t)B * H * n == 0) return 0;
    if (!heads_ok(B, H, op == FAVOR_OP_CAUSAL ? kMaxHeads : kMaxHeadsGridY)) return (size_t)-1;
    switch (op) {
        case FAVOR_OP_FEATURES: return features_ws_bytes(B, H, kind, stab);
        case FAVOR_OP_NONCAUSAL: return noncausal_ws_bytes(B, H, n, d, m, dt);
        case FAVOR_OP_CAUSAL:
            if (chunk != 0 && chunk != 64 && chunk != 128) return (size_t)-1;
            return tc_causal_ok(d, m, dt) ? tc_causal_ws_bytes(B, H, m) : causal_ws_bytes(B, H, d, m);
    }
    return (size_t)-1;
}

favor_status_t favor_features(const void* X, const void* Omega, float* Phi, int B, int H, int n, int d, int m,
                              favor_dtype_t dt, favor_kind_t kind, float relu_eps, favor_stab_t stab, void* workspace,
                              size_t ws_bytes, void* stream) {
    FAVOR_TRY(check_shape(B, H, n, d, m, dt, kind));
    if (stab != FAVOR_STAB_NONE && stab != FAVOR_STAB_ROW && stab != FAVOR_STAB_HEAD) return FAVOR_ERR_INVALID_ARG;
    if (!(relu_eps >= 0.f) || !std::isfinite(relu_eps)) return FAVOR_ERR_INVALID_ARG;
    if ((int64_t)B * H * n == 0) return FAVOR_OK;
    if (!heads_ok(B, H, kMaxHeadsGridY)) return FAVOR_ERR_UNSUPPORTED;
    if (!X || !Phi || (!Omega && kind != FAVOR_ELU)) return FAVOR_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Omega, 16) || !aligned(Phi, 16)) return FAVOR_ERR_MISALIGNED;
    FAVOR_TRY(check_ws(workspace, ws_bytes, features_ws_bytes(B, H, kind, stab)));
    if (kind == FAVOR_ELU && !(Omega = eye_ptr(d, dt))) return FAVOR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == FAVOR_BF16)
        return d == 64 ? tc_features<64>(X, Omega, Phi, B, H, n, m, (int)kind, relu_eps, (int)stab, workspace, s)
                       : tc_features<128>(X, Omega, Phi, B, H, n, m, (int)kind, relu_eps, (int)stab, workspace, s);
    return FAVOR_DISPATCH(dt, d, simt_features, X, Omega, Phi, B, H, n, m, (int)kind, relu_eps, (int)stab, workspace,
                          s);
}

favor_status_t favor_attn_noncausal(const void* Q, const void* K, const void* V, const void* Omega, void* Y, int B,
                                    int H, int n, int d, int m, favor_dtype_t dt, favor_kind_t kind, float relu_eps,
                                    void* workspace, size_t ws_bytes, void* stream) {
    FAVOR_TRY(check_attn_args(Q, K, V, Omega, Y, B, H, n, d, m, dt, kind, relu_eps));
    if ((int64_t)B * H * n == 0) return FAVOR_OK;
    if (!heads_ok(B, H, kMaxHeadsGridY)) return FAVOR_ERR_UNSUPPORTED;
    FAVOR_TRY(check_ws(workspace, ws_bytes, noncausal_ws_bytes(B, H, n, d, m, dt)));
    if (kind == FAVOR_ELU && !(Omega = eye_ptr(d, dt))) return FAVOR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tc_fused_ok(n, d, m, dt)) return tc_fused(Q, K, V, Omega, Y, B, H, n, m, (int)kind, relu_eps, workspace, s);
    if (tc_noncausal_ok(d, m, dt))
        return d == 64 ? tc_noncausal<64>(Q, K, V, Omega, Y, B, H, n, m, (int)kind, relu_eps, workspace, s)
                       : tc_noncausal<128>(Q, K, V, Omega, Y, B, H, n, m, (int)kind, relu_eps, workspace, s);
    return FAVOR_DISPATCH(dt, d, simt_noncausal, Q, K, V, Omega, Y, B, H, n, m, (int)kind, relu_eps, workspace, s);
}

favor_status_t favor_attn_causal(const void* Q, const void* K, const void* V, const void* Omega, void* Y, int B,
                                 int H, int n, int d, int m, int chunk, favor_dtype_t dt, favor_kind_t kind,
                                 float relu_eps, void* workspace, size_t ws_bytes, void* stream) {
    FAVOR_TRY(check_attn_args(Q, K, V, Omega, Y, B, H, n, d, m, dt, kind, relu_eps));
    if (chunk != 0 && chunk != 64 && chunk != 128) return FAVOR_ERR_UNSUPPORTED;
    if ((int64_t)B * H * n == 0) return FAVOR_OK;
    if (!heads_ok(B, H, kMaxHeads)) return FAVOR_ERR_UNSUPPORTED;
    if (kind == FAVOR_ELU && !(Omega = eye_ptr(d, dt))) return FAVOR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tc_causal_ok(d, m, dt)) {
        FAVOR_TRY(check_ws(workspace, ws_bytes, tc_causal_ws_bytes(B, H, m)));
        return tc_causal(Q, K, V, Omega, Y, B, H, n, m, (int)kind, relu_eps, workspace, s);
    }
    FAVOR_TRY(check_ws(workspace, ws_bytes, causal_ws_bytes(B, H, d, m)));
    return FAVOR_DISPATCH(dt, d, simt_causal, Q, K, V, Omega, Y, B, H, n, m, (int)kind, relu_eps, workspace, s);
}

// ------------------------------------------------------------------------------------------------
// favor_attn_noncausal_noalloc: the non-causal path with its scratch in a fixed device array.
// ------------------------------------------------------------------------------------------------
}  // extern "C"

namespace favor {
namespace {

// ---- streaming decode state: S [BH][m][d], z [BH][m], stab [BH][m/64], partials [BH][m/64][d+2]
// (fp32), counter [BH] (u32) ---------------------------------------------------------------------
struct DecodeLayout {
    size_t off_z, off_stab, off_part, off_cnt, total;
};
DecodeLayout decode_layout(int B, int H, int d, int m) {
    const size_t BH = (size_t)B * H, nb = (size_t)m / dec::kBlk;
    DecodeLayout L{};
    L.off_z = align_up(BH * m * d * sizeof(float), 256);
    L.off_stab = L.off_z + align_up(BH * m * sizeof(float), 256);
    L.off_part = L.off_stab + align_up(BH * nb * sizeof(float), 256);
    L.off_cnt = L.off_part + align_up(BH * nb * (d + 2) * sizeof(float), 256);
    L.total = L.off_cnt + align_up(BH * sizeof(unsigned), 256);
    return L;
}

favor_status_t check_decode_state(const void* state, size_t state_bytes, int B, int H, int d, int m) {
    if (!state) return FAVOR_ERR_INVALID_ARG;
    if (!aligned(state, 256)) return FAVOR_ERR_MISALIGNED;
    if (state_bytes < decode_layout(B, H, d, m).total) return FAVOR_ERR_WORKSPACE;
    return FAVOR_OK;
}

template <typename T, int D>
favor_status_t decode_launch(const void* q, const void* k, const void* v, const void* Om, void* y, void* state, int BH,
                             int m, int kind, float eps, cudaStream_t s) {
    const DecodeLayout L = decode_layout(BH, 1, D, m);
    char* base = static_cast<char*>(state);
    const size_t smem = sizeof(float) * dec::decode_smem_floats<D>();
    FAVOR_TRY(traced(FAVOR_KERNEL_DECODE, s, [&] {
        dec::decode_step<T, D><<<dim3(BH, m / dec::kBlk), dec::kThreads, smem, s>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), static_cast<const T*>(Om),
            static_cast<T*>(y), reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + L.off_z),
            reinterpret_cast<float*>(base + L.off_stab), reinterpret_cast<float*>(base + L.off_part),
            reinterpret_cast<unsigned*>(base + L.off_cnt), m, kind, eps * std::sqrt((float)m), feat_scale(D, kind));
    }));
    return cudaGetLastError() == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

template <typename T, int D>
favor_status_t omega_launch(uint64_t seed, int m, bool orthogonal, void* Om, cudaStream_t s) {
    const size_t smem = omg::omega_smem_bytes<D>();
    FAVOR_TRY(set_smem(omg::omega_build<T, D>, smem));
    const int blocks = (m + D - 1) / D;
    FAVOR_TRY(traced(FAVOR_KERNEL_OMEGA, s, [&] {
        omg::omega_build<T, D><<<blocks, omg::kThreads, smem, s>>>(omg::stream_key(seed, omg::kStreamGauss),
                                                                    omg::stream_key(seed, omg::kStreamChi), m,
                                                                    orthogonal ? 1 : 0, static_cast<T*>(Om));
    }));
    return cudaGetLastError() == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

}  // namespace
}  // namespace favor

extern "C" {

size_t favor_decode_state_bytes(int B, int H, int d, int m) {
    if (check_shape(B, H, 1, d, m, FAVOR_BF16, FAVOR_EXP) != FAVOR_OK) return SIZE_MAX;
    if (!heads_ok(B, H, kMaxHeads)) return SIZE_MAX;
    return decode_layout(B, H, d, m).total;
}

favor_status_t favor_decode_init(void* state, size_t state_bytes, int B, int H, int d, int m, void* stream) {
    FAVOR_TRY(check_shape(B, H, 1, d, m, FAVOR_BF16, FAVOR_EXP));
    if ((int64_t)B * H == 0) return FAVOR_OK;
    if (!heads_ok(B, H, kMaxHeads)) return FAVOR_ERR_UNSUPPORTED;
    FAVOR_TRY(check_decode_state(state, state_bytes, B, H, d, m));
    const DecodeLayout L = decode_layout(B, H, d, m);
    char* base = static_cast<char*>(state);
    const int64_t BH = (int64_t)B * H;
    const int64_t nS = BH * m * d;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int blocks = (int)std::min<int64_t>((nS + 255) / 256, 4 * kNumSMs);
    FAVOR_TRY(traced(FAVOR_KERNEL_DECODE_INIT, s, [&] {
        dec::decode_init<<<blocks, 256, 0, s>>>(reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + L.off_z),
                                               reinterpret_cast<float*>(base + L.off_stab),
                                               reinterpret_cast<unsigned*>(base + L.off_cnt), nS, BH * m,
                                               BH * (m / dec::kBlk), BH);
    }));
    return cudaGetLastError() == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

favor_status_t favor_decode_step(const void* q, const void* k, const void* v, const void* Omega, void* y, void* state,
                                 size_t state_bytes, int B, int H, int d, int m, favor_dtype_t dt, favor_kind_t kind,
                                 float relu_eps, void* stream) {
    FAVOR_TRY(check_attn_args(q, k, v, Omega, y, B, H, 1, d, m, dt, kind, relu_eps));
    if ((int64_t)B * H == 0) return FAVOR_OK;
    if (!heads_ok(B, H, kMaxHeads)) return FAVOR_ERR_UNSUPPORTED;
    FAVOR_TRY(check_decode_state(state, state_bytes, B, H, d, m));
    if (kind == FAVOR_ELU && !(Omega = eye_ptr(d, dt))) return FAVOR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return FAVOR_DISPATCH(dt, d, decode_launch, q, k, v, Omega, y, state, B * H, m, (int)kind, relu_eps, s);
}

favor_status_t favor_omega(uint64_t seed, int m, int d, int orthogonal, favor_dtype_t dt, void* Omega, void* stream) {
    if (m < 0 || (dt != FAVOR_F32 && dt != FAVOR_BF16)) return FAVOR_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FAVOR_ERR_UNSUPPORTED;
    if (m == 0) return FAVOR_OK;
    if (!Omega) return FAVOR_ERR_INVALID_ARG;
    if (!aligned(Omega, 16)) return FAVOR_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return FAVOR_DISPATCH(dt, d, omega_launch, seed, m, orthogonal != 0, Omega, s);
}

}  // extern "C"

namespace favor {
namespace {

// In host code this name is only a host-side stand-in: kernels get the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FAVOR_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device (cached per device and context).
favor_status_t noalloc_scratch(void** out) {
    void* p = symbol_address(g_noalloc_scratch, 4);
    if (!p) return FAVOR_ERR_CUDA;
    *out = p;
    return FAVOR_OK;
}

}  // namespace
}  // namespace favor

extern "C" {

favor_status_t favor_attn_noncausal_noalloc(const void* Q, const void* K, const void* V, const void* Omega, void* Y,
                                            int B, int H, int n, int d, int m, favor_dtype_t dt, favor_kind_t kind,
                                            float relu_eps, void* stream) {
    FAVOR_TRY(check_attn_args(Q, K, V, Omega, Y, B, H, n, d, m, dt, kind, relu_eps));
    if ((int64_t)B * H * n == 0) return FAVOR_OK;
    if (!heads_ok(B, H, kMaxHeadsGridY)) return FAVOR_ERR_UNSUPPORTED;
    const size_t need = favor_workspace_bytes(FAVOR_OP_NONCAUSAL, B, H, n, d, m, dt, kind, FAVOR_STAB_NONE, 0);
    if (need > FAVOR_NOALLOC_SCRATCH_BYTES) return FAVOR_ERR_WORKSPACE;
    void* scratch = nullptr;
    FAVOR_TRY(noalloc_scratch(&scratch));
    return favor_attn_noncausal(Q, K, V, Omega, Y, B, H, n, d, m, dt, kind, relu_eps, scratch,
                                FAVOR_NOALLOC_SCRATCH_BYTES, stream);
}

favor_status_t favor_last_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FAVOR_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_favor_error, sizeof(v)) != cudaSuccess) return FAVOR_ERR_CUDA;
    if (v == 0) return FAVOR_OK;
    unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_favor_error, &zero, sizeof(zero)) != cudaSuccess) return FAVOR_ERR_CUDA;
    return (v & kDevErrBounds) ? FAVOR_ERR_BOUNDS : FAVOR_ERR_TIMEOUT;
}

favor_status_t favor_softmax_attn(const void* Q, const void* K, const void* V, void* Y, int B, int H, int n, int d,
                                  int causal, favor_dtype_t dt, void* stream) {
    if (B < 0 || H < 0 || n < 0 || (dt != FAVOR_F32 && dt != FAVOR_BF16)) return FAVOR_ERR_INVALID_ARG;
    if (dt != FAVOR_BF16 || d != 64) return FAVOR_ERR_UNSUPPORTED;
    if ((int64_t)B * H * n == 0) return FAVOR_OK;
    if (!heads_ok(B, H, kMaxHeadsGridY)) return FAVOR_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !Y) return FAVOR_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(Y, 16)) return FAVOR_ERR_MISALIGNED;
    const int BH = B * H;
    CUtensorMap mQ, mK, mV;
    if (!tma::encode_bf16_3d(&mQ, Q, 64, n, BH, 64, tce::kTile) || !tma::encode_bf16_3d(&mK, K, 64, n, BH, 64, tce::kTile) ||
        !tma::encode_bf16_3d(&mV, V, 64, n, BH, 64, tce::kTile))
        return FAVOR_ERR_CUDA;
    tce::ExactParams ep{n, causal ? 1 : 0, kLog2e / std::sqrt((float)d), static_cast<__nv_bfloat16*>(Y)};
    const size_t smem = tce::ExactSmem::bytes();
    FAVOR_TRY(set_smem(tce::exact_attn, smem));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid((n + tce::kTile - 1) / tce::kTile, BH);
    FAVOR_TRY(traced(FAVOR_KERNEL_EXACT, s, [&] { tce::exact_attn<<<grid, tce::kThreads, smem, s>>>(mQ, mK, mV, ep); }));
    return FAVOR_OK;
}

favor_status_t favor_test_set_wait_limit(unsigned long long ns, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyToSymbolAsync(g_favor_test_wait_ns, &ns, sizeof(ns), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return FAVOR_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

favor_status_t favor_trace_enable(int on) {
    std::lock_guard<std::mutex> g(g_trace_mu);
    if (on) release_records();
    g_trace_on = on != 0;
    return FAVOR_OK;
}

favor_status_t favor_trace_read(int* launches, double* total_ms) {
    if (!launches || !total_ms) return FAVOR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(g_trace_mu);
    for (int k = 0; k < FAVOR_KERNEL_COUNT; ++k) {
        launches[k] = 0;
        total_ms[k] = 0.0;
    }
    for (auto& r : g_recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return FAVOR_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return FAVOR_ERR_CUDA;
        launches[r.kid] += 1;
        total_ms[r.kid] += ms;
    }
    return FAVOR_OK;
}

}  // extern "C"
