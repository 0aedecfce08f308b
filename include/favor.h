/*
 * favor.h — C ABI of libfavor.so: FAVOR+ (Performer) attention forward pass on one B300 (sm_103a).
 *
 * What is computed (sources are the pages' titles and sections):
 *   x^ = d^(-1/4) x for every query and key row ("Performer" paper note, *Standard Attention Cost*:
 *   the 1/sqrt(d) of softmax(QK^T/sqrt(d)), split evenly between q and k);
 *   positive random features ("Performer" paper note, *FAVOR+*)
 *       phi_r(x) = exp(w_r^T x^ - |x^|^2/2 - stab) / sqrt(m),     r = 1..m, w_r = row r of Omega,
 *   or the generalized-ReLU family ("Performer for vision", *What Is Performer?*, Key Feature 4)
 *       phi_r(x) = max(0, w_r^T x^) / sqrt(m) + relu_eps;
 *   the state S = Phi(K)^T V (m x d) and normaliser z = Phi(K)^T 1 ("Performer" paper note,
 *   *Kernel Attention View* and *Normalization*);
 *   y_i = phi(q_i)^T S / phi(q_i)^T z, with sums over all keys (non-causal) or over keys j <= i
 *   (causal: prefix sums, "Performer for vision", *How It Works*, Step 2).
 * No n x n matrix is formed on the attention path.
 *
 * Conventions for every entry point:
 *   - Q, K, V, X and Y are contiguous row-major [B, H, n, d] device arrays of the dtype `dt`; Omega is a
 *     contiguous row-major [m, d] device array of the same dtype, shared by queries, keys and all heads.
 *     Callers pass RAW q and k: the d^(-1/4) scaling is applied inside.
 *   - All device pointers must be 16-byte aligned; workspace must be 256-byte aligned.
 *   - Supported shapes: d in {64, 128}; m a multiple of 64 with 64 <= m <= 512; n >= 0; B, H >= 0.
 *     B*H*n == 0 is a valid empty call that returns FAVOR_OK and touches no memory. Head count:
 *     B*H <= 65535 for favor_features and the non-causal calls (heads index a grid dimension of
 *     that size), B*H <= 2^24 for the causal and decode calls; larger counts return
 *     FAVOR_ERR_UNSUPPORTED (favor_workspace_bytes and favor_decode_state_bytes: SIZE_MAX).
 *   - Arithmetic: fp32 inputs are computed in fp32 on CUDA cores; bf16 inputs run on the tensor
 *     cores with fp32 accumulation (features rounded to bf16 between the two contractions).
 *   - Ownership: the caller owns every buffer. The library allocates no device memory; it keeps only
 *     small host-side caches. `workspace` is scratch owned by the caller for the duration of the
 *     call (size from favor_workspace_bytes; it may be NULL when that size is 0).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Every call is
 *     asynchronous on that stream. Argument errors are reported by the return value before anything
 *     is launched; launch failures return FAVOR_ERR_CUDA; device-side failures (a bounded wait that
 *     ran out) are recorded in a device error word read by favor_last_device_error.
 *   - Calls are deterministic: the same inputs give bit-identical outputs.
 *   - Thread safety: calls from several host threads are safe; tracing state is global.
 */
#ifndef FAVOR_H
#define FAVOR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FAVOR_ABI_VERSION 1

typedef enum {
    FAVOR_OK = 0,
    FAVOR_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum value                    */
    FAVOR_ERR_UNSUPPORTED = 2,  /* d, m or chunk outside the supported set                        */
    FAVOR_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned (workspace: 256-byte)          */
    FAVOR_ERR_WORKSPACE = 4,    /* ws_bytes smaller than favor_workspace_bytes(...)                */
    FAVOR_ERR_CUDA = 5,         /* a CUDA runtime/driver call or kernel launch failed              */
    FAVOR_ERR_TIMEOUT = 6,      /* a device-side bounded wait gave up (reported after the fact)    */
    FAVOR_ERR_BOUNDS = 7        /* debug builds only: a device-side index check failed             */
} favor_status_t;

typedef enum { FAVOR_F32 = 0, FAVOR_BF16 = 1 } favor_dtype_t;
/* Feature family:
 *   FAVOR_EXP   positive random features exp(w_r^T x^ - |x^|^2/2 - stab) ("Performer" paper note, *FAVOR+*);
 *   FAVOR_RELU  generalized ReLU max(0, w_r^T x^) + relu_eps ("Performer for vision", Key Feature 4);
 *   FAVOR_ELU   elu(x) + 1 on the raw q and k: x_r + 1 for x_r > 0, exp(x_r) otherwise, feature
 *               dimension d, no projection, no d^(-1/4) scaling (the Linear Transformer's map in the
 *               comparison table of the question page "How do linear attention variants (Performer,
 *               Linformer) achieve O(n) complexity, and what's the quality cost?"; "Performer for
 *               vision", *Kernel Choices*). Calls with this family take m == d and ignore Omega, which
 *               may be NULL; relu_eps is not used. */
typedef enum { FAVOR_EXP = 0, FAVOR_RELU = 1, FAVOR_ELU = 2 } favor_kind_t;

/* Stabiliser of favor_features (exp family only; ignored for ReLU):
 *   NONE: stab = 0;  ROW: per token, stab = max_r u_r(x);  HEAD: per (b, h), stab = max over the
 *   head's tokens j and features r of u_r(x_j), with u_r(x) = w_r^T x^ - |x^|^2/2.
 * With ROW/HEAD the largest feature of a row/head is exactly 1/sqrt(m) (up to rounding). */
typedef enum { FAVOR_STAB_NONE = 0, FAVOR_STAB_ROW = 1, FAVOR_STAB_HEAD = 2 } favor_stab_t;

typedef enum { FAVOR_OP_FEATURES = 0, FAVOR_OP_NONCAUSAL = 1, FAVOR_OP_CAUSAL = 2 } favor_op_t;

/* Bytes of workspace the given call needs (0 if none). Same arguments as the call itself; `stab`
 * and `chunk` are read only for the ops that take them. Returns (size_t)-1 for unsupported shapes. */
size_t favor_workspace_bytes(favor_op_t op, int B, int H, int n, int d, int m, favor_dtype_t dt,
                             favor_kind_t kind, favor_stab_t stab, int chunk);

/*
 * Feature map phi(X) ("Performer" paper note, *FAVOR+*; "Performer for vision", *Kernel Choices*).
 *   X     [B, H, n, d] dtype dt (raw, unscaled), Omega [m, d] dtype dt;
 *   Phi   [B, H, n, m] fp32 output;
 *   stab  see favor_stab_t (exp family); relu_eps the additive floor of the ReLU family.
 * Exists to check phi itself and for callers that compose their own contractions; the attention
 * entry points never write phi to memory.
 */
favor_status_t favor_features(const void* X, const void* Omega, float* Phi, int B, int H, int n, int d, int m,
                              favor_dtype_t dt, favor_kind_t kind, float relu_eps, favor_stab_t stab,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * Non-causal FAVOR+ attention ("Performer" paper note, *Normalization*, second equation;
 * "Performer for vision", *How It Works*, Step 1):
 *   S = Phi(K)^T V, z = Phi(K)^T 1 per (b, h); Y = Phi(Q) S / Phi(Q) z (row-wise divide).
 *   Q, K, V, Y [B, H, n, d] dtype dt; Omega [m, d] dtype dt. Y may not alias Q, K or V.
 * Stabilisers: queries use one constant per row, keys one constant per head (after rescaling of
 * partial sums); both cancel in the ratio, so Y does not depend on them.
 * bf16 with d = 64, m <= 256 and n <= 1024 runs as one launch (a head's 128-token tiles are the
 * CTAs of one thread-block cluster); other bf16 shapes with d = 64, or d = 128 and m <= 256, run a
 * key-state pass, a combine and a query readout on the tensor cores; fp32 and the remaining shapes
 * run on CUDA cores. The workspace holds the partial key states (favor_workspace_bytes).
 */
favor_status_t favor_attn_noncausal(const void* Q, const void* K, const void* V, const void* Omega, void* Y,
                                    int B, int H, int n, int d, int m, favor_dtype_t dt, favor_kind_t kind,
                                    float relu_eps, void* workspace, size_t ws_bytes, void* stream);

/*
 * Causal FAVOR+ attention ("Performer for vision", *How It Works*, Step 2: prefix sums so that
 * each token attends only to itself and earlier tokens; "Performer" paper note, *Normalization*):
 *   y_i = phi(q_i)^T S_i / phi(q_i)^T z_i,  S_i = sum_{j<=i} phi(k_j) v_j^T,  z_i = sum_{j<=i} phi(k_j).
 * Computed as a chunked scan: per chunk, an intra-chunk lower-triangular block plus the carried
 * prefix state. chunk: 0 (implementation default), 64 or 128; the result does not depend on it
 * beyond rounding. bf16 with d = 64 and m <= 512 runs a tensor-core scan, one CTA per 128-feature
 * group and a group of CS = ceil(m / 128) CTAs per head (a persistent grid of at most one CTA per
 * SM, each group taking heads in turn; launched cooperatively when CS > 1), which carries the state
 * every 128 tokens and masks j <= i inside each 128-token tile (two 64-token chunks give exactly
 * that sum); other inputs run on CUDA cores in 16-token steps. Shapes and dtypes as above.
 * Workspace (favor_workspace_bytes): 0 bytes for m <= 128; for m > 128 the CTAs of a group count
 * and exchange their partial output rows through it: for G = min(B*H, 160 / CS) groups, 64 bytes
 * of counters each (the whole rounded up to 256 bytes), then G * 4 * CS * 18432 bytes. Its
 * contents on entry do not matter (the counters are cleared on the stream before the launch). The
 * scan takes every SM of the device: a kernel running beside it on another stream delays its
 * start.
 */
favor_status_t favor_attn_causal(const void* Q, const void* K, const void* V, const void* Omega, void* Y,
                                 int B, int H, int n, int d, int m, int chunk, favor_dtype_t dt,
                                 favor_kind_t kind, float relu_eps, void* workspace, size_t ws_bytes,
                                 void* stream);

/*
 * Non-causal attention for callers that cannot allocate device memory. There is no counterpart on
 * the pages: this is a packaging variant of favor_attn_noncausal, for code that runs where
 * cudaMalloc is unavailable or forbidden (a plugin inside a host application that owns every
 * allocation, a real-time loop that must not block in the allocator, a context whose memory pool
 * is fixed at start-up).
 *
 * It computes exactly what favor_attn_noncausal computes, with the same arguments minus the
 * workspace. Its scratch (the partial key states) lives in one fixed device array of
 * FAVOR_NOALLOC_SCRATCH_BYTES compiled into the library, so every GPU that loads libfavor.so holds
 * that array until the process exits. Shapes whose scratch need (favor_workspace_bytes for
 * FAVOR_OP_NONCAUSAL) exceeds it are rejected with FAVOR_ERR_WORKSPACE before anything runs.
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current) and caches it with the current context; make that first call outside any CUDA
 * stream capture. After a device reset (or any re-creation of the context) the next call looks the
 * address up again, so that call too must be outside stream capture. The call
 * allocates nothing and frees nothing. All calls share the one array: two calls that may overlap
 * on the GPU (different streams, or several host threads) race on it and give undefined results,
 * so serialise them. The array keeps the last call's contents; nothing in it needs to start at
 * zero.
 */
#define FAVOR_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
favor_status_t favor_attn_noncausal_noalloc(const void* Q, const void* K, const void* V, const void* Omega,
                                            void* Y, int B, int H, int n, int d, int m, favor_dtype_t dt,
                                            favor_kind_t kind, float relu_eps, void* stream);

/*
 * Streaming decode ("Performer for vision", *What Is Performer?*, Key Feature 2: attention is
 * accumulated incrementally, enabling streaming inference; *Why Performer Matters*, Streaming and
 * Sampling: autoregressive decoding). The causal form one token at a time: per head a state
 * (S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j) over the tokens seen so far) lives in a
 * caller-owned device buffer, and each step appends one token and returns its output.
 *
 * favor_decode_state_bytes: size of the state for B*H heads (fp32 S [B*H][m][d], z [B*H][m], a key
 *   stabiliser per head and 64-feature block, the blocks' partial sums of the current step, and a
 *   per-head counter; 256-byte aligned pieces); SIZE_MAX for an unsupported shape (d in {64, 128},
 *   m a multiple of 64 in [64, 512]).
 * favor_decode_init: empties the state of every head (no token seen). Asynchronous on `stream`.
 * favor_decode_step: q, k, v, y are [B, H, d] (the new token of every head), Omega [m, d], all of
 *   dtype dt; state as initialised (256-byte aligned, at least favor_decode_state_bytes). Updates
 *   S <- S + phi(k) v^T, z <- z + phi(k) and writes y = phi(q)^T S / phi(q)^T z, so that steps
 *   t = 1..n give exactly the rows of favor_attn_causal over those n tokens (up to rounding).
 *   The key stabiliser is carried in the state and the accumulated S, z are rescaled when it moves;
 *   it cancels in the ratio. Errors as for the attention calls; nothing runs on an error.
 */
size_t favor_decode_state_bytes(int B, int H, int d, int m);
favor_status_t favor_decode_init(void* state, size_t state_bytes, int B, int H, int d, int m, void* stream);
favor_status_t favor_decode_step(const void* q, const void* k, const void* v, const void* Omega, void* y,
                                 void* state, size_t state_bytes, int B, int H, int d, int m, favor_dtype_t dt,
                                 favor_kind_t kind, float relu_eps, void* stream);

/*
 * Random projection Omega built on the device ("Performer for vision", *What Is Performer?*,
 * Orthogonal Features; the "Performer" paper note, FAVOR+ section: positive orthogonal random
 * features). Writes Omega [m, d] (row-major, dtype dt, 16-byte aligned, caller-owned) for `seed`:
 *   orthogonal != 0: for every block of d rows, a d x d matrix of iid N(0, 1) draws whose rows are
 *     orthonormalised in order (modified Gram-Schmidt, fp64), each row then scaled to the length of
 *     an independent N(0, I_d) vector (a chi_d sample); the last block keeps its first m mod d rows;
 *   orthogonal == 0: m rows of iid N(0, 1) draws.
 * Draws: element i of stream s of the seed is the cosine branch of Box-Muller applied to two
 * uniforms from SplitMix64's finaliser (key = splitmix64(splitmix64(seed) ^ s * 0xD1B54A32D192ED03),
 * u1 = ((splitmix64(key + 2i) >> 11) + 1) 2^-53, u2 = (splitmix64(key + 2i + 1) >> 11) 2^-53); the
 * Gaussian blocks are stream 4 (element (b d + r) d + c for row r, column c of block b), the chi
 * lengths stream 5 (elements r d .. r d + d - 1 for row r of Omega). Values are computed in fp64 and
 * rounded to fp32 (to nearest) and then, for bf16, to bf16 (to nearest even). Redrawing the features
 * is a call with a new seed. d in {64, 128}, m >= 0 (m == 0: nothing runs). Asynchronous on
 * `stream`; errors as for the attention calls.
 */
favor_status_t favor_omega(uint64_t seed, int m, int d, int orthogonal, favor_dtype_t dt, void* Omega, void* stream);

/*
 * Exact softmax attention, the operator FAVOR+ approximates ("Performer" paper note, *Standard
 * Attention Cost*: softmax(Q K^T / sqrt(d)) V, quadratic in n), for the speed and divergence
 * comparison the pages ask for ("Linear Attention and the Performer", *Exercise*). Not part of the
 * FAVOR+ path: no n x n matrix is stored (an online softmax over 128-key tiles), but the work is
 * O(n^2 d).
 *   Q, K, V, Y [B, H, n, d]; causal != 0 restricts row i to keys j <= i. bf16 with d = 64 only
 *   (other inputs: FAVOR_ERR_UNSUPPORTED); B*H <= 65535. No workspace. Asynchronous on `stream`.
 */
favor_status_t favor_softmax_attn(const void* Q, const void* K, const void* V, void* Y, int B, int H, int n, int d,
                                  int causal, favor_dtype_t dt, void* stream);

/* Human-readable name of a status code (static storage). */
const char* favor_status_string(favor_status_t status);

/* Synchronises `stream`, then reads and clears the device error word of the current device.
 * Returns FAVOR_OK, FAVOR_ERR_TIMEOUT (a bounded device wait gave up), FAVOR_ERR_BOUNDS (a debug
 * build's device-side index check failed; takes precedence) or FAVOR_ERR_CUDA. */
favor_status_t favor_last_device_error(void* stream);

/* FAVOR_ABI_VERSION of the loaded library. */
int favor_abi_version(void);

/* Test hook for the failure path (no counterpart on the pages). With ns > 0, every bounded device
 * wait of the calls that follow on the current device gives up after ns nanoseconds instead of its
 * normal limit, and the causal tensor-core scan withholds the first arrival its MMA issuer waits
 * for: that wait runs out, the kernel records FAVOR_ERR_TIMEOUT in the device error word, the
 * CTA's other roles stop, its copies in flight are drained and its tensor memory is released; the
 * output of that call is undefined. ns = 0 (the initial state) turns the hook off. Synchronises
 * `stream` after setting the word. Never needed in normal use. */
favor_status_t favor_test_set_wait_limit(unsigned long long ns, void* stream);

/* ---- tracing: per-kernel device time, recorded with CUDA events around every launch ---------- */

typedef enum {
    FAVOR_KERNEL_FEATURES = 0,      /* feature map (favor_features)                          */
    FAVOR_KERNEL_FEATURES_HEAD = 1, /* per-head stabiliser pass of favor_features            */
    FAVOR_KERNEL_STATE = 2,         /* non-causal key-side state reduction (S, z partials)   */
    FAVOR_KERNEL_COMBINE = 3,       /* non-causal combine of the partial states              */
    FAVOR_KERNEL_READOUT = 4,       /* non-causal query-side readout and divide              */
    FAVOR_KERNEL_CAUSAL = 5,        /* causal chunked scan                                    */
    FAVOR_KERNEL_FUSED = 6,         /* single-launch non-causal path for short sequences      */
    FAVOR_KERNEL_DECODE = 7,        /* streaming decode step (favor_decode_step)              */
    FAVOR_KERNEL_DECODE_INIT = 8,   /* decode state reset (favor_decode_init)                 */
    FAVOR_KERNEL_OMEGA = 9,         /* random projection builder (favor_omega)                */
    FAVOR_KERNEL_EXACT = 10,        /* exact softmax attention (favor_softmax_attn)           */
    FAVOR_KERNEL_COUNT = 11
} favor_kernel_id_t;

/* Starts (on != 0) or stops recording. Starting clears previous records. While recording, every
 * launch is bracketed by two events on its stream, which adds a little host overhead. */
favor_status_t favor_trace_enable(int on);

/* Waits for the recorded events and writes, per favor_kernel_id_t, the number of launches and the
 * summed device milliseconds (arrays of FAVOR_KERNEL_COUNT entries). Records stay until the next
 * favor_trace_enable(1). */
favor_status_t favor_trace_read(int* launches, double* total_ms);

/* Name of a kernel id (static storage). */
const char* favor_kernel_name(int kernel_id);

#ifdef __cplusplus
}
#endif

#endif /* FAVOR_H */
