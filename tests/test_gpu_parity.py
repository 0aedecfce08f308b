"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs.

Small cases are compared element by element on every output; the five full-size workloads run in
the launch configuration the benchmark times and are compared on every output of sampled heads
(heads are independent, so a sampled head is checked exactly).
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests.helpers import (assert_close_attn, assert_close_features, device_inputs, head_f64, to_device,
                           torch_dtype)

pytestmark = pytest.mark.gpu

WL = si.WORKLOADS
ORDER = si.workloads.WORKLOAD_ORDER


@pytest.fixture(scope="module")
def favor(cuda_device):
    import kernelized_linear_attention_04_b300 as favor

    return favor


def small(name, **kw):
    return WL[name].with_(**kw)


def run_attn(favor, w, Q, K, V, Om):
    if w.causal:
        return favor.favor_attn_causal(Q, K, V, Om, chunk=w.chunk, kind=w.kind, relu_eps=w.relu_eps)
    return favor.favor_attn_noncausal(Q, K, V, Om, kind=w.kind, relu_eps=w.relu_eps)


def oracle_attn(w, Q, K, V, om64):
    fn = oracle.attn_causal if w.causal else oracle.attn_noncausal
    return fn(Q, K, V, om64, kind=w.kind, relu_eps=w.relu_eps)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------------------------------------
# Small and ragged cases: every output element
# ---------------------------------------------------------------------------------------------

CASES = []
for dtype in ("f32", "bf16"):
    for causal in (False, True):
        for kind in ("exp", "relu"):
            for n in (1, 3, 63, 65, 127, 129, 1000):
                CASES.append((dtype, causal, kind, n, 64, 256))
        for d, m in ((128, 256), (64, 64), (64, 512), (128, 192), (64, 192), (64, 384)):
            CASES.append((dtype, causal, "exp", 200, d, m))


@pytest.mark.parametrize("dtype,causal,kind,n,d,m", CASES)
def test_attention_small_cases(favor, dtype, causal, kind, n, d, m):
    w = si.Workload("case", 2, 3, n, d, m, dtype, causal, kind=kind, seed=77 + n, omega_seed=5 + m)
    Q, K, V, Om, om64 = device_inputs(w)
    Y = run_attn(favor, w, Q, K, V, Om)
    assert favor.last_device_error() == 0
    ref = oracle_attn(w, f64(Q), f64(K), f64(V), om64)
    assert_close_attn(f64(Y), ref, dtype, f"{dtype} causal={causal} {kind} n={n} d={d} m={m}")


# Every feature-group count of the causal tensor-core scan (clusters of 1 to 4 CTAs, the last one
# partly padding when m is not a multiple of 128) and every non-causal tensor-core path: the fused
# single launch (n <= 1024, d = 64), the state / combine / readout kernels beyond it (ReLU and exp,
# d = 64 and 128), and the CUDA-core kernels bf16 falls back to at d = 128 with m > 256.
SCAN_CASES = [(kind, n, m) for kind in ("exp", "relu") for m in (64, 128, 192, 256, 320, 384, 448, 512)
              for n in (130, 515)]


@pytest.mark.parametrize("kind,n,m", SCAN_CASES)
def test_causal_scan_feature_groups(favor, kind, n, m):
    w = si.Workload("case", 1, 3, n, 64, m, "bf16", True, kind=kind, seed=31 + n + m, omega_seed=7 + m)
    Q, K, V, Om, om64 = device_inputs(w)
    Y = run_attn(favor, w, Q, K, V, Om)
    assert favor.last_device_error() == 0
    ref = oracle_attn(w, f64(Q), f64(K), f64(V), om64)
    assert_close_attn(f64(Y), ref, "bf16", f"causal {kind} n={n} m={m}")


# The scan runs a persistent grid: G = min(heads, SMs // CS) groups of CS = ceil(m / 128) CTAs,
# group g taking heads g, g + G, ... one after another, the state, the key stabiliser and NUM
# restarting at each head's first tile. Heads past the first round (and the first and last heads)
# against the oracle, for every family and group size.
ROUND_CASES = [("exp", 512, 300), ("relu", 512, 300), ("exp", 384, 130), ("relu", 256, 300),
               ("exp", 128, 130), ("elu", 64, 200)]


@pytest.mark.parametrize("kind,m,n", ROUND_CASES)
def test_causal_scan_heads_over_rounds(favor, kind, m, n):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cs = -(-m // 128)
    groups = sms // cs
    H = groups + 3  # three groups take a second head
    w = si.Workload("case", 1, H, n, 64, m, "bf16", True, kind=kind, seed=91 + m, omega_seed=13 + m)
    Q, K, V, Om, om64 = device_inputs(w)
    Y = run_attn(favor, w, Q, K, V, Om)
    assert favor.last_device_error() == 0
    heads = [0, 1, groups - 1, groups, groups + 1, H - 1]
    if kind == "elu":  # elu + 1 features of the raw q, k (no Omega)
        ref = oracle.attn_linear_elu(f64(Q[0, heads]), f64(K[0, heads]), f64(V[0, heads]), causal=True)
    else:
        ref = oracle_attn(w, f64(Q[0, heads]), f64(K[0, heads]), f64(V[0, heads]), om64)
    for i, h in enumerate(heads):
        assert_close_attn(f64(Y[0, h]), ref[i], "bf16", f"causal {kind} m={m} n={n} head {h} of {H}")


NONCAUSAL_PATH_CASES = (
    [("relu", n, d, m) for n in (1025, 1500, 4099) for d in (64, 128) for m in (128, 256)]
    + [("exp", n, 64, 256) for n in (1025, 4096)]
    + [("exp", 700, 128, m) for m in (320, 384, 448, 512)]
    + [("relu", 700, 128, 512)]
)


@pytest.mark.parametrize("kind,n,d,m", NONCAUSAL_PATH_CASES)
def test_noncausal_paths(favor, kind, n, d, m):
    w = si.Workload("case", 1, 2, n, d, m, "bf16", False, kind=kind, seed=41 + n + d, omega_seed=9 + m)
    Q, K, V, Om, om64 = device_inputs(w)
    Y = run_attn(favor, w, Q, K, V, Om)
    assert favor.last_device_error() == 0
    ref = oracle_attn(w, f64(Q), f64(K), f64(V), om64)
    assert_close_attn(f64(Y), ref, "bf16", f"non-causal {kind} n={n} d={d} m={m}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [200, 1500])
def test_large_norm_inputs_stay_finite(favor, causal, n):
    """Queries and keys five times the workloads' scale (|q| about 40 at d = 64): every exponent
    stabiliser must follow the real largest exponent, not a norm bound far above it, or all of a
    row's features underflow and num / den becomes 0 / 0."""
    w = si.Workload("case", 1, 2, n, 64, 256, "bf16", causal, seed=57 + n, omega_seed=58)
    Q, K, V, Om, om64 = device_inputs(w)
    Q5 = (Q.float() * 5).to(Q.dtype).contiguous()
    K5 = (K.float() * 5).to(K.dtype).contiguous()
    Y = run_attn(favor, w, Q5, K5, V, Om)
    assert favor.last_device_error() == 0
    assert torch.isfinite(Y.float()).all()
    ref = oracle_attn(w, f64(Q5), f64(K5), f64(V), om64)
    assert_close_attn(f64(Y), ref, "bf16", f"x5 inputs causal={causal} n={n}")


@pytest.mark.parametrize("n,d,m,dtype", [(1000, 64, 256, "bf16"), (3000, 64, 256, "bf16"), (3000, 128, 256, "bf16"),
                                         (700, 128, 512, "bf16"), (700, 64, 256, "f32")])
def test_noncausal_on_poisoned_workspace(favor, n, d, m, dtype):
    """The caller's workspace holds NaN before the call (fused, three-kernel and CUDA-core paths):
    nothing in it may be read before the call itself has written it."""
    w = si.Workload("case", 1, 3, n, d, m, dtype, False, seed=71 + n, omega_seed=72)
    Q, K, V, Om, om64 = device_inputs(w)
    nb = favor.workspace_bytes("noncausal", w.B, w.H, n, d, m, torch_dtype(w))
    ws = torch.full((max(nb, 4) // 4,), float("nan"), dtype=torch.float32, device=Q.device)
    Y = favor.favor_attn_noncausal(Q, K, V, Om, workspace=ws.view(torch.uint8))
    assert favor.last_device_error() == 0
    ref = oracle_attn(w, f64(Q), f64(K), f64(V), om64)
    assert_close_attn(f64(Y), ref, dtype, f"poisoned workspace n={n} d={d} m={m} {dtype}")


@pytest.mark.parametrize("causal", [False, True])
def test_grid_limit_heads(favor, causal):
    """B*H = 65535 heads (the largest count the non-causal calls take) of one token each."""
    w = si.Workload("case", 1, 65535, 1, 64, 64, "bf16", causal, seed=61, omega_seed=62)
    Q, K, V, Om, om64 = device_inputs(w)
    Y = run_attn(favor, w, Q, K, V, Om)
    assert favor.last_device_error() == 0
    ref = oracle_attn(w, f64(Q), f64(K), f64(V), om64)
    assert_close_attn(f64(Y), ref, "bf16", f"65535 heads causal={causal}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind,stab", [("exp", "row"), ("exp", "head"), ("exp", "none"), ("relu", "row")])
@pytest.mark.parametrize("n,d,m", [(1, 64, 64), (77, 64, 256), (300, 128, 256), (129, 64, 512)])
def test_features_small_cases(favor, dtype, kind, stab, n, d, m):
    w = si.Workload("case", 2, 2, n, d, m, dtype, False, kind=kind, seed=9 + n, omega_seed=3 + d)
    Q, _, _, Om, om64 = device_inputs(w)
    P = favor.favor_features(Q, Om, kind=kind, relu_eps=w.relu_eps, stab=stab)
    assert favor.last_device_error() == 0
    ref = oracle.features(f64(Q), om64, kind=kind, relu_eps=w.relu_eps, stab=stab)
    assert_close_features(P.cpu().numpy(), ref, m, f"{dtype} {kind} {stab} n={n}")


# ---------------------------------------------------------------------------------------------
# Degenerate cases with closed forms, determinism, stabiliser growth, empty input
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identical_keys_and_constant_values(favor, causal, dtype):
    w = si.Workload("case", 1, 2, 300, 64, 128, dtype, causal, seed=1, omega_seed=2)
    Q, K, V, Om, om64 = device_inputs(w)
    K1 = K[:, :, :1].expand_as(K).contiguous()
    Y = run_attn(favor, w, Q, K1, V, Om)
    Vf = f64(V)
    if causal:
        expect = np.cumsum(Vf, axis=2) / np.arange(1, w.n + 1)[None, None, :, None]
    else:
        expect = np.broadcast_to(Vf.mean(axis=2, keepdims=True), Vf.shape)
    assert_close_attn(f64(Y), expect, dtype, "identical keys")
    c = torch.linspace(-1, 1, 64, device=V.device).to(V.dtype)
    Vc = c.expand_as(V).contiguous()
    Yc = run_attn(favor, w, Q, K, Vc, Om)
    assert_close_attn(f64(Yc), np.broadcast_to(f64(c), Vf.shape), dtype, "constant values")


@pytest.mark.parametrize("causal", [False, True])
def test_bitwise_deterministic(favor, causal):
    w = si.Workload("case", 2, 4, 2000, 64, 256, "bf16", causal, seed=3, omega_seed=4)
    Q, K, V, Om, _ = device_inputs(w)
    Y1 = run_attn(favor, w, Q, K, V, Om)
    Y2 = run_attn(favor, w, Q, K, V, Om)
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_growing_key_norms_exercise_stabiliser_rescale(favor, causal, dtype):
    """Key magnitudes grow along the sequence, so the running key stabiliser must rise many times
    (and partial states be rescaled) for the result to stay finite and match the oracle."""
    w = si.Workload("case", 1, 2, 1500, 64, 128, dtype, causal, seed=11, omega_seed=12)
    Q, K, V, Om, om64 = device_inputs(w)
    ramp = torch.linspace(0.2, 3.0, w.n, device=K.device)[None, None, :, None]
    K2 = (K.float() * ramp).to(K.dtype).contiguous()
    Y = run_attn(favor, w, Q, K2, V, Om)
    assert torch.isfinite(Y.float()).all()
    ref = oracle_attn(w, f64(Q), f64(K2), f64(V), om64)
    assert_close_attn(f64(Y), ref, dtype, "growing keys")


def test_causal_concentrated_weights(favor):
    """A seed where one key carries about 93% of a query's weight (|y| = 4.18, where a bf16 output
    step is 0.03): the carried prefix state must keep more than bf16 precision for the max-abs gate."""
    w = si.Workload("case", 2, 3, 777, 64, 256, "bf16", True, seed=17 + 777, omega_seed=13 + 256)
    Q, K, V, Om, om64 = device_inputs(w)
    Y = run_attn(favor, w, Q, K, V, Om)
    ref = oracle_attn(w, f64(Q), f64(K), f64(V), om64)
    assert abs(ref[1, 0, 166, 10]) > 4.0
    assert_close_attn(f64(Y), ref, "bf16", "concentrated weights")


def test_empty_sequence(favor):
    Q = torch.zeros(2, 3, 0, 64, device="cuda", dtype=torch.bfloat16)
    Om = torch.zeros(64, 64, device="cuda", dtype=torch.bfloat16)
    assert favor.favor_attn_noncausal(Q, Q, Q, Om).shape == Q.shape
    assert favor.favor_attn_causal(Q, Q, Q, Om).shape == Q.shape
    assert favor.favor_features(Q, Om).shape == (2, 3, 0, 64)


# ---------------------------------------------------------------------------------------------
# Full-size workloads in the benchmark's launch configuration: sampled heads
# ---------------------------------------------------------------------------------------------

SAMPLED_HEADS = {
    "noncausal_f32_B1H1n256d64m128": None,            # every head
    "noncausal_bf16_B1H8n1024d64m256": None,
    "causal_bf16_B4H16n8192d64m256": [(0, 0), (1, 7), (2, 13), (3, 15)],
    "noncausal_bf16_B1H16n65536d128m256": [(0, 0), (0, 11)],
    "causal_relu_bf16_B8H32n32768d64m512": [(0, 0), (7, 31)],
}


@pytest.mark.parametrize("name", ORDER)
def test_full_workload_sampled_heads(favor, name):
    w = WL[name]
    Q, K, V, Om, om64 = device_inputs(w)
    Y = run_attn(favor, w, Q, K, V, Om)
    assert favor.last_device_error() == 0
    heads = SAMPLED_HEADS[name] or [(b, h) for b in range(w.B) for h in range(w.H)]
    del Q, K, V
    Yh = {bh: f64(Y[bh[0], bh[1]]) for bh in heads}
    del Y
    torch.cuda.empty_cache()
    Qs = np.stack([head_f64(w, b, h)["Q"] for b, h in heads])
    Ks = np.stack([head_f64(w, b, h)["K"] for b, h in heads])
    Vs = np.stack([head_f64(w, b, h)["V"] for b, h in heads])
    ref = oracle_attn(w, Qs, Ks, Vs, om64)
    for i, bh in enumerate(heads):
        assert_close_attn(Yh[bh], ref[i], w.dtype, f"{name} head {bh}")


@pytest.mark.parametrize("name", ["noncausal_bf16_B1H8n1024d64m256", "noncausal_bf16_B1H16n65536d128m256"])
def test_full_workload_features_sampled_heads(favor, name):
    w = WL[name]
    full = si.full_inputs(w, "K")
    om_store, om64 = si.omega_for(w)
    K = to_device(full["K"], torch_dtype(w))
    Om = to_device(om_store, torch_dtype(w))
    P = favor.favor_features(K, Om, stab="head")
    for b, h in [(0, 0), (0, w.H - 1)]:
        ref = oracle.features(head_f64(w, b, h)["K"][None], om64, stab="head")[0]
        assert_close_features(P[b, h].cpu().numpy(), ref, w.m, f"{name} head {(b, h)}")
