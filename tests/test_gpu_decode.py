"""GPU parity of the streaming decode step.

n calls of favor_decode_step through the C ABI, one token per head each, must give the rows of the
fp64 oracle's causal recurrence over the same seeded inputs: the decode step is the causal form one
token at a time ("Performer for vision", *What Is Performer?*, Key Feature 2).
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests.helpers import assert_close_attn, device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def favor(cuda_device):
    import kernelized_linear_attention_04_b300 as favor

    return favor


def decode_all(favor, Q, K, V, Om, kind, relu_eps, state=None):
    """Y [B, H, n, d] from n decode steps (a fresh state unless one is given)."""
    B, H, n, d = Q.shape
    if state is None:
        state = favor.decode_state(B, H, d, int(Om.shape[0]))
    Y = torch.empty_like(Q)
    y = torch.empty(B, H, d, dtype=Q.dtype, device=Q.device)
    for t in range(n):
        favor.favor_decode_step(Q[:, :, t].contiguous(), K[:, :, t].contiguous(), V[:, :, t].contiguous(), Om, state,
                                kind=kind, relu_eps=relu_eps, out=y)
        Y[:, :, t] = y
    return Y


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


CASES = [(dt, kind, d, m) for dt in ("f32", "bf16") for kind in ("exp", "relu")
         for d, m in ((64, 64), (64, 256), (128, 256), (64, 512))]


@pytest.mark.parametrize("dtype,kind,d,m", CASES)
def test_decode_steps_match_oracle_causal(favor, dtype, kind, d, m):
    w = si.Workload("decode", 2, 3, 97, d, m, dtype, True, kind=kind, seed=400 + d + m, omega_seed=41 + m)
    Q, K, V, Om, om64 = device_inputs(w)
    Y = decode_all(favor, Q, K, V, Om, w.kind, w.relu_eps)
    torch.cuda.synchronize()
    assert favor.last_device_error() == 0
    ref = oracle.attn_causal(f64(Q), f64(K), f64(V), om64, kind=w.kind, relu_eps=w.relu_eps)
    assert_close_attn(f64(Y), ref, dtype, f"decode {dtype} {kind} d={d} m={m}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_stabiliser_moves_with_growing_keys(favor, dtype):
    # keys whose norms grow along the sequence raise the running key stabiliser again and again,
    # each time rescaling the accumulated state
    w = si.Workload("decode", 1, 2, 120, 64, 128, dtype, True, seed=9, omega_seed=10)
    Q, K, V, Om, om64 = device_inputs(w)
    grow = torch.linspace(0.5, 3.0, K.shape[2], device=K.device).view(1, 1, -1, 1)
    K = (K.float() * grow).to(K.dtype).contiguous()
    Y = decode_all(favor, Q, K, V, Om, "exp", w.relu_eps)
    ref = oracle.attn_causal(f64(Q), f64(K), f64(V), om64, kind="exp")
    assert_close_attn(f64(Y), ref, dtype, f"decode growing keys {dtype}")


def test_decode_init_empties_the_state(favor):
    w = si.Workload("decode", 1, 4, 40, 64, 256, "bf16", True, seed=5, omega_seed=6)
    Q, K, V, Om, _ = device_inputs(w)
    state = favor.decode_state(1, 4, 64, 256)
    decode_all(favor, Q[:, :, :25], K[:, :, :25], V[:, :, :25], Om, "exp", 1e-3, state=state)
    favor.favor_decode_init(state, 1, 4, 64, 256)
    again = decode_all(favor, Q, K, V, Om, "exp", 1e-3, state=state)
    fresh = decode_all(favor, Q, K, V, Om, "exp", 1e-3)
    assert torch.equal(again, fresh)


def test_decode_agrees_with_the_causal_scan(favor):
    w = si.Workload("decode", 2, 2, 300, 64, 256, "bf16", True, seed=77, omega_seed=78)
    Q, K, V, Om, om64 = device_inputs(w)
    Yd = decode_all(favor, Q, K, V, Om, "exp", 1e-3)
    Yc = favor.favor_attn_causal(Q, K, V, Om)
    ref = oracle.attn_causal(f64(Q), f64(K), f64(V), om64)
    assert_close_attn(f64(Yd), ref, "bf16", "decode")
    assert_close_attn(f64(Yc), ref, "bf16", "causal scan")
    assert float((Yd.float() - Yc.float()).abs().max()) <= 2e-2
