"""elu + 1 linear attention on the device against the oracle's linear form.

The feature map elu(x) + 1 (feature dimension d, no random projection, no d^(-1/4) scaling) runs
through the same kernels as the random-feature families, with the identity as the projection:
the causal tensor-core scan, the non-causal tensor-core paths (single launch and state / combine /
readout), the CUDA-core kernels (fp32, and bf16 where the tensor-core kernels do not apply), the
feature map itself and the streaming decode step. Oracle: ``oracle.attn_linear_elu``.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests.helpers import assert_close_attn, assert_close_features, device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def favor(cuda_device):
    import kernelized_linear_attention_04_b300 as favor

    return favor


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


CASES = ([(dt, causal, n, 64) for dt in ("bf16", "f32") for causal in (False, True) for n in (1, 65, 200, 1000, 1500)]
         + [(dt, causal, 300, 128) for dt in ("bf16", "f32") for causal in (False, True)])


@pytest.mark.parametrize("dtype,causal,n,d", CASES)
def test_elu_attention_small_cases(favor, dtype, causal, n, d):
    w = si.Workload("case", 2, 3, n, d, d, dtype, causal, kind="elu", seed=91 + n, omega_seed=92)
    Q, K, V, _, _ = device_inputs(w)
    fn = favor.favor_attn_causal if causal else favor.favor_attn_noncausal
    Y = fn(Q, K, V, None, kind="elu")
    assert favor.last_device_error() == 0
    ref = oracle.attn_linear_elu(_f64(Q), _f64(K), _f64(V), causal=causal)
    assert_close_attn(_f64(Y), ref, dtype, f"elu {dtype} causal={causal} n={n} d={d}")


@pytest.mark.parametrize("name", ["noncausal_bf16_B1H8n1024d64m256", "causal_bf16_B4H16n8192d64m256"])
def test_elu_at_workload_shapes(favor, name):
    """The two bf16 d = 64 workload shapes with the elu + 1 map (m = d); sampled heads."""
    w = si.WORKLOADS[name].with_(kind="elu", m=64)
    Q, K, V, _, _ = device_inputs(w)
    fn = favor.favor_attn_causal if w.causal else favor.favor_attn_noncausal
    Y = fn(Q, K, V, None, kind="elu")
    assert favor.last_device_error() == 0
    for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
        ref = oracle.attn_linear_elu(_f64(Q[b, h]), _f64(K[b, h]), _f64(V[b, h]), causal=w.causal)
        assert_close_attn(_f64(Y[b, h]), ref, "bf16", f"{name} elu head {(b, h)}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_elu_features(favor, dtype):
    w = si.Workload("case", 2, 2, 77, 64, 64, dtype, False, kind="elu", seed=93, omega_seed=94)
    Q, _, _, _, _ = device_inputs(w)
    P = favor.favor_features(Q, None, kind="elu", stab="none")
    ref = oracle.elu1_features(_f64(Q))
    assert_close_features(P.cpu().numpy(), ref, 64, f"elu features {dtype}")


def test_elu_decode_matches_causal(favor):
    """n streaming decode steps give the rows of the causal elu + 1 attention."""
    w = si.Workload("case", 1, 4, 40, 64, 64, "bf16", True, kind="elu", seed=95, omega_seed=96)
    Q, K, V, _, _ = device_inputs(w)
    state = favor.decode_state(w.B, w.H, w.d, w.d)
    ys = []
    for i in range(w.n):
        ys.append(favor.favor_decode_step(Q[:, :, i].contiguous(), K[:, :, i].contiguous(), V[:, :, i].contiguous(),
                                          None, state, kind="elu"))
    Y = torch.stack(ys, dim=2)
    assert favor.last_device_error() == 0
    ref = oracle.attn_linear_elu(_f64(Q), _f64(K), _f64(V), causal=True)
    assert_close_attn(_f64(Y), ref, "bf16", "elu decode")
