"""Exact softmax attention on the device (the comparator of the speed and divergence sweep)
against the oracle's exact softmax(Q K^T / sqrt(d)) V, element by element."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests.helpers import BF16_MAX_ABS, BF16_REL_L2, device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def favor(cuda_device):
    import kernelized_linear_attention_04_b300 as favor

    return favor


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 5, 127, 128, 129, 300, 1024, 1500])
def test_exact_attention_matches_oracle(favor, causal, n):
    w = si.Workload("case", 2, 3, n, 64, 64, "bf16", causal, seed=101 + n, omega_seed=1)
    Q, K, V, _, _ = device_inputs(w)
    Y = favor.favor_softmax_attn(Q, K, V, causal=causal)
    assert favor.last_device_error() == 0
    ref = oracle.softmax_attention(_f64(Q), _f64(K), _f64(V), causal=causal)
    y = _f64(Y)
    assert np.isfinite(y).all()
    err = np.abs(y - ref)
    assert err.max() <= BF16_MAX_ABS, err.max()
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) <= BF16_REL_L2


def test_exact_attention_large_scores(favor):
    """Queries and keys scaled so that scores span hundreds: the online maximum must keep every
    exponential finite and one dominant key per row must come through."""
    w = si.Workload("case", 1, 2, 700, 64, 64, "bf16", False, seed=111, omega_seed=1)
    Q, K, V, _, _ = device_inputs(w)
    Q4 = (Q.float() * 4).to(Q.dtype)
    K4 = (K.float() * 4).to(K.dtype)
    Y = favor.favor_softmax_attn(Q4, K4, V)
    ref = oracle.softmax_attention(_f64(Q4), _f64(K4), _f64(V))
    y = _f64(Y)
    assert np.isfinite(y).all()
    assert np.abs(y - ref).max() <= BF16_MAX_ABS


def test_exact_attention_rejects_unsupported(favor):
    x = torch.zeros(1, 1, 8, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(favor.FavorError):
        favor.favor_softmax_attn(x, x, x)


def test_sweep_against_exact_attention(favor):
    """bench.py --sweep: one JSON object per (form, n, m) with both wall clocks and the divergence of
    FAVOR+ from the exact kernel; the divergence at n = 256 agrees with the same comparison made
    by the oracle in fp64 on the same seeded inputs (up to the bf16 rounding of both GPU outputs,
    amplified by the small norm of the exact output of diffuse attention)."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--sweep", "--sweep-n", "256,1024",
                          "--sweep-m", "64,128"], capture_output=True, text=True, timeout=600, check=True).stdout
    pts = [json.loads(line) for line in out.splitlines() if line.startswith("{")]
    assert len(pts) == 8
    assert {(p["form"], p["n"], p["m"]) for p in pts} == {(f, n, m) for f in ("noncausal", "causal")
                                                          for n in (256, 1024) for m in (64, 128)}
    for p in pts:
        assert p["favor_ms"] > 0 and p["exact_ms"] > 0 and np.isfinite(p["rel_l2"]) and p["rel_l2"] > 0
    p = next(p for p in pts if p["form"] == "noncausal" and p["n"] == 256 and p["m"] == 64)
    w = si.Workload("sweep", 1, 8, 256, 64, 64, "bf16", False, kind="exp", seed=101 + 256, omega_seed=7)
    full = si.full_inputs(w)
    q, k, v = (si.to_f64(full[t]) for t in ("Q", "K", "V"))
    _, om64 = si.omega_for(w)
    yf = oracle.attn_noncausal(q, k, v, om64, kind="exp")
    ye = oracle.softmax_attention(q, k, v)
    ref = np.linalg.norm(yf - ye) / np.linalg.norm(ye)
    assert abs(p["rel_l2"] - ref) <= 0.3 * ref, (p["rel_l2"], ref)
