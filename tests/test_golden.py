"""The stored tiny case: oracle regression + 50-digit brute force of the explicit sums (CPU)."""
import json
import os

import mpmath
import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
G = json.load(open(os.path.join(HERE, "golden", "tiny_favor.json")))
mpmath.mp.dps = 50


def _arr(key):
    return np.array(G[key], dtype=np.float64)


def _brute(kind, causal):
    """y_i = sum_j k(q_i, k_j) v_j / sum_j k(q_i, k_j) with k(q, k) = sum_r phi_r(q) phi_r(k),
    every sum written out, in 50-digit arithmetic, no stabilisers."""
    n, d, m = G["n"], G["d"], G["m"]
    Q, K, V, W = G["Q"], G["K"], G["V"], G["Omega"]
    s = mpmath.mpf(d) ** mpmath.mpf(-0.25)

    def phi(x):
        xh = [s * mpmath.mpf(c) for c in x]
        h = sum(c * c for c in xh) / 2
        out = []
        for r in range(m):
            p = sum(mpmath.mpf(W[r][c]) * xh[c] for c in range(d))
            if kind == "exp":
                out.append(mpmath.exp(p - h) / mpmath.sqrt(m))
            else:
                out.append(max(p, 0) / mpmath.sqrt(m) + mpmath.mpf(1e-3))
        return out

    PQ = [phi(q) for q in Q]
    PK = [phi(k) for k in K]
    Y = np.zeros((n, d))
    for i in range(n):
        js = range(i + 1) if causal else range(n)
        kij = {j: sum(PQ[i][r] * PK[j][r] for r in range(m)) for j in js}
        den = sum(kij.values())
        for c in range(d):
            Y[i, c] = float(sum(kij[j] * mpmath.mpf(V[j][c]) for j in js) / den)
    return Y


@pytest.mark.parametrize("kind", ["exp", "relu"])
@pytest.mark.parametrize("causal", [False, True])
def test_golden_matches_oracle_and_brute_force(kind, causal):
    key = f"Y_{'causal' if causal else 'noncausal'}_{kind}"
    stored = _arr(key)
    Q, K, V, om = _arr("Q")[None], _arr("K")[None], _arr("V")[None], _arr("Omega")
    fn = oracle.attn_causal if causal else oracle.attn_noncausal
    assert np.allclose(fn(Q, K, V, om, kind=kind)[0], stored, rtol=1e-14, atol=1e-15)
    assert np.allclose(_brute(kind, causal), stored, rtol=1e-12, atol=1e-14)


def test_golden_features():
    stored = _arr("Phi_Q_row_exp")
    assert np.allclose(oracle.features(_arr("Q")[None], _arr("Omega"), stab="row")[0], stored, rtol=1e-14)
