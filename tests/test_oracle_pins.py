"""Pins of the fp64 oracle against what the pages and mathematics fix (CPU only).

Each test names the fact it checks. None of them re-types the oracle's own arithmetic: they use
brute force (the explicit n x n form), expectations over the random projection, closed forms,
invariants and special cases.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si

RNG = np.random.default_rng(20201)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ---------------------------------------------------------------------------------------------
# Feature map ("Performer" paper note, FAVOR+: positive random features, E[phi(q)^T phi(k)] = exp(q^T k))
# ---------------------------------------------------------------------------------------------

def test_exp_features_are_positive_and_row_stabilised():
    d, m, n = 16, 48, 37
    om = si.build_omega(1, m, d)
    X = rand(2, n, d)
    P = oracle.features(X, om, stab="row")
    assert (P > 0).all()
    # with the per-row stabiliser the largest feature of each row is exp(0)/sqrt(m)
    assert np.allclose(P.max(axis=-1), 1 / math.sqrt(m), rtol=1e-15, atol=0)
    Ph = oracle.features(X, om, stab="head")
    assert np.allclose(Ph.reshape(2, -1).max(axis=-1), 1 / math.sqrt(m), rtol=1e-15, atol=0)
    P0 = oracle.features(X, om, stab="none")
    # the stabilisers only rescale whole rows / whole heads
    ratio_row = P0 / P
    assert np.allclose(ratio_row, ratio_row[..., :1], rtol=1e-12)
    ratio_head = P0 / Ph
    assert np.allclose(ratio_head, ratio_head[:, :1, :1], rtol=1e-12)


def _block_estimates(q, k, om, d, kind, eps=0.0):
    """phi(q)^T phi(k) split into one term per orthogonal block of d features."""
    pq = oracle.features(q[None], om, kind=kind, relu_eps=eps, stab="none")[0]
    pk = oracle.features(k[None], om, kind=kind, relu_eps=eps, stab="none")[0]
    return (pq * pk).reshape(-1, d).sum(axis=1)  # sum over each block; total = sum of these


@pytest.mark.parametrize("orthogonal", [True, False])
@pytest.mark.parametrize("case", range(3))
def test_exp_features_are_unbiased_for_the_softmax_kernel(orthogonal, case):
    """E_w[phi(q)^T phi(k)] = exp(q^T k / sqrt(d)) for raw q, k (the d^-1/4 scaling is inside)."""
    d, T = 16, 20000
    g = np.random.default_rng(100 + case)
    qh = g.standard_normal(d); qh *= g.uniform(0.2, 1.0) / np.linalg.norm(qh)
    kh = g.standard_normal(d); kh *= g.uniform(0.2, 1.0) / np.linalg.norm(kh)
    q, k = qh * d ** 0.25, kh * d ** 0.25
    om = si.build_omega(1000 + case, T * d, d, orthogonal=orthogonal)
    blocks = _block_estimates(q, k, om, d, "exp")
    total = blocks.sum()                       # = phi(q)^T phi(k) with m = T*d features
    stderr = blocks.std(ddof=1) * math.sqrt(T)  # std of the sum of T iid block terms
    target = math.exp(qh @ kh)
    assert abs(total - target) < 4 * stderr, (total, target, stderr)
    # and it is a real test: dropping the -|x|^2/2 term moves the mean far outside the band
    assert abs(total * math.exp(0.5 * (qh @ qh + kh @ kh)) - target) > 4 * stderr


def test_relu_features_match_arccos_kernel_expectation():
    """E_w[phi(q)^T phi(k)] for phi = ReLU(w^T x^)/sqrt(m) + eps, closed form via the order-1
    arc-cosine kernel: E[(w.a)+ (w.b)+] = |a||b|(sin t + (pi - t) cos t) / (2 pi), E[(w.a)+] = |a|/sqrt(2 pi)."""
    d, T, eps = 16, 20000, 1e-3
    g = np.random.default_rng(7)
    qh = g.standard_normal(d) * 0.3
    kh = g.standard_normal(d) * 0.3
    q, k = qh * d ** 0.25, kh * d ** 0.25
    m = T * d
    om = si.build_omega(77, m, d)
    blocks = _block_estimates(q, k, om, d, "relu", eps)
    total = blocks.sum()
    stderr = blocks.std(ddof=1) * math.sqrt(T)
    a, b = np.linalg.norm(qh), np.linalg.norm(kh)
    t = math.acos(np.clip(qh @ kh / (a * b), -1, 1))
    k1 = a * b * (math.sin(t) + (math.pi - t) * math.cos(t)) / (2 * math.pi)
    expect = k1 + eps * math.sqrt(m) * (a + b) / math.sqrt(2 * math.pi) + m * eps * eps
    assert abs(total - expect) < 4 * stderr, (total, expect, stderr)


def test_relu_features_floor_and_zero_projection():
    d, m = 8, 24
    om = si.build_omega(3, m, d)
    X = rand(1, 20, d)
    P = oracle.features(X, om, kind="relu", relu_eps=1e-3)
    assert (P >= 1e-3).all()
    # a row of Omega orthogonal to x gives exactly the floor; -x flips which features are active
    xs = X[0]
    Pn = oracle.features(-X, om, kind="relu", relu_eps=1e-3)
    active = P[0] > 1e-3
    assert np.all(Pn[0][active] == 1e-3)
    assert np.allclose(P[0] - 1e-3 + Pn[0] - 1e-3, np.abs(xs @ om.T) * d ** -0.25 / math.sqrt(m), atol=1e-15)


# ---------------------------------------------------------------------------------------------
# Associativity and normalisation ("Performer" paper note, Kernel Attention View / Normalization;
# linear-attention lesson: (phi(Q) phi(K)^T) V == phi(Q) (phi(K)^T V))
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 5, 33, 64])
@pytest.mark.parametrize("d,m", [(4, 8), (16, 32), (16, 8)])
@pytest.mark.parametrize("kind", ["exp", "relu"])
def test_linear_forms_equal_quadratic_forms(n, d, m, kind):
    om = si.build_omega(n + d + m, m, d)
    Q, K, V = rand(2, n, d), rand(2, n, d), rand(2, n, d)
    for causal, fn in ((False, oracle.attn_noncausal), (True, oracle.attn_causal)):
        lin = fn(Q, K, V, om, kind=kind)
        quad = oracle.attn_quadratic(Q, K, V, om, causal=causal, kind=kind)
        assert np.allclose(lin, quad, rtol=1e-12, atol=1e-13), (causal, np.abs(lin - quad).max())


def test_causal_first_token_and_prefix_structure():
    d, m, n = 16, 32, 50
    om = si.build_omega(2, m, d)
    Q, K, V = rand(1, n, d), rand(1, n, d), rand(1, n, d)
    Y = oracle.attn_causal(Q, K, V, om)
    assert np.allclose(Y[0, 0], V[0, 0], rtol=1e-14, atol=1e-15)
    # y_i depends only on tokens <= i: truncating the sequence changes nothing before the cut
    Yt = oracle.attn_causal(Q[:, :20], K[:, :20], V[:, :20], om)
    assert np.allclose(Yt, Y[:, :20], rtol=1e-14, atol=1e-15)
    # the last causal row equals the non-causal row (the prefix is the whole sequence)
    Yn = oracle.attn_noncausal(Q, K, V, om)
    assert np.allclose(Y[0, -1], Yn[0, -1], rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kind", ["exp", "relu"])
def test_implied_attention_is_a_row_stochastic_convex_combination(causal, kind):
    d, m, n = 16, 64, 40
    om = si.build_omega(4, m, d)
    Q, K, V = rand(1, n, d), rand(1, n, d), rand(1, n, d)
    A = oracle.implied_attention(Q, K, om, causal=causal, kind=kind)
    mask = np.tril(np.ones((n, n), bool)) if causal else np.ones((n, n), bool)
    assert (A[0][mask] > 0).all() and (A[0][~mask] == 0).all()
    assert np.allclose(A.sum(-1), 1, atol=1e-13)
    Y = (oracle.attn_causal if causal else oracle.attn_noncausal)(Q, K, V, om, kind=kind)
    for i in range(n):
        lo = V[0, : i + 1].min(0) if causal else V[0].min(0)
        hi = V[0, : i + 1].max(0) if causal else V[0].max(0)
        assert (Y[0, i] >= lo - 1e-12).all() and (Y[0, i] <= hi + 1e-12).all()


# ---------------------------------------------------------------------------------------------
# Special cases with closed forms
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["exp", "relu"])
def test_identical_keys_give_the_mean_of_values(kind):
    d, m, n = 16, 32, 30
    om = si.build_omega(5, m, d)
    Q, V = rand(1, n, d), rand(1, n, d)
    K = np.repeat(rand(1, 1, d), n, axis=1)
    Yn = oracle.attn_noncausal(Q, K, V, om, kind=kind)
    assert np.allclose(Yn, V.mean(axis=1, keepdims=True), rtol=1e-12, atol=1e-13)
    Yc = oracle.attn_causal(Q, K, V, om, kind=kind)
    prefix_mean = np.cumsum(V, axis=1) / np.arange(1, n + 1)[None, :, None]
    assert np.allclose(Yc, prefix_mean, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("fn", [oracle.attn_noncausal, oracle.attn_causal])
def test_constant_values_single_token_and_linearity(fn):
    d, m, n = 16, 32, 25
    om = si.build_omega(6, m, d)
    Q, K = rand(1, n, d), rand(1, n, d)
    c = rand(d)
    assert np.allclose(fn(Q, K, np.broadcast_to(c, (1, n, d)), om), c, rtol=1e-12)
    assert np.allclose(fn(Q[:, :1], K[:, :1], Q[:, :1] * 0 + c, om), c, rtol=1e-12)
    V1, V2 = rand(1, n, d), rand(1, n, d)
    lhs = fn(Q, K, 2.5 * V1 - 0.75 * V2, om)
    rhs = 2.5 * fn(Q, K, V1, om) - 0.75 * fn(Q, K, V2, om)
    assert np.allclose(lhs, rhs, rtol=1e-11, atol=1e-12)


def test_noncausal_is_invariant_to_joint_key_value_permutation():
    d, m, n = 16, 32, 41
    om = si.build_omega(7, m, d)
    Q, K, V = rand(1, n, d), rand(1, n, d), rand(1, n, d)
    p = RNG.permutation(n)
    assert np.allclose(oracle.attn_noncausal(Q, K, V, om), oracle.attn_noncausal(Q, K[:, p], V[:, p], om), rtol=1e-12)


@pytest.mark.parametrize("fn", [oracle.attn_noncausal, oracle.attn_causal])
def test_stabiliser_invariance(fn):
    d, m, n = 16, 64, 33
    om = si.build_omega(8, m, d)
    Q, K, V = rand(3, n, d), rand(3, n, d), rand(3, n, d)
    ref = fn(Q, K, V, om, mode="canonical")
    assert np.allclose(fn(Q, K, V, om, mode="none"), ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(fn(Q, K, V, om, mode="bound"), ref, rtol=1e-12, atol=1e-13)


def test_canonical_stabiliser_survives_large_inputs():
    # unstabilised exponents overflow fp64 here; the canonical stabilisers keep Y finite and convex
    d, m, n = 16, 32, 20
    om = si.build_omega(9, m, d)
    Q, K, V = rand(1, n, d, scale=60.0), rand(1, n, d, scale=60.0), rand(1, n, d)
    assert not np.isfinite(oracle.attn_noncausal(Q, K, V, om, mode="none")).all()
    Y = oracle.attn_noncausal(Q, K, V, om)
    assert np.isfinite(Y).all()
    assert (Y >= V.min(1) - 1e-12).all() and (Y <= V.max(1) + 1e-12).all()


# ---------------------------------------------------------------------------------------------
# Exact softmax helper and convergence of FAVOR+ towards it as m grows
# ---------------------------------------------------------------------------------------------

def test_softmax_helper_against_library_softmax():
    import scipy.special

    Q, K, V = rand(2, 9, 8), rand(2, 9, 8), rand(2, 9, 8)
    ref = scipy.special.softmax(Q @ np.swapaxes(K, -1, -2) / math.sqrt(8), axis=-1) @ V
    assert np.allclose(oracle.softmax_attention(Q, K, V), ref, rtol=1e-13)
    # one dominant key -> its value
    K2 = K.copy(); K2[0, 4] = Q[0, 0] * 1e3
    assert np.allclose(oracle.softmax_attention(Q[:, :1], K2, V)[0, 0], V[0, 4], atol=1e-12)


def test_favor_converges_to_softmax_attention_as_m_grows():
    d, n = 16, 256
    ms = [16, 64, 256, 1024, 4096]
    errs = np.zeros((8, len(ms)))
    for s in range(8):
        g = np.random.default_rng(500 + s)
        # sigma = d^-1/4 puts |q^| near 1, where the estimator's variance (which grows like
        # exp(|q^ + k^|^2)) lets the Monte-Carlo rate show at these m
        Q, K = 0.5 * g.standard_normal((1, n, d)), 0.5 * g.standard_normal((1, n, d))
        V = g.standard_normal((1, n, d))
        ex = oracle.softmax_attention(Q, K, V)
        for i, m in enumerate(ms):
            om = si.build_omega(600 + s, m, d)
            Y = oracle.attn_noncausal(Q, K, V, om)
            errs[s, i] = np.linalg.norm(Y - ex) / np.linalg.norm(ex)
    ge = np.exp(np.log(errs).mean(axis=0))
    assert (np.diff(ge) < 0).all(), ge
    slope = np.polyfit(np.log(ms), np.log(ge), 1)[0]
    assert -0.75 <= slope <= -0.3, (slope, ge)


def test_orthogonal_features_variance_report(capsys):
    """Reported only: the pages claim orthogonal projections lower the estimator's variance."""
    d, T = 16, 4000
    g = np.random.default_rng(3)
    q, k = g.standard_normal(d) * 0.5, g.standard_normal(d) * 0.5
    out = {}
    for orth in (True, False):
        b = _block_estimates(q * d ** 0.25, k * d ** 0.25, si.build_omega(31, T * d, d, orthogonal=orth), d, "exp")
        out[orth] = b.var(ddof=1)
    print(f"block-estimate variance: orthogonal {out[True]:.4g}, iid {out[False]:.4g}")
