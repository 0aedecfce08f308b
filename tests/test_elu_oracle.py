"""Pins of the oracle's elu + 1 linear attention (CPU).

oracle.attn_linear_elu computes phi(Q) (phi(K)^T V) / phi(Q) (phi(K)^T 1) with phi = elu + 1 (the
Linear Transformer's feature map, named in the comparison table of the question page "How do linear
attention variants (Performer, Linformer) achieve O(n) complexity, and what's the quality cost?"
and in "Performer for vision", *Kernel Choices*). Each pin fixes it by something other than its own
formula: a library elu, a hand-computed example, closed forms, and invariants.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def test_feature_map_is_library_elu_plus_one():
    x = np.concatenate([np.linspace(-30, 30, 2001), [0.0, -0.0, 1e-300, -1e-300]])
    # the library forms expm1(x) + 1 in fp64 for x <= 0, exact up to the final addition's rounding
    # (half an ulp of 1); the oracle's exp(x) is the same value without that rounding
    ref = torch.nn.functional.elu(torch.from_numpy(x), alpha=1.0).numpy() + 1.0
    np.testing.assert_allclose(oracle.elu1_features(x), ref, rtol=1e-15, atol=2.0**-53)
    assert np.all(oracle.elu1_features(x) > 0)


def test_hand_computed_example():
    # one query q = 0.5 over keys 1 and -1 with values 2 and 4 (d = 1):
    # phi(k) = 2 and e^-1, so y = (2 * 2 + e^-1 * 4) / (2 + e^-1); phi(q) cancels
    Q = np.array([[0.5]])
    K = np.array([[1.0], [-1.0]])
    V = np.array([[2.0], [4.0]])
    y = oracle.attn_linear_elu(Q, K, V, causal=False)
    e = math.exp(-1.0)
    assert y.shape == (1, 1)
    assert abs(y[0, 0] - (4.0 + 4.0 * e) / (2.0 + e)) < 1e-15
    # causal, two queries: row 0 sees key 0 only, row 1 both keys
    Qc = np.array([[0.5], [-2.0]])
    yc = oracle.attn_linear_elu(Qc, K, V, causal=True)
    assert abs(yc[0, 0] - 2.0) < 1e-15
    assert abs(yc[1, 0] - (4.0 + 4.0 * e) / (2.0 + e)) < 1e-15


def test_multidimensional_hand_example():
    # d = 2: phi(q) = (1, 3), phi(k0) = (2, 1), phi(k1) = (1, e^-2); scores 5 and 1 + 3 e^-2
    Q = np.array([[0.0, 2.0]])
    K = np.array([[1.0, 0.0], [0.0, -2.0]])
    V = np.array([[1.0, -1.0], [3.0, 5.0]])
    a0, a1 = 5.0, 1.0 + 3.0 * math.exp(-2.0)
    ref = (a0 * V[0] + a1 * V[1]) / (a0 + a1)
    np.testing.assert_allclose(oracle.attn_linear_elu(Q, K, V, causal=False)[0], ref, rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_plain_and_prefix_means(causal):
    r = rng(1)
    n, d = 40, 8
    Q = r.normal(size=(n, d))
    K = np.tile(r.normal(size=(1, d)), (n, 1))
    V = r.normal(size=(n, d))
    y = oracle.attn_linear_elu(Q, K, V, causal=causal)
    ref = np.cumsum(V, axis=0) / np.arange(1, n + 1)[:, None] if causal else np.tile(V.mean(axis=0), (n, 1))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_pass_through(causal):
    r = rng(2)
    Q, K = r.normal(size=(2, 3, 50, 16)), r.normal(size=(2, 3, 50, 16))
    c = r.normal(size=16)
    V = np.broadcast_to(c, (2, 3, 50, 16))
    np.testing.assert_allclose(oracle.attn_linear_elu(Q, K, V, causal=causal), np.broadcast_to(c, V.shape),
                               rtol=1e-12, atol=1e-13)


def test_causal_rows_are_noncausal_attention_over_their_prefix():
    r = rng(3)
    n, d = 30, 8
    Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, d))
    yc = oracle.attn_linear_elu(Q, K, V, causal=True)
    for i in (0, 1, 17, n - 1):
        yi = oracle.attn_linear_elu(Q[i:i + 1], K[:i + 1], V[:i + 1], causal=False)
        np.testing.assert_allclose(yc[i], yi[0], rtol=1e-12, atol=1e-14)


def test_noncausal_is_invariant_to_permuting_the_keys():
    r = rng(4)
    n, d = 64, 16
    Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, d))
    p = r.permutation(n)
    np.testing.assert_allclose(oracle.attn_linear_elu(Q, K, V, causal=False),
                               oracle.attn_linear_elu(Q, K[p], V[p], causal=False), rtol=1e-12, atol=1e-14)


def test_outputs_are_convex_combinations_of_the_values():
    # phi > 0, so every output row lies inside the box spanned by the (visible) value rows
    r = rng(5)
    Q, K, V = r.normal(size=(3, 80, 8)), r.normal(size=(3, 80, 8)), r.normal(size=(3, 80, 8))
    for causal in (False, True):
        y = oracle.attn_linear_elu(Q, K, V, causal=causal)
        assert np.all(y <= V.max(axis=-2, keepdims=True) + 1e-12)
        assert np.all(y >= V.min(axis=-2, keepdims=True) - 1e-12)
