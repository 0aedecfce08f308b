"""Property-based pins of the oracle (CPU only): identities that hold for every shape, drawn at random.

- the linear forms equal the explicit n x n forms ("Performer" paper note, *Kernel Attention View*
  and *Normalization*; "Performer for vision", *How It Works*, Steps 1 and 2);
- every stabiliser mode gives the same output (the constants cancel in the ratio);
- causal row i is the non-causal attention of query i over keys 0..i.
"""
import numpy as np
from hypothesis import given, settings
from hypothesis import strategies as st

import oracle
import seeded_inputs as si

shapes = st.tuples(st.integers(1, 3), st.integers(1, 12), st.sampled_from([4, 8, 16]), st.integers(1, 4))


def draw(seed, h, n, d, mblk, scale):
    g = np.random.default_rng(seed)
    Q, K, V = (g.standard_normal((h, n, d)) * scale for _ in range(3))
    return Q, K, V, si.build_omega(seed % 1000, mblk * d, d)


@settings(max_examples=40, deadline=None)
@given(shapes, st.integers(0, 2**31 - 1), st.sampled_from(["exp", "relu"]), st.booleans(), st.floats(0.1, 2.0))
def test_linear_forms_equal_quadratic_forms(shape, seed, kind, causal, scale):
    h, n, d, mblk = shape
    Q, K, V, om = draw(seed, h, n, d, mblk, scale)
    fn = oracle.attn_causal if causal else oracle.attn_noncausal
    lin = fn(Q, K, V, om, kind=kind)
    quad = oracle.attn_quadratic(Q, K, V, om, causal=causal, kind=kind)
    assert np.allclose(lin, quad, rtol=1e-9, atol=1e-11)


@settings(max_examples=40, deadline=None)
@given(shapes, st.integers(0, 2**31 - 1), st.booleans(), st.floats(0.1, 2.0))
def test_stabiliser_modes_agree(shape, seed, causal, scale):
    h, n, d, mblk = shape
    Q, K, V, om = draw(seed, h, n, d, mblk, scale)
    fn = oracle.attn_causal if causal else oracle.attn_noncausal
    ref = fn(Q, K, V, om, mode="canonical")
    for mode in ("none", "bound"):
        assert np.allclose(fn(Q, K, V, om, mode=mode), ref, rtol=1e-9, atol=1e-12)


@settings(max_examples=30, deadline=None)
@given(shapes, st.integers(0, 2**31 - 1), st.sampled_from(["exp", "relu"]))
def test_causal_rows_are_prefix_attention(shape, seed, kind):
    h, n, d, mblk = shape
    Q, K, V, om = draw(seed, h, n, d, mblk, 1.0)
    yc = oracle.attn_causal(Q, K, V, om, kind=kind)
    i = int(np.random.default_rng(seed).integers(0, n))
    # (the oracle takes as many queries as keys: attend with the prefix's queries, read row i)
    yi = oracle.attn_noncausal(Q[:, :i + 1], K[:, :i + 1], V[:, :i + 1], om, kind=kind)
    assert np.allclose(yc[:, i], yi[:, i], rtol=1e-9, atol=1e-12)
