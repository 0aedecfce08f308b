"""Pins of the oracle's random projection builder (CPU).

oracle.omega_orf follows "Performer for vision", *What Is Performer?*, Orthogonal Features, and
the "Performer" paper note's FAVOR+ section: Gaussian blocks of d rows, orthonormalised in order,
each row rescaled to a chi_d length. Every pin checks it against something other than itself: a
library QR factorisation, the lengths of the raw draws, exact orthogonality, the raw draws
themselves for the unstructured variant.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si


def unit_rows(om):
    return om / np.linalg.norm(om, axis=1, keepdims=True)


@pytest.mark.parametrize("m,d", [(64, 64), (200, 64), (256, 128)])
def test_rows_are_gram_schmidt_of_the_gaussian_blocks(m, d):
    # Gram-Schmidt on the rows of G gives G = L E with L lower triangular (positive diagonal) and E
    # orthonormal; a library QR of G^T = Q R gives the same E up to the signs of R's diagonal.
    seed = 31 + m
    om = oracle.omega_orf(seed, m, d)
    nblk = -(-m // d)
    G = si.normal(seed, 4, nblk * d * d).reshape(nblk, d, d)
    E = unit_rows(om)
    for b in range(nblk):
        Q, R = np.linalg.qr(G[b].T)
        ref = (Q * np.sign(np.diag(R))[None, :]).T
        rows = min(d, m - b * d)
        assert np.abs(E[b * d:b * d + rows] - ref[:rows]).max() < 1e-10


@pytest.mark.parametrize("m,d", [(100, 64), (384, 128)])
def test_row_lengths_are_the_chi_draws(m, d):
    seed = 5
    om = oracle.omega_orf(seed, m, d)
    chi = np.linalg.norm(si.normal(seed, 5, m * d).reshape(m, d), axis=1)
    np.testing.assert_allclose(np.linalg.norm(om, axis=1), chi, rtol=1e-12)


def test_rows_of_a_block_are_exactly_orthogonal_and_blocks_are_independent():
    d, m = 64, 192
    om = oracle.omega_orf(8, m, d)
    E = unit_rows(om)
    for b in range(m // d):
        blk = E[b * d:(b + 1) * d]
        assert np.abs(blk @ blk.T - np.eye(d)).max() < 1e-12
    # two different blocks are independent draws, not orthogonal to each other
    cross = E[:d] @ E[d:2 * d].T
    assert np.abs(cross).max() > 0.2


def test_last_block_keeps_its_first_rows():
    full = oracle.omega_orf(3, 128, 64)
    part = oracle.omega_orf(3, 70, 64)
    assert part.shape == (70, 64)
    assert np.array_equal(part, full[:70])
    assert oracle.omega_orf(3, 0, 64).shape == (0, 64)


def test_unstructured_variant_is_the_raw_draws():
    m, d = 90, 64
    om = oracle.omega_orf(12, m, d, orthogonal=False)
    raw = si.normal(12, 4, 2 * d * d).reshape(2 * d, d)[:m]
    assert np.array_equal(om, raw)


def test_rows_are_marginally_standard_gaussian():
    # each row chi_d * (uniform unit vector) is N(0, I_d): entries have mean 0 and variance 1
    om = oracle.omega_orf(2024, 64 * 64, 64)
    assert abs(om.mean()) < 0.01
    assert abs(om.var() - 1.0) < 0.02


def test_seed_changes_the_draw_and_matches_the_workload_input_builder():
    a = oracle.omega_orf(1, 64, 64)
    b = oracle.omega_orf(2, 64, 64)
    assert np.abs(a - b).max() > 1.0
    # the workloads' Omega (built by the input module) is the same definition
    assert np.abs(a - si.build_omega(1, 64, 64)).max() < 1e-12
