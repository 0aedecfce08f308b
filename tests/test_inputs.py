"""Pins of the seeded input generator and of the Omega builder (CPU)."""
import numpy as np
import pytest
import scipy.stats
import torch

import seeded_inputs as si


def test_generator_is_counter_based():
    a = si.normal(7, si.TID_Q, 1000)
    b = si.normal(7, si.TID_Q, 400, offset=600)
    assert np.array_equal(a[600:], b)
    assert np.array_equal(a, si.normal(7, si.TID_Q, 1000))
    assert not np.array_equal(a, si.normal(8, si.TID_Q, 1000))
    assert not np.array_equal(a, si.normal(7, si.TID_K, 1000))


def test_generator_is_standard_normal():
    n = 400_000
    x = si.normal(11, si.TID_V, n)
    assert abs(x.mean()) < 4 / np.sqrt(n)
    assert abs(x.var() - 1) < 4 * np.sqrt(2 / n)
    assert scipy.stats.kstest(x[:100_000], "norm").pvalue > 1e-4
    # independent streams are uncorrelated
    y = si.normal(11, si.TID_Q, n)
    assert abs(np.corrcoef(x, y)[0, 1]) < 4 / np.sqrt(n)


def test_sigma_and_dtype_rounding():
    x64 = si.normal(3, si.TID_K, 5000, sigma=0.5)
    x32 = si.normal(3, si.TID_K, 5000, sigma=0.5, dtype="f32")
    assert np.array_equal(x32, x64.astype(np.float32))
    bits = si.normal(3, si.TID_K, 5000, sigma=0.5, dtype="bf16")
    # round-to-nearest-even of the fp32 value, as torch rounds fp32 -> bf16
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    assert np.array_equal(si.bf16_bits_to_f32(bits), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("m,d", [(128, 64), (256, 64), (256, 128), (40, 16), (7, 4)])
def test_omega_blocks_are_orthogonal(m, d):
    om = si.build_omega(5, m, d)
    assert om.shape == (m, d)
    for b0 in range(0, m, d):
        blk = om[b0:b0 + d]
        gram = blk @ blk.T
        norms2 = np.sum(blk * blk, axis=1)
        assert np.allclose(gram, np.diag(norms2), rtol=0, atol=1e-11 * norms2.max())


def test_gram_schmidt_matches_library_qr():
    # Rows orthonormalised by Gram-Schmidt equal the Q factor of QR(G^T) up to the sign of each row.
    d = 16
    G = si.normal(21, si.TID_G, d * d).reshape(d, d)
    E = si._gram_schmidt_rows(G)
    Qf, R = np.linalg.qr(G.T)
    Qr = (Qf * np.sign(np.diag(R))).T
    assert np.allclose(E, Qr, atol=1e-12)


def test_omega_rows_have_chi_norms():
    d, m = 16, 16 * 2000
    om = si.build_omega(9, m, d)
    r2 = np.sum(om * om, axis=1)
    # |w|^2 ~ chi^2_d: mean d, variance 2d
    assert abs(r2.mean() - d) < 4 * np.sqrt(2 * d / m)
    assert abs(r2.var() - 2 * d) < 4 * np.sqrt((8 * d * d + 48 * d) / m)  # var of sample variance of chi^2_d
    # each coordinate is marginally N(0, 1)
    assert scipy.stats.kstest(om[:, 3], "norm").pvalue > 1e-4


def test_omega_iid_rows_are_the_gaussian_stream():
    om = si.build_omega(4, 10, 8, orthogonal=False)
    assert np.array_equal(om, si.normal(4, si.TID_G, 2 * 64)[:80].reshape(10, 8))


def test_workload_heads_are_slices_of_full_tensors():
    w = si.get_workload("noncausal_bf16_B1H8n1024d64m256").with_(n=32, H=3)
    full = si.full_inputs(w)
    h = si.head_inputs(w, 0, 2)
    for t in "QKV":
        assert np.array_equal(full[t][0, 2], h[t])
