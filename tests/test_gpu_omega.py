"""GPU parity of the on-device random projection builder (favor_omega) against the fp64 oracle.

Both sides compute Omega in fp64 from the same counter-based draws ("Performer for vision", *What
Is Performer?*, Orthogonal Features); the device rounds to fp32 (to nearest) and then to bf16 (to
nearest even). The bound per element is the rounding of the output type plus an absolute 1e-9 for
the fp64 differences of the two Gram-Schmidt orders (about 1e-12 at d = 128), and all but a rare
element on a rounding boundary must equal the oracle's value rounded the same way.
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


def rounded(x64: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    f32 = x64.astype(np.float32)
    if dtype == torch.bfloat16:
        return si.bf16_bits_to_f32(si.f32_to_bf16_bits(f32)).astype(np.float64)
    return f32.astype(np.float64)


def check_against_oracle(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, what: str):
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, what
    unit = 2.0**-24 if dtype == torch.float32 else 2.0**-8 + 2.0**-23
    err = np.abs(g - ref)
    bound = unit * np.abs(ref) + 1e-9
    assert np.all(err <= bound), f"{what}: worst excess {float((err - bound).max()):.3g}"
    off = int(np.count_nonzero(g != rounded(ref, dtype)))
    assert off <= max(1, ref.size // 1000), f"{what}: {off} of {ref.size} elements differ from the rounded oracle"


CASES = ([(64, m) for m in (1, 37, 64, 200, 256, 512, 1000)] + [(128, m) for m in (1, 130, 256, 512)])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("orthogonal", [True, False], ids=["orf", "iid"])
@pytest.mark.parametrize("d,m", CASES)
def test_omega_matches_oracle(favor, d, m, orthogonal, dtype):
    seed = 1000 + 7 * m + d
    om = favor.favor_omega(seed, m, d, dtype=dtype, orthogonal=orthogonal)
    torch.cuda.synchronize()
    assert favor.last_device_error() == 0
    ref = oracle.omega_orf(seed, m, d, orthogonal=orthogonal)
    check_against_oracle(om, ref, dtype, f"omega d={d} m={m} orthogonal={orthogonal}")


def test_rows_of_a_block_are_orthogonal_on_the_device(favor):
    d, m = 128, 256
    om = favor.favor_omega(77, m, d, dtype=torch.float32).double().cpu().numpy()
    for b in range(m // d):
        blk = om[b * d:(b + 1) * d]
        g = blk @ blk.T
        nrm = np.sqrt(np.diag(g))
        assert np.abs(g / np.outer(nrm, nrm) - np.eye(d)).max() < 1e-6


def test_same_seed_same_draw_new_seed_redraws(favor):
    a = favor.favor_omega(5, 256, 64)
    b = favor.favor_omega(5, 256, 64)
    c = favor.favor_omega(6, 256, 64)
    assert torch.equal(a, b)
    assert float((a.float() - c.float()).abs().max()) > 1.0


def test_device_omega_is_the_workload_projection(favor):
    # the Omega of the attention workloads (built on the host by the input module) is the same draw
    w = si.get_workload("noncausal_bf16_B1H8n1024d64m256")
    bits, _ = si.omega_for(w)
    host = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    dev = favor.favor_omega(w.omega_seed, w.m, w.d, dtype=torch.bfloat16).cpu()
    assert int((dev != host).sum()) <= 2


def test_attention_with_a_device_built_omega_matches_oracle(favor):
    w = si.Workload("omega_e2e", 1, 4, 300, 64, 256, "bf16", False, seed=21, omega_seed=22)
    Q, K, V, _, _ = device_inputs(w)
    Om = favor.favor_omega(1234, 256, 64, dtype=torch.bfloat16)
    Y = favor.favor_attn_noncausal(Q, K, V, Om)
    torch.cuda.synchronize()
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    ref = oracle.attn_noncausal(f64(Q), f64(K), f64(V), f64(Om))
    assert_close_attn(f64(Y), ref, "bf16", "attention with device Omega")


def test_empty_and_unsupported(favor):
    assert favor.favor_omega(1, 0, 64).shape == (0, 64)
    with pytest.raises(favor.FavorError):
        favor.favor_omega(1, 64, 96)
