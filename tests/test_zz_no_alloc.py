"""favor_attn_noncausal_noalloc: the non-causal entry point for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc (a plugin whose host application owns every
device allocation, a real-time loop that must never enter the allocator, a process whose memory
pool is fixed at start-up). For them the library offers one entry point whose scratch lives in a
fixed device array compiled into libfavor.so. These tests call it through the C ABI and compare it
with favor_attn_noncausal (which takes a caller-owned workspace) on two calls in a row, so that the
second call runs on scratch left over from the first. This file is named to be collected last.
"""
import ctypes

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


def _noalloc_c_call(favor, Q, K, V, Om, Y, w):
    """Calls the C entry point directly with raw device pointers on the current stream."""
    vp = ctypes.c_void_p
    return favor.lib.favor_attn_noncausal_noalloc(
        vp(Q.data_ptr()), vp(K.data_ptr()), vp(V.data_ptr()), vp(Om.data_ptr()), vp(Y.data_ptr()),
        w.B, w.H, w.n, w.d, w.m, 1 if w.dtype == "bf16" else 0, 0 if w.kind == "exp" else 1, w.relu_eps,
        vp(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_workspace_entry_point_twice(favor, dtype):
    # The d = 128 case runs first and fills the scratch; the fused (n <= 1024, d = 64) case then runs
    # on what it left behind. Each call is checked against the workspace entry point and the oracle.
    cases = [si.Workload("noalloc_b", 2, 3, 777, 128, 192, dtype, False, seed=503, omega_seed=504),
             si.Workload("noalloc_a", 1, 8, 1024, 64, 256, dtype, False, seed=501, omega_seed=502)]
    for w in cases:  # two calls in a row; the second reuses scratch the first one filled
        assert favor.workspace_bytes("noncausal", w.B, w.H, w.n, w.d, w.m,
                                     torch.bfloat16 if dtype == "bf16" else torch.float32) \
            <= favor.NOALLOC_SCRATCH_BYTES
        Q, K, V, Om, om64 = device_inputs(w)
        ref = favor.favor_attn_noncausal(Q, K, V, Om)
        Y = torch.full_like(Q, float("nan"))
        assert _noalloc_c_call(favor, Q, K, V, Om, Y, w) == 0
        torch.cuda.synchronize()
        assert favor.last_device_error() == 0
        got = Y.float().cpu().numpy().astype(np.float64)
        assert_close_attn(got, ref.float().cpu().numpy().astype(np.float64), dtype, f"noalloc {w.name}")
        f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
        oref = oracle.attn_noncausal(f64(Q), f64(K), f64(V), om64, kind=w.kind, relu_eps=w.relu_eps)
        assert_close_attn(got, oref, dtype, f"noalloc {w.name} vs oracle")


def test_noalloc_rejects_shapes_beyond_its_scratch(favor):
    w = si.Workload("too_big", 4, 64, 65536, 128, 512, "bf16", False)
    need = favor.workspace_bytes("noncausal", w.B, w.H, w.n, w.d, w.m, torch.bfloat16)
    assert need > favor.NOALLOC_SCRATCH_BYTES
    # Small real buffers are enough: the size check fails before any pointer is used.
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    vp = ctypes.c_void_p
    st = favor.lib.favor_attn_noncausal_noalloc(vp(t.data_ptr()), vp(t.data_ptr()), vp(t.data_ptr()),
                                                vp(t.data_ptr()), vp(t.data_ptr()), w.B, w.H, w.n, w.d, w.m, 1, 0,
                                                1e-3, vp(torch.cuda.current_stream().cuda_stream))
    assert st == 4  # FAVOR_ERR_WORKSPACE
