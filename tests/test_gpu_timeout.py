"""The bounded-wait failure path on the device, exercised without any fault or hang.

Every mbarrier wait in the tensor-core kernels gives up after a time limit (in the causal scan, once
the CTA's watchdog lane has seen no progress for that long), records FAVOR_ERR_TIMEOUT in the device
error word, tells the CTA's other roles to stop, drains its copies in flight and frees its tensor
memory. m = 128 runs the scan's single-CTA instance, m = 512 a group of four CTAs. favor_test_set_wait_limit arms a test hook that shortens the limit to a
millisecond and makes the causal scan withhold one arrival, so that one wait runs out for sure;
the test then checks that the status reaches the host and that the next normal call on the same
device still matches the oracle.
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


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("m", [128, 512])
def test_wait_timeout_is_reported_and_the_device_stays_usable(favor, m):
    w = si.Workload("case", 1, 2, 600, 64, m, "bf16", True, kind="relu", seed=81, omega_seed=82)
    Q, K, V, Om, om64 = device_inputs(w)
    stream = torch.cuda.current_stream()
    assert favor.last_device_error() == 0
    assert favor.lib.favor_test_set_wait_limit(1_000_000, favor._stream_handle(stream)) == 0  # 1 ms
    try:
        favor.favor_attn_causal(Q, K, V, Om, kind=w.kind, relu_eps=w.relu_eps)
        torch.cuda.synchronize()
    finally:
        assert favor.lib.favor_test_set_wait_limit(0, favor._stream_handle(stream)) == 0
    assert favor.last_device_error() == 6  # FAVOR_ERR_TIMEOUT, and the word is cleared
    assert favor.last_device_error() == 0
    # the context is intact: the same call now runs to completion and matches the oracle
    Y = favor.favor_attn_causal(Q, K, V, Om, kind=w.kind, relu_eps=w.relu_eps)
    assert favor.last_device_error() == 0
    ref = oracle.attn_causal(_f64(Q), _f64(K), _f64(V), om64, kind=w.kind, relu_eps=w.relu_eps)
    assert_close_attn(_f64(Y), ref, "bf16", f"after timeout m={m}")
