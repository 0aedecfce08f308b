"""Shared test plumbing: seeded inputs on the device, oracle references per head, tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import seeded_inputs as si

# Tolerances of the attention outputs against the fp64 oracle.
F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 1e-2
# Feature map: error relative to the row's scale max(1/sqrt(m), largest |phi| of the row) -- with a
# stabiliser the largest feature is at most 1/sqrt(m); without one it can be far larger. fp32
# arithmetic on both input dtypes; the inputs themselves are exact on both sides.
FEATURES_SCALED_ABS = 2e-5


def torch_dtype(w) -> torch.dtype:
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def to_device(a: np.ndarray, dtype: torch.dtype, device="cuda") -> torch.Tensor:
    """Generator output (float32 values or bf16 bit patterns) -> device tensor of `dtype`."""
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    assert t.dtype == dtype
    return t.to(device)


def device_inputs(w, device="cuda"):
    """(Q, K, V, Omega) device tensors and the float64 Omega of workload w."""
    full = si.full_inputs(w)
    om_store, om64 = si.omega_for(w)
    dt = torch_dtype(w)
    return (to_device(full["Q"], dt, device), to_device(full["K"], dt, device), to_device(full["V"], dt, device),
            to_device(om_store, dt, device), om64)


def head_f64(w, b, h):
    hi = si.head_inputs(w, b, h)
    return {k: si.to_f64(v) for k, v in hi.items()}


def assert_close_attn(y_gpu: np.ndarray, y_ref: np.ndarray, dtype: str, what: str = ""):
    y_gpu = np.asarray(y_gpu, np.float64)
    err = np.abs(y_gpu - y_ref)
    assert np.isfinite(y_gpu).all(), f"{what}: non-finite output"
    max_abs = float(err.max()) if err.size else 0.0
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"{what}: max-abs {max_abs:.3g} > {F32_MAX_ABS}"
    else:
        rel = float(np.linalg.norm(y_gpu - y_ref) / max(np.linalg.norm(y_ref), 1e-30))
        assert max_abs <= BF16_MAX_ABS, f"{what}: max-abs {max_abs:.3g} > {BF16_MAX_ABS}"
        assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3g} > {BF16_REL_L2}"
    return max_abs


def assert_close_features(p_gpu: np.ndarray, p_ref: np.ndarray, m: int, what: str = ""):
    if p_ref.size == 0:
        return
    scale = np.maximum(np.abs(p_ref).max(axis=-1, keepdims=True), 1 / math.sqrt(m))
    err = float((np.abs(np.asarray(p_gpu, np.float64) - p_ref) / scale).max())
    assert err <= FEATURES_SCALED_ABS, f"{what}: max |dphi| / row scale = {err:.3g} > {FEATURES_SCALED_ABS}"
