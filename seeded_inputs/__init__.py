"""Seeded synthetic inputs for FAVOR+ attention, shared by the fp64 oracle and the CUDA path.

This module holds no FAVOR+ arithmetic. It produces:

* Q, K, V as iid N(0, sigma^2) samples from a counter-based generator (``gen.c``), rounded to the
  workload dtype (fp32, or bf16 by round-to-nearest-even), so both sides see identical values;
* the random projection Omega (m x d), the one random draw the method makes. It is built as the
  "Performer" paper note's FAVOR+ section and the "Performer for vision" page's *Orthogonal
  Features* paragraph describe it: Gaussian blocks of d rows, orthogonalised, then each row
  rescaled to an independent chi_d length so that every row is still marginally N(0, I_d).

Everything is a function of (seed, tensor id, flat element index), so one head of a multi-GB
workload can be rebuilt on its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import WORKLOADS, Workload, get_workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_gen.so")
_lib = None
_lock = threading.Lock()

# Tensor ids of the counter-based streams.
TID_Q, TID_K, TID_V, TID_G, TID_CHI = 1, 2, 3, 4, 5


def build_library(force: bool = False) -> str:
    """Compile ``gen.c`` into ``_gen.so`` next to it (gcc, OpenMP). Returns the path."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_library())
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            for name in ("si_normal_f64", "si_normal_f32", "si_normal_bf16"):
                getattr(lib, name).argtypes = [u64, u64, u64, i64, dbl, vp]
                getattr(lib, name).restype = None
            lib.si_f32_to_bf16.argtypes = [vp, i64, vp]
            lib.si_bf16_to_f32.argtypes = [vp, i64, vp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def normal(seed: int, tensor_id: int, count: int, *, offset: int = 0, sigma: float = 1.0,
           dtype: str = "f64") -> np.ndarray:
    """``count`` samples of N(0, sigma^2) at flat indices ``offset .. offset+count-1``.

    dtype "f64" returns float64, "f32" float32, "bf16" the uint16 bit patterns of bf16 values.
    """
    lib = _load()
    if dtype == "f64":
        out = np.empty(count, np.float64)
        lib.si_normal_f64(seed, tensor_id, offset, count, sigma, _ptr(out))
    elif dtype == "f32":
        out = np.empty(count, np.float32)
        lib.si_normal_f32(seed, tensor_id, offset, count, sigma, _ptr(out))
    elif dtype == "bf16":
        out = np.empty(count, np.uint16)
        lib.si_normal_bf16(seed, tensor_id, offset, count, sigma, _ptr(out))
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().si_f32_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    bits = np.ascontiguousarray(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().si_bf16_to_f32(_ptr(bits), bits.size, _ptr(out))
    return out


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact float64 view of generator output in any of its dtypes."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------------------------
# Omega: the method's random projection (an input to both sides)
# ----------------------------------------------------------------------------------------------

def _gram_schmidt_rows(G: np.ndarray) -> np.ndarray:
    """Modified Gram-Schmidt on the rows of each d x d matrix in a stack [..., d, d] (fp64)."""
    E = np.array(G, dtype=np.float64, copy=True)
    d = E.shape[-2]
    for i in range(d):
        v = E[..., i, :]
        for j in range(i):
            e = E[..., j, :]
            v -= np.sum(v * e, axis=-1, keepdims=True) * e
        v /= np.linalg.norm(v, axis=-1, keepdims=True)
        E[..., i, :] = v
    return E


def build_omega(seed: int, m: int, d: int, *, orthogonal: bool = True) -> np.ndarray:
    """The m x d projection Omega in float64.

    orthogonal=True: ceil(m/d) blocks, each a d x d Gaussian matrix (stream TID_G) whose rows are
    orthonormalised by modified Gram-Schmidt and then scaled row by row to the length of an
    independent d-dimensional Gaussian vector (stream TID_CHI), i.e. a chi_d sample. The last
    block keeps its first m mod d rows when d does not divide m.
    orthogonal=False: m iid N(0, I_d) rows (stream TID_G), the unstructured baseline.
    """
    if m <= 0 or d <= 0:
        raise ValueError("m and d must be positive")
    nblk = -(-m // d)
    G = normal(seed, TID_G, nblk * d * d).reshape(nblk, d, d)
    if not orthogonal:
        return np.ascontiguousarray(G.reshape(nblk * d, d)[:m])
    E = _gram_schmidt_rows(G).reshape(nblk * d, d)[:m]
    chi = np.linalg.norm(normal(seed, TID_CHI, m * d).reshape(m, d), axis=1)
    return np.ascontiguousarray(E * chi[:, None])


def omega_for(w: "Workload") -> tuple[np.ndarray, np.ndarray]:
    """Omega for workload ``w``: (values in the workload dtype's storage, exact float64 copy)."""
    om = build_omega(w.omega_seed, w.m, w.d, orthogonal=True).astype(np.float32)
    if w.dtype == "bf16":
        bits = f32_to_bf16_bits(om)
        return bits, to_f64(bits)
    return om, om.astype(np.float64)


def head_inputs(w: "Workload", b: int, h: int, which: str = "QKV") -> dict:
    """Inputs of one (b, h) head of workload ``w`` in storage dtype: {'Q': n x d, ...}."""
    per_head = w.n * w.d
    off = (b * w.H + h) * per_head
    tids = {"Q": TID_Q, "K": TID_K, "V": TID_V}
    return {t: normal(w.seed, tids[t], per_head, offset=off, sigma=w.sigma, dtype=w.dtype).reshape(w.n, w.d)
            for t in which}


def full_inputs(w: "Workload", which: str = "QKV") -> dict:
    """All of Q, K, V of workload ``w`` as [B, H, n, d] arrays in storage dtype."""
    cnt = w.B * w.H * w.n * w.d
    tids = {"Q": TID_Q, "K": TID_K, "V": TID_V}
    return {t: normal(w.seed, tids[t], cnt, sigma=w.sigma, dtype=w.dtype).reshape(w.B, w.H, w.n, w.d)
            for t in which}
