"""fp64 oracle for FAVOR+ attention. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import this package. The CUDA path (``kernelized_linear_attention_04_b300``) never imports it, and
the two share no code: the only common dependency is ``seeded_inputs`` (random draws, no method
arithmetic).

Contents
--------
* ``features`` / ``attn_noncausal`` / ``attn_causal``: plain fp64 C loops (``favor_oracle.c``),
  OpenMP over heads. See that file for the passages each step follows.
* ``attn_quadratic``: the explicit n x n form (Phi(Q) Phi(K)^T, optional lower-triangular mask,
  row-normalised, times V) of the "Performer" paper note's *Kernel Attention View* and
  *Normalization* equations, for tiny brute-force checks of the linear forms.
* ``softmax_attention``: exact softmax(Q K^T / sqrt(d)) V, the operator FAVOR+ approximates
  (same page, *Standard Attention Cost*); used only for the convergence check.
* ``omega_orf``: the random projection Omega (orthogonal random features: Gaussian blocks
  orthonormalised in order, rows scaled to chi_d lengths), the reference for the device builder.
* ``elu1_features`` / ``attn_linear_elu``: linear attention with the deterministic elu + 1 feature
  map (no projection), non-causal and causal.

Every function takes raw (unscaled) Q, K, X; the d^(-1/4) scaling is applied inside.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "favor_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_favor_oracle.so")
_lib = None
_lock = threading.Lock()

KINDS = {"exp": 0, "relu": 1}
STABS = {"none": 0, "row": 1, "head": 2}
ATT_MODES = {"canonical": 0, "none": 1, "bound": 2}


def build_library(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math). Returns the library path."""
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
            vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_features.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, dbl, i32]
            for name in ("oracle_noncausal", "oracle_causal"):
                getattr(lib, name).argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, dbl, i32]
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_get_threads.restype = i32
            _lib = lib
    return _lib


def set_threads(t: int) -> None:
    _load().oracle_set_threads(int(t))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _heads(X: np.ndarray) -> tuple[int, int, int]:
    if X.ndim < 2:
        raise ValueError("expected [..., n, d]")
    n, d = X.shape[-2], X.shape[-1]
    return int(np.prod(X.shape[:-2], dtype=np.int64)), n, d


def features(X, omega, *, kind: str = "exp", relu_eps: float = 1e-3, stab: str = "row") -> np.ndarray:
    """phi(X) for X [..., n, d] and Omega [m, d] -> [..., n, m] (fp64)."""
    X, omega = _f64(X), _f64(omega)
    nh, n, d = _heads(X)
    m = omega.shape[0]
    if omega.shape[1] != d:
        raise ValueError("Omega must be m x d")
    out = np.empty(X.shape[:-1] + (m,), np.float64)
    _load().oracle_features(_ptr(X), _ptr(omega), _ptr(out), nh, n, d, m, KINDS[kind], relu_eps, STABS[stab])
    return out


def _attn(fn_name, Q, K, V, omega, kind, relu_eps, mode):
    Q, K, V, omega = _f64(Q), _f64(K), _f64(V), _f64(omega)
    if not (Q.shape == K.shape == V.shape):
        raise ValueError("Q, K, V must have the same [..., n, d] shape")
    nh, n, d = _heads(Q)
    m = omega.shape[0]
    if omega.shape[1] != d:
        raise ValueError("Omega must be m x d")
    Y = np.empty_like(Q)
    getattr(_load(), fn_name)(_ptr(Q), _ptr(K), _ptr(V), _ptr(omega), _ptr(Y), nh, n, d, m,
                              KINDS[kind], relu_eps, ATT_MODES[mode])
    return Y


def attn_noncausal(Q, K, V, omega, *, kind: str = "exp", relu_eps: float = 1e-3, mode: str = "canonical"):
    """Non-causal FAVOR+ attention, Y = Phi(Q) S / Phi(Q) z with S = Phi(K)^T V, z = Phi(K)^T 1."""
    return _attn("oracle_noncausal", Q, K, V, omega, kind, relu_eps, mode)


def attn_causal(Q, K, V, omega, *, kind: str = "exp", relu_eps: float = 1e-3, mode: str = "canonical"):
    """Causal FAVOR+ attention by the per-token prefix-sum recurrence (j <= i)."""
    return _attn("oracle_causal", Q, K, V, omega, kind, relu_eps, mode)


def attn_quadratic(Q, K, V, omega, *, causal: bool, kind: str = "exp", relu_eps: float = 1e-3):
    """Explicit n x n form: A = Phi(Q) Phi(K)^T (lower-triangular if causal), Y = (A V) / (A 1).

    Phi(Q) uses per-row stabilisers and Phi(K) one per head, so A itself is a positive scalar
    multiple of the unstabilised kernel matrix in every row; the row normalisation removes it.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    PQ = features(Q, omega, kind=kind, relu_eps=relu_eps, stab="row")
    PK = features(K, omega, kind=kind, relu_eps=relu_eps, stab="head")
    A = PQ @ np.swapaxes(PK, -1, -2)
    if causal:
        A = np.tril(A)
    return (A @ V) / A.sum(axis=-1, keepdims=True)


def implied_attention(Q, K, omega, *, causal: bool, kind: str = "exp", relu_eps: float = 1e-3):
    """Row-normalised attention matrix FAVOR+ implies (tiny inputs only)."""
    PQ = features(Q, omega, kind=kind, relu_eps=relu_eps, stab="row")
    PK = features(K, omega, kind=kind, relu_eps=relu_eps, stab="head")
    A = PQ @ np.swapaxes(PK, -1, -2)
    if causal:
        A = np.tril(A)
    return A / A.sum(axis=-1, keepdims=True)


def softmax_attention(Q, K, V, *, causal: bool = False):
    """Exact softmax(Q K^T / sqrt(d)) V with max subtraction (the operator being approximated)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    d = Q.shape[-1]
    s = (Q @ np.swapaxes(K, -1, -2)) / np.sqrt(d)
    if causal:
        n = s.shape[-1]
        s = np.where(np.tril(np.ones((n, n), bool)), s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return (e / e.sum(axis=-1, keepdims=True)) @ V


def omega_orf(seed: int, m: int, d: int, *, orthogonal: bool = True) -> np.ndarray:
    """The random projection Omega [m, d] in fp64, as the device builder defines it.

    Orthogonal random features ("Performer for vision", *What Is Performer?*, Orthogonal Features;
    the "Performer" paper note, FAVOR+ section): for each block b of d rows, G_b is a d x d matrix of
    N(0, 1) draws (element (b d + r) d + c of the generator's stream 4); its rows are orthonormalised
    in order (row r minus its components along the already finished rows 0 .. r-1, one at a time,
    then divided by its length); row r of Omega is that unit row times chi_r, the length of the
    d draws r d .. r d + d - 1 of stream 5, so that it is again marginally N(0, I_d). The last block
    keeps its first m - b d rows. orthogonal=False: the m iid Gaussian rows themselves.
    The draws come from ``seeded_inputs.normal``; everything else is written out here.
    """
    import seeded_inputs as si

    if m < 0 or d <= 0:
        raise ValueError("m must be >= 0 and d > 0")
    nblk = -(-m // d)
    G = si.normal(seed, 4, nblk * d * d).reshape(nblk, d, d)
    if not orthogonal:
        return np.ascontiguousarray(G.reshape(nblk * d, d)[:m])
    E = np.empty_like(G)
    for b in range(nblk):
        for r in range(d):
            v = G[b, r].copy()
            for j in range(r):
                v = v - np.dot(v, E[b, j]) * E[b, j]
            E[b, r] = v / np.sqrt(np.dot(v, v))
    x = si.normal(seed, 5, m * d).reshape(m, d)
    chi = np.sqrt(np.einsum("rc,rc->r", x, x))
    return np.ascontiguousarray(E.reshape(nblk * d, d)[:m] * chi[:, None])


def elu1_features(X) -> np.ndarray:
    """phi(x) = elu(x) + 1 elementwise (x for x > 0 plus 1, exp(x) for x <= 0), feature dimension d.

    The Linear Transformer's feature map, as the comparison table of the question page "How do linear
    attention variants (Performer, Linformer) achieve O(n) complexity, and what's the quality cost?"
    and "Performer for vision", *Kernel Choices*, name it: deterministic, positive, no projection.
    Applied to the raw q and k (no d^(-1/4) scaling: the map defines its own kernel phi(q)^T phi(k)
    and approximates nothing).
    """
    X = _f64(X)
    return np.where(X > 0.0, X + 1.0, np.exp(np.minimum(X, 0.0)))


def attn_linear_elu(Q, K, V, *, causal: bool) -> np.ndarray:
    """Linear attention with phi = elu + 1: Y = phi(Q) (phi(K)^T V) / phi(Q) (phi(K)^T 1).

    The associativity form ("Linear Attention and the Performer", *The kernelization trick*;
    "Performer for vision", *How It Works*, Step 1): the d x d state phi(K)^T V and the d-vector
    phi(K)^T 1 first, then one product per query. Causal: the same with the keys j <= i, by
    cumulative sums over the tokens (Step 2, prefix sums). [..., n, d] inputs.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    PQ, PK = elu1_features(Q), elu1_features(K)
    if not causal:
        S = np.swapaxes(PK, -1, -2) @ V          # [..., d, d_v]
        z = PK.sum(axis=-2)                       # [..., d]
        return (PQ @ S) / (PQ @ z[..., None])
    S = np.cumsum(PK[..., :, :, None] * V[..., :, None, :], axis=-3)   # [..., n, d, d_v]
    z = np.cumsum(PK, axis=-2)                                        # [..., n, d]
    num = np.einsum("...ir,...irc->...ic", PQ, S)
    den = np.einsum("...ir,...ir->...i", PQ, z)
    return num / den[..., None]
