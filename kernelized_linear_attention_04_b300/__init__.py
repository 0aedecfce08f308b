"""FAVOR+ (Performer) attention forward pass on B300: thin Python binding over libfavor.so.

Every step of the computation runs in the library's CUDA kernels; this module only marshals torch
tensors (device memory, streams) into the C ABI declared in ``include/favor.h``. There is no CPU
path: if the library cannot be loaded, importing this package raises.

    import kernelized_linear_attention_04_b300 as favor
    Y = favor.favor_attn_noncausal(Q, K, V, Omega)            # [B, H, n, d] bf16/fp32 CUDA tensors
    Y = favor.favor_attn_causal(Q, K, V, Omega, chunk=64)
    Phi = favor.favor_features(X, Omega, stab="head")
    state = favor.decode_state(B, H, d, m, device)             # streaming decode, one token per step
    y = favor.favor_decode_step(q, k, v, Omega, state)         # q, k, v: [B, H, d]
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "FavorError", "favor_features", "favor_attn_noncausal", "favor_attn_causal", "favor_attn_noncausal_noalloc",
    "favor_softmax_attn",
    "workspace_bytes", "NOALLOC_SCRATCH_BYTES",
    "decode_state_bytes", "decode_state", "favor_decode_init", "favor_decode_step", "favor_omega",
    "last_device_error", "trace_enable", "trace_read", "abi_version", "lib", "LIB_PATH",
    "KERNEL_NAMES", "EXPORTED_SYMBOLS",
]

LIB_PATH = _build.LIB

_DTYPES = {torch.float32: 0, torch.bfloat16: 1}
_KINDS = {"exp": 0, "relu": 1, "elu": 2}
_STABS = {"none": 0, "row": 1, "head": 2}
_OPS = {"features": 0, "noncausal": 1, "causal": 2}
_STATUS = {0: "FAVOR_OK", 1: "FAVOR_ERR_INVALID_ARG", 2: "FAVOR_ERR_UNSUPPORTED", 3: "FAVOR_ERR_MISALIGNED",
           4: "FAVOR_ERR_WORKSPACE", 5: "FAVOR_ERR_CUDA", 6: "FAVOR_ERR_TIMEOUT", 7: "FAVOR_ERR_BOUNDS"}
KERNEL_COUNT = 11
# Size of the library's fixed scratch array used by favor_attn_noncausal_noalloc.
NOALLOC_SCRATCH_BYTES = 16 << 20

# Every function include/favor.h declares.
EXPORTED_SYMBOLS = (
    "favor_workspace_bytes", "favor_features", "favor_attn_noncausal", "favor_attn_causal",
    "favor_status_string", "favor_last_device_error", "favor_abi_version", "favor_trace_enable",
    "favor_trace_read", "favor_kernel_name", "favor_attn_noncausal_noalloc",
    "favor_decode_state_bytes", "favor_decode_init", "favor_decode_step", "favor_omega",
    "favor_test_set_wait_limit", "favor_softmax_attn",
)


class FavorError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.favor_status_string(status).decode() if lib is not None else _STATUS.get(status, str(status))
        super().__init__(f"{where}: {msg}")


def _load() -> ctypes.CDLL:
    path = _build.build() if _build.is_stale() else LIB_PATH  # fails loudly if it cannot build
    L = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.favor_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32]
    L.favor_workspace_bytes.restype = sz
    L.favor_features.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    L.favor_features.restype = i32
    L.favor_attn_noncausal.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp]
    L.favor_attn_noncausal.restype = i32
    L.favor_attn_causal.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp]
    L.favor_attn_causal.restype = i32
    L.favor_attn_noncausal_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp]
    L.favor_attn_noncausal_noalloc.restype = i32
    L.favor_status_string.argtypes = [i32]
    L.favor_status_string.restype = ctypes.c_char_p
    L.favor_last_device_error.argtypes = [vp]
    L.favor_last_device_error.restype = i32
    L.favor_abi_version.restype = i32
    L.favor_trace_enable.argtypes = [i32]
    L.favor_trace_enable.restype = i32
    L.favor_trace_read.argtypes = [vp, vp]
    L.favor_trace_read.restype = i32
    L.favor_kernel_name.argtypes = [i32]
    L.favor_kernel_name.restype = ctypes.c_char_p
    L.favor_decode_state_bytes.argtypes = [i32, i32, i32, i32]
    L.favor_decode_state_bytes.restype = sz
    L.favor_decode_init.argtypes = [vp, sz, i32, i32, i32, i32, vp]
    L.favor_decode_init.restype = i32
    L.favor_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, sz, i32, i32, i32, i32, i32, i32, f32, vp]
    L.favor_decode_step.restype = i32
    L.favor_omega.argtypes = [ctypes.c_uint64, i32, i32, i32, i32, vp, vp]
    L.favor_omega.restype = i32
    L.favor_softmax_attn.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    L.favor_softmax_attn.restype = i32
    L.favor_test_set_wait_limit.argtypes = [ctypes.c_ulonglong, vp]
    L.favor_test_set_wait_limit.restype = i32
    return L


lib: ctypes.CDLL = _load()
KERNEL_NAMES = tuple(lib.favor_kernel_name(i).decode() for i in range(KERNEL_COUNT))


def abi_version() -> int:
    return int(lib.favor_abi_version())


def _check(status: int, where: str) -> None:
    if status != 0:
        raise FavorError(status, where)


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _require_cuda(**tensors) -> None:
    """Every given tensor must live on the current CUDA device: the kernels launch there and take
    raw pointers, so a host tensor or another GPU's memory is rejected here, before any launch."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other tensors on {dev}")
    if dev is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"the tensors are on {dev} but the current CUDA device is {torch.cuda.current_device()}")


def _dims(X: torch.Tensor, name: str) -> tuple[int, int, int, int]:
    if X.dim() != 4:
        raise ValueError(f"{name} must be [B, H, n, d], got shape {tuple(X.shape)}")
    if not X.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if X.dtype not in _DTYPES:
        raise TypeError(f"{name} must be float32 or bfloat16, got {X.dtype}")
    return tuple(int(s) for s in X.shape)  # type: ignore[return-value]


def workspace_bytes(op: str, B: int, H: int, n: int, d: int, m: int, dtype: torch.dtype, *, kind: str = "exp",
                    stab: str = "row", chunk: int = 0) -> int:
    """Workspace bytes a call needs (raises FavorError(UNSUPPORTED) for shapes the library rejects)."""
    v = lib.favor_workspace_bytes(_OPS[op], B, H, n, d, m, _DTYPES[dtype], _KINDS[kind], _STABS[stab], chunk)
    if v == ctypes.c_size_t(-1).value:
        raise FavorError(2, "favor_workspace_bytes")
    return int(v)


def _workspace(nbytes: int, like: torch.Tensor, workspace):
    if nbytes == 0:
        return workspace, 0 if workspace is None else workspace.numel() * workspace.element_size()
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=like.device)
    return workspace, workspace.numel() * workspace.element_size()


def favor_features(X: torch.Tensor, Omega: torch.Tensor | None, *, kind: str = "exp", relu_eps: float = 1e-3,
                   stab: str = "row", out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """phi(X) as fp32 [B, H, n, m] for raw X [B, H, n, d] and Omega [m, d] (same dtype). kind="elu":
    phi = elu(X) + 1 with m = d; Omega is not used (pass None)."""
    B, H, n, d = _dims(X, "X")
    m = d if kind == "elu" else int(Omega.shape[0])
    if kind == "elu":
        Omega = None
    if out is None:
        out = torch.empty((B, H, n, m), dtype=torch.float32, device=X.device)
    ws, wsb = _workspace(workspace_bytes("features", B, H, n, d, m, X.dtype, kind=kind, stab=stab), X, workspace)
    _require_cuda(X=X, Omega=Omega, out=out, workspace=ws)
    _check(lib.favor_features(_ptr(X), _ptr(Omega), _ptr(out), B, H, n, d, m, _DTYPES[X.dtype], _KINDS[kind],
                              relu_eps, _STABS[stab], _ptr(ws), wsb, _stream_handle(stream)), "favor_features")
    return out


def _attn_prep(Q, K, V, Omega, out, kind="exp"):
    B, H, n, d = _dims(Q, "Q")
    if K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("Q, K, V must have the same shape")
    if out is None:
        out = torch.empty_like(Q)
    if kind == "elu":  # elu + 1 features: feature dimension d, no projection (Omega is not used)
        if not (Q.dtype == K.dtype == V.dtype):
            raise TypeError("Q, K and V must share one dtype")
        return B, H, n, d, d, out
    if not (Q.dtype == K.dtype == V.dtype == Omega.dtype):
        raise TypeError("Q, K, V and Omega must share one dtype")
    if Omega.dim() != 2 or Omega.shape[1] != d or not Omega.is_contiguous():
        raise ValueError("Omega must be a contiguous [m, d] tensor")
    return B, H, n, d, int(Omega.shape[0]), out


def favor_attn_noncausal(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, Omega: torch.Tensor | None, *,
                         kind: str = "exp", relu_eps: float = 1e-3, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = Phi(Q)(Phi(K)^T V) / Phi(Q)(Phi(K)^T 1), all keys."""
    B, H, n, d, m, out = _attn_prep(Q, K, V, Omega, out, kind)
    Omega = None if kind == "elu" else Omega
    ws, wsb = _workspace(workspace_bytes("noncausal", B, H, n, d, m, Q.dtype, kind=kind), Q, workspace)
    _require_cuda(Q=Q, K=K, V=V, Omega=Omega, out=out, workspace=ws)
    _check(lib.favor_attn_noncausal(_ptr(Q), _ptr(K), _ptr(V), _ptr(Omega), _ptr(out), B, H, n, d, m,
                                    _DTYPES[Q.dtype], _KINDS[kind], relu_eps, _ptr(ws), wsb, _stream_handle(stream)),
           "favor_attn_noncausal")
    return out


def favor_attn_causal(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, Omega: torch.Tensor | None, *, chunk: int = 64,
                      kind: str = "exp", relu_eps: float = 1e-3, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal FAVOR+ attention (keys j <= i) as a chunked prefix-sum scan."""
    B, H, n, d, m, out = _attn_prep(Q, K, V, Omega, out, kind)
    Omega = None if kind == "elu" else Omega
    ws, wsb = _workspace(workspace_bytes("causal", B, H, n, d, m, Q.dtype, kind=kind, chunk=chunk), Q, workspace)
    _require_cuda(Q=Q, K=K, V=V, Omega=Omega, out=out, workspace=ws)
    _check(lib.favor_attn_causal(_ptr(Q), _ptr(K), _ptr(V), _ptr(Omega), _ptr(out), B, H, n, d, m, chunk,
                                 _DTYPES[Q.dtype], _KINDS[kind], relu_eps, _ptr(ws), wsb, _stream_handle(stream)),
           "favor_attn_causal")
    return out


def favor_softmax_attn(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, causal: bool = False,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exact softmax(Q K^T / sqrt(d)) V (the operator FAVOR+ approximates), O(n^2 d) work; bf16,
    d = 64. For speed and divergence comparisons."""
    B, H, n, d = _dims(Q, "Q")
    if K.shape != Q.shape or V.shape != Q.shape or not (Q.dtype == K.dtype == V.dtype):
        raise ValueError("Q, K, V must have the same shape and dtype")
    if out is None:
        out = torch.empty_like(Q)
    _require_cuda(Q=Q, K=K, V=V, out=out)
    _check(lib.favor_softmax_attn(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, n, d, 1 if causal else 0,
                                  _DTYPES[Q.dtype], _stream_handle(stream)), "favor_softmax_attn")
    return out


def favor_attn_noncausal_noalloc(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, Omega: torch.Tensor | None, *,
                                 kind: str = "exp", relu_eps: float = 1e-3, out: torch.Tensor | None = None,
                                 stream=None) -> torch.Tensor:
    """Same result as favor_attn_noncausal, for callers that cannot allocate device scratch.

    The library keeps the scratch in one fixed device array of NOALLOC_SCRATCH_BYTES, so this call
    allocates nothing on the device (pass `out` to avoid even the output allocation here). Calls
    share that array: do not let two of them overlap on the GPU. Make the first call on a device
    outside stream capture (it looks up the array's address).
    """
    B, H, n, d, m, out = _attn_prep(Q, K, V, Omega, out, kind)
    Omega = None if kind == "elu" else Omega
    _require_cuda(Q=Q, K=K, V=V, Omega=Omega, out=out)
    _check(lib.favor_attn_noncausal_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(Omega), _ptr(out), B, H, n, d, m,
                                            _DTYPES[Q.dtype], _KINDS[kind], relu_eps, _stream_handle(stream)),
           "favor_attn_noncausal_noalloc")
    return out


def last_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status (0 = none)."""
    return int(lib.favor_last_device_error(_stream_handle(stream)))


def trace_enable(on: bool = True) -> None:
    _check(lib.favor_trace_enable(1 if on else 0), "favor_trace_enable")


def trace_read() -> dict[str, tuple[int, float]]:
    """{kernel name: (launches, total device ms)} of the launches recorded since trace_enable(True)."""
    launches = (ctypes.c_int * KERNEL_COUNT)()
    total = (ctypes.c_double * KERNEL_COUNT)()
    _check(lib.favor_trace_read(ctypes.cast(launches, ctypes.c_void_p), ctypes.cast(total, ctypes.c_void_p)),
           "favor_trace_read")
    return {KERNEL_NAMES[i]: (int(launches[i]), float(total[i])) for i in range(KERNEL_COUNT)}


# ---- streaming decode ------------------------------------------------------------------------------

def decode_state_bytes(B: int, H: int, d: int, m: int) -> int:
    """Bytes of the decode state of B*H heads (raises FavorError(UNSUPPORTED) for unsupported d, m)."""
    v = lib.favor_decode_state_bytes(B, H, d, m)
    if v == ctypes.c_size_t(-1).value:
        raise FavorError(2, "favor_decode_state_bytes")
    return int(v)


def favor_decode_init(state: torch.Tensor, B: int, H: int, d: int, m: int, stream=None) -> torch.Tensor:
    """Empties the decode state (no token seen) of every head."""
    _require_cuda(state=state)
    _check(lib.favor_decode_init(_ptr(state), state.numel() * state.element_size(), B, H, d, m,
                                 _stream_handle(stream)), "favor_decode_init")
    return state


def decode_state(B: int, H: int, d: int, m: int, device="cuda", stream=None) -> torch.Tensor:
    """A new, empty decode state (a uint8 device buffer owned by the caller)."""
    state = torch.empty(decode_state_bytes(B, H, d, m), dtype=torch.uint8, device=device)
    return favor_decode_init(state, B, H, d, m, stream)


def favor_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, Omega: torch.Tensor | None,
                      state: torch.Tensor, *, kind: str = "exp", relu_eps: float = 1e-3,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Appends one token per head (q, k, v: [B, H, d]) to `state` and returns its output y [B, H, d].
    kind="elu": m = d and Omega is not used (pass None)."""
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if t.dim() != 3 or not t.is_contiguous() or t.dtype not in _DTYPES:
            raise ValueError(f"{name} must be a contiguous [B, H, d] float32/bfloat16 tensor")
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("q, k and v must have the same shape and dtype")
    B, H, d = (int(x) for x in q.shape)
    if kind == "elu":
        Omega, m = None, d
    else:
        if Omega.dim() != 2 or Omega.shape[1] != d or Omega.dtype != q.dtype or not Omega.is_contiguous():
            raise ValueError("Omega must be a contiguous [m, d] tensor of the same dtype as q")
        m = int(Omega.shape[0])
    if out is None:
        out = torch.empty_like(q)
    _require_cuda(q=q, k=k, v=v, Omega=Omega, state=state, out=out)
    _check(lib.favor_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(Omega), _ptr(out), _ptr(state),
                                 state.numel() * state.element_size(), B, H, d, m, _DTYPES[q.dtype], _KINDS[kind],
                                 relu_eps, _stream_handle(stream)), "favor_decode_step")
    return out


# ---- random projection -------------------------------------------------------------------------------

def favor_omega(seed: int, m: int, d: int, *, dtype=torch.bfloat16, orthogonal: bool = True, out=None,
                device="cuda", stream=None) -> torch.Tensor:
    """Omega [m, d] for `seed`, built on the device: orthogonal random features (Gaussian blocks of
    d rows orthonormalised in order, each row scaled to a chi_d length), or iid Gaussian rows."""
    if dtype not in _DTYPES:
        raise TypeError("dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty(m, d, dtype=dtype, device=device)
    elif out.shape != (m, d) or out.dtype != dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous [{m}, {d}] {dtype} tensor")
    _require_cuda(out=out)
    _check(lib.favor_omega(ctypes.c_uint64(int(seed) & (2**64 - 1)), m, d, 1 if orthogonal else 0, _DTYPES[dtype],
                           _ptr(out), _stream_handle(stream)), "favor_omega")
    return out
