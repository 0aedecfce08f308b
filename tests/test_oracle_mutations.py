"""The oracle's pins catch plausible mistakes (CPU only).

Each case compiles a copy of the fp64 oracle with one planted mistake (a dropped term, a wrong scale
or sign, a shifted index, a transposed operand, a missing denominator), swaps it in for the real one
and checks that the facts the pins test no longer hold; the unmodified source, built the same way,
passes the same checks. The mistakes live only in temporary copies; the oracle itself is untouched.
"""
import contextlib
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
import seeded_inputs as si

SRC = os.path.join(os.path.dirname(oracle.__file__), "favor_oracle.c")

MUTATIONS = {
    # exponents u_r = w_r^T x^ without the -|x^|^2/2 correction
    "dropped_norm_term": ("    for (int r = 0; r < m; ++r) u[r] -= h;", "    for (int r = 0; r < m; ++r) u[r] -= 0.0 * h;"),
    # queries and keys scaled by d^(-1/2) instead of d^(-1/4)
    "wrong_scale": ("static void project(const double* x, const double* omega, int d, int m, double* proj, double* half_norm2) {\n"
                    "    const double s = pow((double)d, -0.25);",
                    "static void project(const double* x, const double* omega, int d, int m, double* proj, double* half_norm2) {\n"
                    "    const double s = pow((double)d, -0.5);"),
    # exp(-u) instead of exp(u)
    "wrong_sign": ("phi[r] = exp(phi[r] - stab) * inv_sqrt_m;", "phi[r] = exp(-phi[r] - stab) * inv_sqrt_m;"),
    # the causal scan reads the previous token's key
    "shifted_key_index": ("            feature_row(Kh + i * d, omega, d, m, kind, relu_eps, ks, phi);",
                          "            feature_row(Kh + (i > 0 ? i - 1 : 0) * d, omega, d, m, kind, relu_eps, ks, phi);"),
    # the readout takes S (m x d) as if it were d x m
    "transposed_state": ("num += phi[r] * S[(int64_t)r * d + c];\n                Yh[i * d + c] = num / den;\n            }\n        }\n"
                         "        free(S); free(z); free(phi); free(tmp);\n    }\n}\n\n/*\n * Causal",
                         "num += phi[r] * S[((int64_t)c * m + r) % ((int64_t)m * d)];\n                Yh[i * d + c] = num / den;\n"
                         "            }\n        }\n        free(S); free(z); free(phi); free(tmp);\n    }\n}\n\n/*\n * Causal"),
    # non-causal output not divided by the normaliser
    "missing_denominator": ("                Yh[i * d + c] = num / den;\n            }\n        }\n        free(S); free(z); free(phi); free(tmp);\n    }\n}\n\n/*\n * Causal",
                            "                Yh[i * d + c] = num + 0.0 * den;\n            }\n        }\n        free(S); free(z); free(phi); free(tmp);\n    }\n}\n\n/*\n * Causal"),
}


def build_variant(tmp_path, name, mutation):
    src = open(SRC).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) == 1, f"mutation site of {name} not found exactly once"
        src = src.replace(old, new)
    c_file = tmp_path / f"{name}.c"
    c_file.write_text(src)
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(c_file), "-lm"])
    lib = ctypes.CDLL(str(so))
    vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_features.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, dbl, i32]
    for fn in ("oracle_noncausal", "oracle_causal"):
        getattr(lib, fn).argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, dbl, i32]
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_get_threads.restype = i32
    return lib


@contextlib.contextmanager
def oracle_library(lib):
    oracle._load()  # the real library is loaded (and stays cached) before it is swapped out
    saved = oracle._lib
    oracle._lib = lib
    try:
        yield
    finally:
        oracle._lib = saved


def pin_failures() -> list[str]:
    """The facts the pins check, evaluated on whichever library the oracle currently uses."""
    g = np.random.default_rng(7)
    failures = []
    # unbiasedness: E_w[phi(q)^T phi(k)] = exp(q^T k / sqrt(d)) for raw q, k (Monte Carlo over Omega)
    d, T = 16, 2500
    qh = g.standard_normal(d); qh *= 0.8 / np.linalg.norm(qh)
    kh = g.standard_normal(d); kh *= 0.6 / np.linalg.norm(kh)
    q, k = qh * d ** 0.25, kh * d ** 0.25
    om = si.build_omega(55, T * d, d)
    pq = oracle.features(q[None, None], om, stab="none")[0, 0]
    pk = oracle.features(k[None, None], om, stab="none")[0, 0]
    if abs(float(pq @ pk) / math.exp(float(q @ k) / math.sqrt(d)) - 1.0) > 0.02:
        failures.append("unbiased")
    # the linear forms equal the explicit n x n forms (non-causal and causally masked)
    n, d, m = 9, 8, 24
    omq = si.build_omega(3, m, d)
    Q, K, V = g.standard_normal((2, n, d)), g.standard_normal((2, n, d)), g.standard_normal((2, n, d))
    for causal, fn in ((False, oracle.attn_noncausal), (True, oracle.attn_causal)):
        lin = fn(Q, K, V, omq)
        quad = oracle.attn_quadratic(Q, K, V, omq, causal=causal)
        if not np.allclose(lin, quad, rtol=1e-9, atol=1e-12):
            failures.append(f"quadratic_{'causal' if causal else 'noncausal'}")
    # constant values pass through; the first causal token attends to itself only
    Vc = np.broadcast_to(g.standard_normal(d), (2, n, d)).copy()
    for name, fn in (("noncausal", oracle.attn_noncausal), ("causal", oracle.attn_causal)):
        if not np.allclose(fn(Q, K, Vc, omq), Vc, rtol=1e-9, atol=1e-12):
            failures.append(f"constant_{name}")
    if not np.allclose(oracle.attn_causal(Q, K, V, omq)[:, 0], V[:, 0], rtol=1e-9, atol=1e-12):
        failures.append("first_token")
    return failures


def test_unmodified_source_passes_every_check(tmp_path):
    with oracle_library(build_variant(tmp_path, "control", None)):
        assert pin_failures() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    with oracle_library(build_variant(tmp_path, name, MUTATIONS[name])):
        failed = pin_failures()
    assert failed, f"planted mistake {name} passed every pin check"


# ---------------------------------------------------------------------------------------------
# The Python parts of the oracle (Omega builder, elu + 1 attention): their source with one planted
# mistake, executed in a scratch namespace, fails the facts their pins check.
# ---------------------------------------------------------------------------------------------

def mutated(fn_name, old, new):
    import inspect

    src = inspect.getsource(getattr(oracle, fn_name))
    if old is not None:
        assert src.count(old) == 1, f"mutation site in {fn_name} not found exactly once"
        src = src.replace(old, new)
    ns = dict(vars(oracle))
    exec(compile(src, f"<mutated {fn_name}>", "exec"), ns)
    return ns[fn_name], ns


def omega_failures(omega_fn) -> list[str]:
    with np.errstate(all="ignore"):  # a mutated builder may overflow; the checks still decide
        return _omega_failures(omega_fn)


def _omega_failures(omega_fn) -> list[str]:
    failures = []
    seed, m, d = 11, 130, 64
    om = omega_fn(seed, m, d)
    nblk = -(-m // d)
    G = si.normal(seed, 4, nblk * d * d).reshape(nblk, d, d)
    E = om / np.linalg.norm(om, axis=1, keepdims=True)
    for b in range(nblk):
        Qr, Rr = np.linalg.qr(G[b].T)
        rows = min(d, m - b * d)
        if np.abs(E[b * d:b * d + rows] - ((Qr * np.sign(np.diag(Rr))[None, :]).T)[:rows]).max() > 1e-10:
            failures.append("qr")
            break
    chi = np.linalg.norm(si.normal(seed, 5, m * d).reshape(m, d), axis=1)
    if not np.allclose(np.linalg.norm(om, axis=1), chi, rtol=1e-12):
        failures.append("chi")
    return failures


OMEGA_MUTATIONS = {
    "classical_step_uses_raw_row": ("v = v - np.dot(v, E[b, j]) * E[b, j]", "v = v - np.dot(G[b, r], E[b, j]) * E[b, j] * 0.999"),
    "no_normalisation": ("E[b, r] = v / np.sqrt(np.dot(v, v))", "E[b, r] = v"),
    "chi_from_wrong_stream": ("x = si.normal(seed, 5, m * d)", "x = si.normal(seed, 4, m * d)"),
    "columns_instead_of_rows": ("v = G[b, r].copy()", "v = G[b, :, r].copy()"),
}


def test_unmodified_omega_source_passes():
    fn, _ = mutated("omega_orf", None, None)
    assert omega_failures(fn) == []


@pytest.mark.parametrize("name", sorted(OMEGA_MUTATIONS))
def test_planted_omega_mistake_is_caught(name):
    fn, _ = mutated("omega_orf", *OMEGA_MUTATIONS[name])
    with np.errstate(all="ignore"):
        assert omega_failures(fn), f"planted mistake {name} passed the Omega pins"


def elu_failures(features_fn, attn_fn) -> list[str]:
    try:
        with np.errstate(all="ignore"):
            return _elu_failures(features_fn, attn_fn)
    except (ValueError, FloatingPointError) as e:  # a mistake that breaks the shapes fails the pins too
        return [f"error: {e}"]


def _elu_failures(features_fn, attn_fn) -> list[str]:
    import torch

    failures = []
    x = np.linspace(-6, 6, 241)
    ref = torch.nn.functional.elu(torch.from_numpy(x)).numpy() + 1.0
    if not np.allclose(features_fn(x), ref, rtol=1e-15, atol=2.0**-53):
        failures.append("library_elu")
    e = math.exp(-1.0)
    y = attn_fn(np.array([[0.5]]), np.array([[1.0], [-1.0]]), np.array([[2.0], [4.0]]), causal=False)
    if abs(y[0, 0] - (4.0 + 4.0 * e) / (2.0 + e)) > 1e-15:
        failures.append("hand_example")
    yc = attn_fn(np.array([[0.5], [-2.0]]), np.array([[1.0], [-1.0]]), np.array([[2.0], [4.0]]), causal=True)
    if not (abs(yc[0, 0] - 2.0) < 1e-15):
        failures.append("first_token")
    return failures


ELU_MUTATIONS = {
    "without_plus_one": ("elu1_features", "X + 1.0, np.exp(np.minimum(X, 0.0))", "X, np.exp(np.minimum(X, 0.0)) - 1.0"),
    "relu_plus_one": ("elu1_features", "np.exp(np.minimum(X, 0.0))", "np.ones_like(X)"),
    "exclusive_prefix": ("attn_linear_elu", "S = np.cumsum(PK[..., :, :, None] * V[..., :, None, :], axis=-3)",
                         "S = np.cumsum(PK[..., :, :, None] * V[..., :, None, :], axis=-3) - PK[..., :, :, None] * V[..., :, None, :]"),
    "keys_as_queries": ("attn_linear_elu", "S = np.swapaxes(PK, -1, -2) @ V", "S = np.swapaxes(PQ, -1, -2) @ V"),
}


def test_unmodified_elu_source_passes():
    feat, _ = mutated("elu1_features", None, None)
    attn, _ = mutated("attn_linear_elu", None, None)
    assert elu_failures(feat, attn) == []


@pytest.mark.parametrize("name", sorted(ELU_MUTATIONS))
def test_planted_elu_mistake_is_caught(name):
    target, old, new = ELU_MUTATIONS[name]
    if target == "elu1_features":
        feat, _ = mutated("elu1_features", old, new)
        _, ns2 = mutated("attn_linear_elu", None, None)
        ns2["elu1_features"] = feat          # the attention uses the mutated feature map
        attn = ns2["attn_linear_elu"]
    else:
        feat = oracle.elu1_features
        attn, _ = mutated("attn_linear_elu", old, new)
    assert elu_failures(feat, attn), f"planted mistake {name} passed the elu pins"
