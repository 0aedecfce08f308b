"""The debug build of the library (libfavor_debug.so, compiled with -DFAVOR_DEBUG; FAVOR_DEBUG=1 makes
the binding load it): every computed-address access of the tensor-core kernels to global, shared and
ring memory is checked against its buffer, and a failed check is recorded as FAVOR_ERR_BOUNDS in the
device error word instead of touching memory. It stands in for a memory checker. The small and
ragged parity cases run under it in a child process: each of them asserts that the device error
word is clear after its call, so a failed check fails the case."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(args, timeout):
    env = dict(os.environ, FAVOR_DEBUG="1")
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_the_debug_build_is_the_one_loaded():
    r = _child(["-c", "import kernelized_linear_attention_04_b300 as f; print(f.LIB_PATH)"], 600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().endswith("libfavor_debug.so"), r.stdout


def test_small_parity_cases_under_the_debug_build(cuda_device):
    r = _child(["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                os.path.join("tests", "test_gpu_parity.py"), os.path.join("tests", "test_gpu_elu.py"),
                os.path.join("tests", "test_gpu_exact.py"),
                "-k", "small_cases or feature_groups or noncausal_paths or large_norm or matches_oracle"], 1500)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
