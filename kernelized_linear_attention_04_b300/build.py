"""Builds libfavor.so in-tree with nvcc for sm_103a.

    python -m kernelized_linear_attention_04_b300.build [--force] [--verbose] [--debug]

--debug (or FAVOR_DEBUG=1 in the environment, which also makes the Python binding load it) builds
libfavor_debug.so with -DFAVOR_DEBUG: every computed-index device access is checked against its
buffer, and a failed check is reported as FAVOR_ERR_BOUNDS instead of touching memory.
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
DEBUG = os.environ.get("FAVOR_DEBUG", "") == "1"
LIB_RELEASE = os.path.join(HERE, "libfavor.so")
LIB_DEBUG = os.path.join(HERE, "libfavor_debug.so")
LIB = LIB_DEBUG if DEBUG else LIB_RELEASE
MAIN = os.path.join(CSRC, "favor_api.cu")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
    "-I", os.path.join(ROOT, "include"),
]


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + [os.path.join(ROOT, "include", "favor.h")])


def is_stale(debug: bool = DEBUG) -> bool:
    lib = LIB_DEBUG if debug else LIB_RELEASE
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in _sources())


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False, debug: bool = DEBUG) -> str:
    """Compile (if stale or forced) and return the library path (the debug variant if `debug`)."""
    lib = LIB_DEBUG if debug else LIB_RELEASE
    if not force and not is_stale(debug):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *(["-DFAVOR_DEBUG"] if debug else []), *(["-Xptxas", "-v"] if verbose else []),
           "-o", tmp, MAIN]
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="pass -Xptxas -v (registers, spills, smem)")
    ap.add_argument("--debug", action="store_true", help="build libfavor_debug.so (device bounds checks)")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug=a.debug or DEBUG))
    sys.exit(0)
