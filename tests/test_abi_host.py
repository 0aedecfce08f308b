"""The C-ABI library loads, exports what include/favor.h declares, and rejects bad arguments on the
host before launching anything (CPU; no compute calls)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "favor.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(favor_[a-z_]+)\s*\(", text)))


def test_library_loads_and_exports_every_declared_symbol():
    import kernelized_linear_attention_04_b300 as favor

    decl = declared_functions()
    assert set(decl) == set(favor.EXPORTED_SYMBOLS), decl
    out = subprocess.run(["nm", "-D", "--defined-only", favor.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (favor_\w+)", out))
    for name in decl:
        assert name in exported, name
        assert hasattr(favor.lib, name)
    assert favor.abi_version() == 1


def test_status_strings_and_kernel_names():
    import kernelized_linear_attention_04_b300 as favor

    for code in range(8):
        assert favor.lib.favor_status_string(code).decode().startswith("FAVOR_")
    assert favor.KERNEL_NAMES[0] == "features"
    assert favor.KERNEL_NAMES[-1] == "exact"


def test_workspace_sizes():
    import kernelized_linear_attention_04_b300 as favor

    bf = torch.bfloat16
    assert favor.workspace_bytes("features", 1, 8, 1024, 64, 256, bf, stab="row") == 0
    assert favor.workspace_bytes("features", 1, 8, 1024, 64, 256, bf, stab="head") >= 8 * 4
    assert favor.workspace_bytes("noncausal", 1, 8, 0, 64, 256, bf) == 0
    nc = favor.workspace_bytes("noncausal", 1, 8, 1024, 64, 256, bf)
    assert nc % 256 == 0 and nc >= 8 * (256 * 64 + 256) * 4
    with pytest.raises(favor.FavorError):
        favor.workspace_bytes("noncausal", 1, 8, 1024, 96, 256, bf)
    with pytest.raises(favor.FavorError):
        favor.workspace_bytes("causal", 1, 8, 1024, 64, 256, bf, chunk=48)


def test_workspace_sizes_per_path():
    # Short bf16 sequences (n <= 8 tiles of 128, d = 64, m <= 256) run the single-launch kernel, whose
    # workspace is the per-tile fp32 partial states: [BH][T][m_pad][64] S, [BH][T][2][m_pad] z and
    # [BH][8] stabilisers, each piece rounded up to 256 bytes.
    import kernelized_linear_attention_04_b300 as favor

    bf, f32 = torch.bfloat16, torch.float32
    BH, T, mp = 8, 8, 256
    up = lambda b: (b + 255) // 256 * 256
    fused = up(BH * T * mp * 64 * 4) + up(BH * T * 2 * mp * 4) + up(BH * 8 * 4)
    assert favor.workspace_bytes("noncausal", 1, 8, 1024, 64, 256, bf) == fused
    # m = 192 pads to 256 features
    assert favor.workspace_bytes("noncausal", 1, 8, 1024, 64, 192, bf) == fused
    # one tile per head
    assert favor.workspace_bytes("noncausal", 1, 8, 100, 64, 256, bf) == up(BH * mp * 256) + up(BH * 2 * mp * 4) + up(BH * 32)
    # longer sequences run the three-kernel path, whose workspace does not grow with n beyond the splits
    assert favor.workspace_bytes("noncausal", 1, 8, 4096, 64, 256, bf) > 0
    # the tensor-core causal scans keep the state in TMEM; with more than 128 features the CTAs of a
    # group combine their partial rows through a ring of 4 tiles x CS CTAs x 9 x 128 rows x 16 bytes,
    # after 16 u32 counters per group (256-byte piece), for min(B*H, 160 // CS) groups
    for m in (64, 128):
        assert favor.workspace_bytes("causal", 4, 16, 8192, 64, m, bf) == 0
    for BH, m, cs in ((64, 192, 2), (64, 256, 2), (64, 384, 3), (64, 512, 4), (256, 512, 4), (7, 384, 3),
                      (1000, 512, 4), (1000, 384, 3), (1000, 256, 2)):
        groups = min(BH, 160 // cs)
        assert favor.workspace_bytes("causal", 1, BH, 8192, 64, m, bf) == up(groups * 64) + groups * 4 * cs * 9 * 128 * 16
    # streaming decode state: fp32 S [BH][m][d], z [BH][m], stabilisers [BH][m/64], block partials
    # [BH][m/64][d+2], u32 counter [BH]; 256-byte pieces
    up = lambda b: (b + 255) // 256 * 256
    assert favor.decode_state_bytes(2, 3, 64, 256) == (6 * 256 * 64 * 4 + 6 * 256 * 4 + up(6 * 4 * 4)
                                                       + up(6 * 4 * 66 * 4) + up(6 * 4))
    assert favor.decode_state_bytes(1, 1, 128, 512) == (512 * 128 * 4 + 512 * 4 + up(8 * 4) + up(8 * 130 * 4)
                                                        + up(4))
    with pytest.raises(favor.FavorError):
        favor.decode_state_bytes(1, 1, 96, 256)
    # head-count limits (see include/favor.h): grid-y paths take at most 65535 heads
    assert favor.workspace_bytes("noncausal", 1, 65535, 16, 64, 64, bf) > 0
    with pytest.raises(favor.FavorError):
        favor.workspace_bytes("noncausal", 1, 65536, 16, 64, 64, bf)
    with pytest.raises(favor.FavorError):
        favor.workspace_bytes("features", 2, 40000, 16, 64, 64, bf, stab="head")
    assert favor.workspace_bytes("causal", 1, 65536, 16, 64, 64, bf) == 0
    with pytest.raises(favor.FavorError):
        favor.decode_state_bytes(1 << 13, 1 << 12, 64, 64)
    # fp32, and bf16 with d = 128, take the CUDA-core scan, whose state lives in the workspace
    assert favor.workspace_bytes("causal", 1, 2, 300, 64, 256, f32) >= 2 * (256 * 64 + 256) * 4
    assert favor.workspace_bytes("causal", 1, 2, 300, 128, 256, bf) >= 2 * (256 * 128 + 256) * 4


# Argument checks. Fake (never dereferenced) addresses are only passed where an earlier check
# must fail; to keep even that off a real device these run only without a GPU.
needs_no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks")


@needs_no_gpu
def test_argument_checks_reject_before_launch():
    import kernelized_linear_attention_04_b300 as favor

    L = favor.lib
    P = ctypes.c_void_p(0x10000)      # aligned fake pointer
    Mis = ctypes.c_void_p(0x10008)    # 8-byte aligned only
    N = ctypes.c_void_p(0)
    S = ctypes.c_void_p(0)
    nc = L.favor_attn_noncausal
    # null pointer
    assert nc(P, N, P, P, P, 1, 1, 16, 64, 64, 1, 0, 0.0, P, 1 << 20, S) == 1
    # unsupported d / m
    assert nc(P, P, P, P, P, 1, 1, 16, 96, 64, 1, 0, 0.0, P, 1 << 20, S) == 2
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 100, 1, 0, 0.0, P, 1 << 20, S) == 2
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 1024, 1, 0, 0.0, P, 1 << 20, S) == 2
    # bad enums / sizes / eps
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 64, 7, 0, 0.0, P, 1 << 20, S) == 1
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 64, 1, 5, 0.0, P, 1 << 20, S) == 1
    assert nc(P, P, P, P, P, -1, 1, 16, 64, 64, 1, 0, 0.0, P, 1 << 20, S) == 1
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 64, 1, 1, -1.0, P, 1 << 20, S) == 1
    # misaligned
    assert nc(P, P, Mis, P, P, 1, 1, 16, 64, 64, 1, 0, 0.0, P, 1 << 20, S) == 3
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 64, 1, 0, 0.0, ctypes.c_void_p(0x10010), 1 << 20, S) == 3
    # workspace too small / missing
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 64, 1, 0, 0.0, P, 16, S) == 4
    assert nc(P, P, P, P, P, 1, 1, 16, 64, 64, 1, 0, 0.0, N, 1 << 20, S) == 1
    # empty call is a no-op even with null pointers
    assert nc(N, N, N, N, N, 1, 1, 0, 64, 64, 1, 0, 0.0, N, 0, S) == 0
    assert nc(N, N, N, N, N, 0, 4, 16, 64, 64, 1, 0, 0.0, N, 0, S) == 0
    ca = L.favor_attn_causal
    assert ca(P, P, P, P, P, 1, 1, 16, 64, 64, 32, 1, 0, 0.0, P, 1 << 20, S) == 2
    assert ca(N, N, N, N, N, 1, 1, 0, 64, 64, 64, 1, 0, 0.0, N, 0, S) == 0
    ft = L.favor_features
    assert ft(P, P, N, 1, 1, 16, 64, 64, 1, 0, 0.0, 1, N, 0, S) == 1
    assert ft(P, P, P, 1, 1, 16, 64, 64, 1, 0, 0.0, 9, N, 0, S) == 1
    assert ft(P, P, P, 1, 1, 16, 64, 64, 1, 0, 0.0, 2, N, 0, S) == 1       # head stab needs workspace
    # streaming decode: state checks come after the tensor checks; empty batches are no-ops
    ds = L.favor_decode_step
    need = L.favor_decode_state_bytes(1, 1, 64, 64)
    assert ds(P, N, P, P, P, P, need, 1, 1, 64, 64, 1, 0, 0.0, S) == 1           # null k
    assert ds(P, P, P, P, P, N, need, 1, 1, 64, 64, 1, 0, 0.0, S) == 1           # null state
    assert ds(P, P, P, P, P, ctypes.c_void_p(0x10010), need, 1, 1, 64, 64, 1, 0, 0.0, S) == 3  # state alignment
    assert ds(P, P, P, P, P, P, need - 1, 1, 1, 64, 64, 1, 0, 0.0, S) == 4       # state too small
    assert ds(P, P, P, P, P, P, need, 1, 1, 96, 64, 1, 0, 0.0, S) == 2           # unsupported d
    assert ds(N, N, N, N, N, N, 0, 0, 4, 64, 64, 1, 0, 0.0, S) == 0              # no heads
    di = L.favor_decode_init
    assert di(N, need, 1, 1, 64, 64, S) == 1
    assert di(P, need - 1, 1, 1, 64, 64, S) == 4
    assert di(N, 0, 0, 1, 64, 64, S) == 0
    # head-count limits: rejected before anything is launched (empty calls stay no-ops)
    assert nc(P, P, P, P, P, 65536, 1, 16, 64, 64, 1, 0, 0.0, P, 1 << 30, S) == 2
    assert nc(P, P, P, P, P, 256, 256, 16, 64, 64, 1, 0, 0.0, P, 1 << 30, S) == 2
    assert nc(N, N, N, N, N, 65536, 1, 0, 64, 64, 1, 0, 0.0, N, 0, S) == 0
    assert L.favor_attn_noncausal_noalloc(P, P, P, P, P, 65536, 1, 16, 64, 64, 1, 0, 0.0, S) == 2
    assert ft(P, P, P, 65536, 1, 16, 64, 64, 1, 0, 0.0, 1, N, 0, S) == 2
    assert ca(P, P, P, P, P, 1 << 13, 1 << 12, 16, 64, 64, 64, 1, 0, 0.0, P, 1 << 20, S) == 2
    assert ds(P, P, P, P, P, P, need, 1 << 13, 1 << 12, 64, 64, 1, 0, 0.0, S) == 2
    assert di(P, need, 1 << 13, 1 << 12, 64, 64, S) == 2
    # random projection builder: every failing check comes before the launch; m = 0 is a no-op
    om = L.favor_omega
    assert om(1, 64, 96, 1, 1, P, S) == 2          # unsupported d
    assert om(1, 64, 64, 1, 1, N, S) == 1          # null output
    assert om(1, 64, 64, 1, 1, Mis, S) == 3        # misaligned output
    assert om(1, -1, 64, 1, 1, P, S) == 1          # negative m
    assert om(1, 64, 64, 1, 7, P, S) == 1          # bad dtype
    assert om(1, 0, 64, 1, 1, N, S) == 0           # nothing to build


def test_python_binding_validates_shapes():
    import kernelized_linear_attention_04_b300 as favor

    q = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        favor.favor_attn_noncausal(q, q, q[:, :, :2], torch.zeros(64, 64))
    with pytest.raises(TypeError):
        favor.favor_attn_noncausal(q, q, q, torch.zeros(64, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        favor.favor_attn_noncausal(q[0], q[0], q[0], torch.zeros(64, 64))


def test_python_binding_rejects_host_tensors_before_any_launch():
    # a host pointer handed to a kernel would be an illegal address on the GPU: the binding refuses
    # tensors that are not on the current CUDA device (checked after the shape and dtype checks)
    import kernelized_linear_attention_04_b300 as favor

    q = torch.zeros(1, 1, 4, 64)
    om = torch.zeros(64, 64)
    for fn in (favor.favor_attn_noncausal, favor.favor_attn_causal, favor.favor_attn_noncausal_noalloc):
        with pytest.raises(ValueError, match="CUDA tensor"):
            fn(q, q, q, om)
    with pytest.raises(ValueError, match="CUDA tensor"):
        favor.favor_features(q, om)
    with pytest.raises(ValueError, match="CUDA tensor"):
        favor.favor_omega(1, 64, 64, device="cpu")
    t = torch.zeros(1, 1, 64)
    state = torch.zeros(favor.decode_state_bytes(1, 1, 64, 64), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        favor.favor_decode_init(state, 1, 1, 64, 64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        favor.favor_decode_step(t, t, t, om, state)


def test_plain_c_program_links_and_calls_the_library(tmp_path):
    # the boundary is a C ABI: a C99 program (no Python, no torch) includes the header, links the
    # library and calls its host-side entry points; its answers match the binding's
    import shutil

    import kernelized_linear_attention_04_b300 as favor

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_favor.c"
    src.write_text(r'''
#include <stdio.h>
#include "favor.h"
int main(void) {
    size_t ws = favor_workspace_bytes(FAVOR_OP_NONCAUSAL, 1, 8, 4096, 64, 256, FAVOR_BF16, FAVOR_EXP,
                                      FAVOR_STAB_ROW, 0);
    size_t st = favor_decode_state_bytes(2, 3, 64, 256);
    /* argument errors come back as status codes, nothing is launched */
    favor_status_t bad = favor_attn_causal(0, 0, 0, 0, 0, 1, 1, 16, 96, 64, 64, FAVOR_BF16, FAVOR_EXP, 0.f, 0, 0, 0);
    printf("%d %zu %zu %d %s\n", favor_abi_version(), ws, st, (int)bad, favor_status_string(bad));
    return 0;
}
''')
    exe = tmp_path / "use_favor"
    libdir = os.path.dirname(favor.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lfavor", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    bf = torch.bfloat16
    assert int(out[0]) == favor.abi_version()
    assert int(out[1]) == favor.workspace_bytes("noncausal", 1, 8, 4096, 64, 256, bf)
    assert int(out[2]) == favor.decode_state_bytes(2, 3, 64, 256)
    assert int(out[3]) == 2 and out[4].startswith("FAVOR_ERR_UNSUPPORTED")
