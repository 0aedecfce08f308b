"""Host logic of bench.py on the CPU: the algorithmic work behind the roofline figures, the clock
summary, argument checks, and the multi-rank plumbing (barrier, max over ranks; the reference arm
printing on rank 0 only) run as world-size-2 gloo ranks."""
import json
import math
import os
import socket
import subprocess
import sys
import tempfile

import pytest

import bench
import seeded_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_path_work_of_the_headline_workload():
    w = si.get_workload("noncausal_bf16_B1H8n1024d64m256")
    flops, nbytes = bench.path_work(w)
    tokens = 8 * 1024
    assert flops == 8 * 256 * 64 * tokens                      # two projections, state, readout
    assert nbytes == 4 * 64 * 2 * tokens + 256 * 64 * 2 == 4227072   # Q, K, V, Y and Omega once
    assert bench.kernel_work(w, "fused") == (flops, nbytes)
    fs, bs = bench.kernel_work(w, "state")
    fr, br = bench.kernel_work(w, "readout")
    assert fs + fr == flops
    assert bs + br == nbytes + 256 * 64 * 2                    # each of the two reads Omega
    assert bench.kernel_work(w, "combine") == (0.0, 0.0)


def test_tensor_core_path_per_workload():
    want = {"noncausal_f32_B1H1n256d64m128": False, "noncausal_bf16_B1H8n1024d64m256": True,
            "causal_bf16_B4H16n8192d64m256": True, "noncausal_bf16_B1H16n65536d128m256": True,
            "causal_relu_bf16_B8H32n32768d64m512": True}
    assert set(want) == set(si.workloads.WORKLOAD_ORDER)
    for name, tc in want.items():
        assert bench.tensor_core_path(si.get_workload(name)) is tc, name


@pytest.mark.parametrize("m,d", [(1, 64), (64, 64), (100, 64), (256, 64), (256, 128), (300, 128)])
def test_omega_flops_count_the_gram_schmidt_operations(m, d):
    # brute-force count: every ordered pair of rows i < k in a block costs a dot product and an
    # update (2d + 2d); every row a normalisation (2d + d) and its chi length (2d)
    total = 0
    for b in range(math.ceil(m / d)):
        r = min(d, m - b * d)
        for i in range(r):
            total += 4 * d * (r - 1 - i) + 3 * d + 2 * d
    assert bench.omega_flops(m, d) == total


def test_clock_summary_reads_nvidia_smi_lines():
    s = bench.ClockSampler(0)
    s.proc = object()  # stands for the running sampler
    s.out = tempfile.TemporaryFile(mode="w+")
    s.out.write("0, 2032, 2032, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
                "0, 1900, 2032, 1100.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
                "0, 2032, 2032, 950.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
                "not a sample\n")
    assert s.summary() == {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"], "samples": 3}
    s.proc = None
    assert s.summary()["samples"] == 0


def test_argument_checks():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])          # fewer than 3 warm-up steps
    env = dict(os.environ)
    os.environ.pop("WORLD_SIZE", None)
    try:
        with pytest.raises(SystemExit):
            bench.main(["--gpus", "2"])          # N > 1 only under torchrun with N processes
    finally:
        os.environ.clear()
        os.environ.update(env)


def test_sweep_form_choices():
    # --sweep covers both forms by default; --sweep-form narrows it; anything else is refused
    out = subprocess.run([sys.executable, "bench.py", "--help"], cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                         capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and "--sweep-form {both,noncausal,causal}" in out.stdout
    with pytest.raises(SystemExit):
        bench.main(["--sweep", "--sweep-form", "sideways"])


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = """
import json, sys, torch
sys.path.insert(0, {root!r})
import bench
rank, ws = bench.dist_setup("gloo")
bench.barrier()
v = bench.max_over_ranks(1.5 + 2.0 * rank, torch.device("cpu"))
bench.barrier()
print(json.dumps({{"rank": rank, "ws": ws, "max": v}}))
torch.distributed.destroy_process_group()
"""


def rank_env(rank: int, ws: int, port: int) -> dict:
    env = dict(os.environ)
    env.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
               WORLD_SIZE=str(ws))
    return env


def test_max_over_ranks_and_barrier_with_two_gloo_ranks():
    port = free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT.format(root=ROOT)], env=rank_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["ws"] == 2
        assert o["max"] == 3.5       # the larger of 1.5 (rank 0) and 3.5 (rank 1), on every rank


def test_reference_arm_prints_on_rank_zero_only():
    port = free_port()
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--workload", "noncausal_f32_B1H1n256d64m128"]
    res = [subprocess.run(cmd, env=rank_env(r, 2, port), capture_output=True, text=True, timeout=300)
           for r in (1, 0)]
    assert res[0].returncode == 0 and res[0].stdout.strip() == ""
    assert res[1].returncode == 0, res[1].stderr[-2000:]
    line = json.loads(res[1].stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
