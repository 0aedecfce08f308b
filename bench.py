#!/usr/bin/env python3
"""FAVOR+ attention benchmark: one JSON line with tokens/s, roofline fraction, e2e and CPU baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full FAVOR+ attention call (every kernel of the path: features, state, readout for
the non-causal form; the chunked scan for the causal form) over one batch of seeded synthetic input
already resident in HBM. The default workload is the largest one that fits a single GPU: causal
generalized-ReLU features, (B, H, n, d) = (8, 32, 32768, 64) with m = 512, bf16 in / fp32
accumulate. The other workloads are selected with --workload.

Timing: W untimed warm-up steps; K timed steps bracketed by a barrier and device synchronisation;
each step timed by CUDA events on the launching stream; L2 flushed (a 512 MB write) before every
timed step when the step's inputs are smaller than 2x L2; SM clocks and throttle reasons sampled with
nvidia-smi from the warm-up through the timed region. Multi-GPU (torchrun): every rank runs an independent replica of the workload (the
path has no exchange step), `value` is the tokens of all ranks over the slowest rank's time.

--impl reference times the fp64 CPU oracle (the only reference implementation: the pages ship no
code) on the host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "FAVOR+ attention tokens/s (B*H*n per s) and % of HBM/tensor roofline"
DEFAULT_WORKLOAD = "causal_relu_bf16_B8H32n32768d64m512"
L2_BYTES = 126 * 1024 * 1024
FLUSH_BYTES = 512 * 1024 * 1024
# A device-side wait (about 2.5 ms at 2 GHz) enqueued before a timed loop, so that the host queues
# the loop's launches ahead of the device: a host stall (an nvidia-smi sample, the interpreter) then
# never shows up as an idle gap between a step's start and end events.
QUEUE_AHEAD_CYCLES = 5_000_000

# Nominal unit counts used where a kernel is bound by plain CUDA-core arithmetic:
# 148 SMs x 128 fp32 FMA lanes x 2 flop x 2.032 GHz.
FP32_SIMT_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12
# Nominal dense FP64 rate of a B300 (far below its low-precision tensor rates).
FP64_PEAK_TFLOPS = 1.25

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the committed ncu
# captures, valid only while the kernel sources hash to `src`.
NCU_TRAFFIC: dict[str, dict] = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one launch (ncu --set full, see
    # profiles/nc_fused_noncausal_bf16_B1H8n1024d64m256.md); "src" is kernel_source_hash("fused")
    "noncausal_bf16_B1H8n1024d64m256:fused": {"bytes": 3253248, "src": "09c185d466e8dabc"},
    # profiles/causal_scan_relu_bf16_B8H32n32768d64m512.md: a 32-head x 8192-token capture
    # (118,248,960 bytes) scaled by the 32x more tokens of the full launch
    "causal_relu_bf16_B8H32n32768d64m512:causal": {"bytes": 3783966720, "src": "4f9a3a0886ca0d83"},
    # profiles/causal_scan_exp_bf16_B4H16n8192d64m256.md: the full launch captured
    "causal_bf16_B4H16n8192d64m256:causal": {"bytes": 250125312, "src": "4f9a3a0886ca0d83"},
}


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# The source files each kernel is compiled from (its traffic figure is void once any of them changes).
KERNEL_SOURCES = {
    "fused": ["tc.cuh", "tc_noncausal.cuh", "tc_fused.cuh"],
    "state": ["tc.cuh", "tc_noncausal.cuh"], "combine": ["tc.cuh", "tc_noncausal.cuh"],
    "readout": ["tc.cuh", "tc_noncausal.cuh"],
    "causal": ["tc.cuh", "tc_noncausal.cuh", "tc_scan.cuh"],
    "exact": ["tc.cuh", "tc_noncausal.cuh", "tc_exact.cuh"],
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kernelized_linear_attention_04_b300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(csrc))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------------------------------------
# Algorithmic work per kernel (per launch). Per token per head the whole path does
# 8 m d flops (two projections, the state contraction and the readout contraction) and moves
# 4 d s bytes (read Q, K, V, write Y; s = element size). Omega is counted once per launch.
# ------------------------------------------------------------------------------------------------

def kernel_work(w, kernel: str) -> tuple[float, float]:
    """(algorithmic flops, algorithmic HBM bytes) of one launch of `kernel` on workload w."""
    T, s, md = w.tokens, w.elem_bytes, w.m * w.d
    om = w.m * w.d * s
    if kernel == "state":        # project K, accumulate S and z; reads K, V
        return 4.0 * md * T, 2.0 * w.d * s * T + om
    if kernel == "readout":      # project Q, contract with S, divide; reads Q, writes Y
        return 4.0 * md * T, 2.0 * w.d * s * T + om
    if kernel in ("causal", "fused"):  # the whole path in one kernel
        return 8.0 * md * T, 4.0 * w.d * s * T + om
    if kernel == "combine":      # partial states -> one state per head
        return 0.0, 0.0
    if kernel.startswith("features"):
        return 2.0 * md * T, (w.d * s + w.m * 4) * T + om
    return 0.0, 0.0


def tensor_core_path(w) -> bool:
    """True when the library runs workload w on its tcgen05 kernels (bf16; non-causal with d = 64, or
    d = 128 with m <= 256 after padding to a multiple of 128; causal with d = 64 and m <= 512)."""
    if w.dtype != "bf16":
        return False
    m_pad = -(-w.m // 128) * 128
    if w.causal:
        return w.d == 64 and m_pad <= 512
    return w.d == 64 or m_pad <= 256


def path_work(w) -> tuple[float, float]:
    return 8.0 * w.m * w.d * w.tokens, 4.0 * w.d * w.elem_bytes * w.tokens + w.m * w.d * w.elem_bytes


# ------------------------------------------------------------------------------------------------
# Clock sampling (nvidia-smi) during the warm-up and timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clocks and throttle reasons with `nvidia-smi -lms` while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    FLAGS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 100):
        self.index = device_index
        self.period_ms = period_ms
        self.proc = None
        self.err = ""
        self.out = None

    def __enter__(self):
        import subprocess
        import tempfile

        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.period_ms}"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)  # let the first sample land before the timed region starts
        except Exception as e:  # pragma: no cover - reported in the JSON line
            self.proc, self.err = None, str(e)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "error": self.err}
        self.out.seek(0)
        mhz, maxes, reasons = [], [], set()
        for line in self.out.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.FLAGS, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(mhz)}


# ------------------------------------------------------------------------------------------------
# Distributed plumbing (replicas; barrier + max over ranks only)
# ------------------------------------------------------------------------------------------------

def dist_setup(backend: str):
    import torch.distributed as dist

    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    rank = dist.get_rank() if dist.is_initialized() else 0
    return rank, ws


def barrier():
    import torch.distributed as dist

    if dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device) -> float:
    import torch
    import torch.distributed as dist

    if not dist.is_initialized():
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline object, and the whole --impl reference arm)
# ------------------------------------------------------------------------------------------------

def oracle_sample(w, budget_s: float) -> tuple[list[tuple[int, int]], int]:
    """A bounded sample of workload w for one oracle timing step: up to one head per host thread
    (the oracle runs its heads in parallel) and the first n' tokens of each, n' sized from a short
    calibration run so that one step takes about `budget_s`. A causal prefix is exactly the first
    n' rows of the full result; a non-causal prefix is the same computation over n' tokens."""
    import oracle

    cores = oracle.get_threads()
    heads = [(i // w.H, i % w.H) for i in range(min(w.heads, cores))]
    n_cal = min(w.n, 128)
    inputs = oracle_inputs(w, heads, n_cal)
    oracle_step(w, inputs)  # first touch
    t0 = time.perf_counter()
    oracle_step(w, inputs)
    per_token = max(time.perf_counter() - t0, 1e-6) / n_cal
    n_pre = int(max(1, min(w.n, budget_s / per_token)))
    return heads, n_pre


def oracle_inputs(w, heads, n_pre: int):
    Q, K, V = [], [], []
    for b, h in heads:
        hi = si.head_inputs(w, b, h)
        Q.append(si.to_f64(hi["Q"][:n_pre]))
        K.append(si.to_f64(hi["K"][:n_pre]))
        V.append(si.to_f64(hi["V"][:n_pre]))
    return np.stack(Q), np.stack(K), np.stack(V), si.omega_for(w)[1]


def oracle_step(w, inputs):
    import oracle

    Q, K, V, om = inputs
    fn = oracle.attn_causal if w.causal else oracle.attn_noncausal
    return fn(Q, K, V, om, kind=w.kind, relu_eps=w.relu_eps)


def sample_note(w, heads, n_pre: int) -> str:
    return (f"{len(heads)} of {w.heads} heads x the first {n_pre} of {w.n} tokens each, fp64 C loops, "
            f"OpenMP over heads")


def cpu_baseline(w, target_s: float = 12.0) -> dict:
    import oracle

    heads, n_pre = oracle_sample(w, budget_s=min(4.0, target_s / 3))
    inputs = oracle_inputs(w, heads, n_pre)
    oracle_step(w, inputs)  # load / first-touch
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_step(w, inputs)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s or reps >= 1000:
            break
    tokens = reps * len(heads) * n_pre
    return {"value": tokens / el, "unit": "tokens/s", "cores": oracle.get_threads(), "kind": "oracle",
            "sample": f"{sample_note(w, heads, n_pre)}; {reps} repetitions, {el:.1f} s wall"}


def run_reference(args, w):
    rank, ws = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    import oracle

    # the whole run (warm-up and timed steps) within about two minutes of host time
    heads, n_pre = oracle_sample(w, budget_s=min(0.5, 120.0 / (args.steps + args.warmup)))
    inputs = oracle_inputs(w, heads, n_pre)
    for _ in range(args.warmup):
        oracle_step(w, inputs)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, inputs)
        times.append(time.perf_counter() - t0)
    tok = len(heads) * n_pre
    value = tok * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "timing": "host wall clock (time.perf_counter) around each step, fp64 C loops on the host cores",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.get_threads(), "kind": "oracle",
                         "sample": f"{sample_note(w, heads, n_pre)}, per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def l2_policy(w) -> tuple[bool, str]:
    """Whether the timed steps flush L2 first (inputs smaller than twice L2), and how to say so."""
    flush = path_work(w)[1] < 2 * L2_BYTES
    return flush, ("flushed before every timed step (512 MB write)" if flush else "inputs larger than L2")


def workload_config(w) -> dict:
    """The `config` object of a bench line; both arms print exactly this for the same workload."""
    c = {"workload": w.name, "form": "causal" if w.causal else "non-causal", "features": w.kind,
         "B": w.B, "H": w.H, "n": w.n, "d": w.d, "m": w.m, "inputs": f"iid N(0, {w.sigma}^2)"}
    if w.causal:
        c["chunk"] = w.chunk
    c["l2"] = l2_policy(w)[1]
    return c


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

def run_ours(args, w):
    import torch

    rank, world = dist_setup("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import kernelized_linear_attention_04_b300 as favor

    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    full = si.full_inputs(w)
    om_store, _ = si.omega_for(w)

    def pinned(a):
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
        return t.pin_memory()

    hQ, hK, hV, hOm = pinned(full["Q"]), pinned(full["K"]), pinned(full["V"]), pinned(om_store)
    del full
    Q, K, V, Om = (t.to(dev) for t in (hQ, hK, hV, hOm))
    Y = torch.empty_like(Q)
    hY = torch.empty(Y.shape, dtype=dt).pin_memory()
    op = "causal" if w.causal else "noncausal"
    wsb = favor.workspace_bytes(op, w.B, w.H, w.n, w.d, w.m, dt, kind=w.kind, chunk=w.chunk if w.causal else 0)
    wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        # on the current stream: the bench's stream, or the side stream of a graph capture
        st = torch.cuda.current_stream()
        if w.causal:
            favor.favor_attn_causal(Q, K, V, Om, chunk=w.chunk, kind=w.kind, relu_eps=w.relu_eps, out=Y,
                                    workspace=wsp, stream=st)
        else:
            favor.favor_attn_noncausal(Q, K, V, Om, kind=w.kind, relu_eps=w.relu_eps, out=Y, workspace=wsp,
                                       stream=st)

    flush, _ = l2_policy(w)
    fbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def timed_loop(n_steps, body):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
        torch.cuda._sleep(QUEUE_AHEAD_CYCLES)
        for a, b in evs:
            if fbuf is not None:
                fbuf.zero_()
            a.record(stream)
            body()
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def timed_graph(n_steps, body):
        # the steps (each behind its L2 flush, bracketed by event-record nodes) captured into one
        # CUDA graph and launched once: no host work can fall between a step's two events
        evs = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(n_steps)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for a, b in evs:
                if fbuf is not None:
                    fbuf.zero_()
                a.record()
                body()
                b.record()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    # -- device-resident throughput (clocks sampled from the warm-up on, so the GPU is under load) --
    sampler = ClockSampler(local)
    with sampler:
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        assert favor.last_device_error() == 0
        barrier()
        torch.cuda.synchronize()
        try:
            ms, timing = timed_graph(args.steps, call), "one CUDA graph of the timed steps"
        except RuntimeError as e:  # capture unsupported here: eager launches, queued ahead of the device
            torch.cuda.synchronize()
            ms, timing = timed_loop(args.steps, call), f"eager launches (graph capture failed: {str(e)[:80]})"
        assert favor.last_device_error() == 0
        barrier()
        torch.cuda.synchronize()
    ms_per_step = max_over_ranks(sum(ms) / len(ms), dev)
    value = world * w.tokens / (ms_per_step * 1e-3)

    # -- per-kernel durations (same loop, launches bracketed by events inside the library) -----
    favor.trace_enable(True)
    timed_loop(args.steps, call)
    tr = favor.trace_read()
    favor.trace_enable(False)
    launched = {k: v for k, v in tr.items() if v[0] > 0}
    launches_per_step = sum(v[0] for v in launched.values()) / args.steps
    dom = max(launched, key=lambda k: launched[k][1])
    dom_ms = eager_ms = launched[dom][1] / launched[dom][0]
    dur_src = "events around each launch, eager"
    if timing.startswith("one CUDA graph") and launches_per_step == 1:
        # the step is this one launch: its graph-timed duration carries no host launch latency
        dom_ms, dur_src = sum(ms) / len(ms), "graph-timed step (the step is this one launch)"
        if dom == "causal" and w.m > 128:
            dur_src += ", after the clear of the scan's group counters (a memset of G x 64 bytes)"
    flops, nbytes = kernel_work(w, dom)
    peaks, peak_kind = load_peaks()
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    simt = not tensor_core_path(w)
    if simt:
        t_cmp, cmp_unit, cmp_peak, cmp_bound = flops / (FP32_SIMT_PEAK_TFLOPS * 1e12), "TFLOP/s", FP32_SIMT_PEAK_TFLOPS, "alu"
        cmp_note = "nominal fp32 FFMA: 148 SMs x 128 lanes x 2 flop x 2.032 GHz"
    else:
        t_cmp, cmp_unit, cmp_peak, cmp_bound = flops / (peaks["bf16_tflops"] * 1e12), "TFLOP/s", peaks["bf16_tflops"], "tensor"
        cmp_note = f"bf16 dense, {peak_kind} burst"
    if t_hbm >= t_cmp:
        ach, peak, unit, bound, note = nbytes / (dom_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s", "hbm", f"HBM copy, {peak_kind}"
    else:
        ach, peak, unit, bound, note = flops / (dom_ms * 1e-3) / 1e12, cmp_peak, cmp_unit, cmp_bound, cmp_note
    src = kernel_source_hash(dom)
    tr_entry = NCU_TRAFFIC.get(f"{w.name}:{dom}")
    traffic = tr_entry["bytes"] if tr_entry and tr_entry.get("src") == src else None
    roofline = {"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                "traffic": traffic, "kernel": dom, "kernel_ms": dom_ms, "duration_source": dur_src,
                "kernel_ms_eager": eager_ms, "peak_source": note,
                "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
                "kernels_ms": {k: v[1] / v[0] for k, v in launched.items()}}
    # whole-path roofline fraction (the slower of flops at the tensor peak and bytes at HBM)
    pf, pb = path_work(w)
    t_roof = max(pf / (peaks["bf16_tflops"] * 1e12), pb / (peaks["hbm_gbs"] * 1e9))

    # -- end to end through the public API with host buffers ----------------------------------
    def e2e_body():
        Q.copy_(hQ, non_blocking=True)
        K.copy_(hK, non_blocking=True)
        V.copy_(hV, non_blocking=True)
        Om.copy_(hOm, non_blocking=True)
        call()
        hY.copy_(Y, non_blocking=True)

    for _ in range(2):
        e2e_body()
    barrier()
    torch.cuda.synchronize()
    ms_e2e = timed_loop(args.steps, e2e_body)
    barrier()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(ms_e2e) / len(ms_e2e), dev)
    h2d = sum(t.numel() * t.element_size() for t in (hQ, hK, hV, hOm))
    d2h = hY.numel() * hY.element_size()
    assert favor.last_device_error() == 0

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": workload_config(w), "timing": timing,
            "path_roofline_frac": (t_roof * 1e3) / ms_per_step,
            "roofline": roofline,
            "e2e": {"value": world * w.tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": sampler.summary(),
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line))
    import torch.distributed as dist

    if dist.is_initialized():
        dist.destroy_process_group()
    return 0


def run_decode(args, w):
    """Streaming decode: one favor_decode_step per timed step, one new token for each of the
    workload's B*H heads (its d, m, dtype and feature family; n is not used). Memory-bound: the
    step reads and writes the fp32 state S [m x d] and z [m] of every head."""
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import kernelized_linear_attention_04_b300 as favor

    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    steps_tokens = args.warmup + args.steps
    # one token per head per step, drawn once (synthetic, iid N(0, sigma^2)); Omega from the workload
    toks = torch.randn(3, steps_tokens + args.steps, w.B, w.H, w.d, generator=g) * w.sigma
    toks = toks.to(dt).to(dev)
    om_store, _ = si.omega_for(w)
    Om = (torch.from_numpy(om_store.view(np.int16)).view(torch.bfloat16) if om_store.dtype == np.uint16
          else torch.from_numpy(om_store)).to(dev)
    state = favor.decode_state(w.B, w.H, w.d, w.m)
    y = torch.empty(w.B, w.H, w.d, dtype=dt, device=dev)

    def step(i):
        favor.favor_decode_step(toks[0, i], toks[1, i], toks[2, i], Om, state, kind=w.kind, relu_eps=w.relu_eps, out=y)

    BH = w.B * w.H
    s_el = 4 if dt == torch.float32 else 2
    nbytes = BH * (2 * w.m * w.d * 4 + 2 * w.m * 4 + 4 * w.d * s_el) + w.m * w.d * s_el
    # every timed step starts from a cold L2 (a 512 MB write) unless the state is larger than L2
    flush = nbytes < 2 * L2_BYTES
    fbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def timed(n0):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda._sleep(QUEUE_AHEAD_CYCLES)
        for i, (a, b) in enumerate(evs):
            if fbuf is not None:
                fbuf.zero_()
            a.record()
            step(n0 + i)
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def timed_graph(n0):
        # the K steps (each behind its L2 flush, bracketed by event-record nodes) captured into one
        # CUDA graph and launched once: no host work can fall between a step's two events
        evs = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(args.steps)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i, (a, b) in enumerate(evs):
                if fbuf is not None:
                    fbuf.zero_()
                a.record()
                step(n0 + i)
                b.record()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    # clocks sampled from the warm-up on, so that the timed steps start on a busy GPU
    sampler = ClockSampler(0)
    with sampler:
        for i in range(args.warmup):
            if fbuf is not None:
                fbuf.zero_()
            step(i)
        torch.cuda.synchronize()
        assert favor.last_device_error() == 0
        try:
            per_step, timing = timed_graph(args.warmup), "one CUDA graph of the timed steps"
        except RuntimeError as e:  # capture unsupported here: eager launches, queued ahead of the device
            per_step, timing = timed(args.warmup), f"eager launches (graph capture failed: {str(e)[:80]})"
        assert favor.last_device_error() == 0
    ms = sum(per_step) / len(per_step)
    favor.trace_enable(True)
    timed(args.warmup)
    tr = favor.trace_read()
    favor.trace_enable(False)
    k_ms = eager_ms = tr["decode"][1] / tr["decode"][0]
    dur_src = "events around each launch, eager"
    if timing.startswith("one CUDA graph"):
        # a decode step is exactly one launch of the kernel
        k_ms, dur_src = ms, "graph-timed step (the step is this one launch)"
    peaks, peak_kind = load_peaks()
    ach = nbytes / (k_ms * 1e-3) / 1e9
    line = {
        "metric": "FAVOR+ streaming decode tokens/s (B*H new tokens per s)", "value": BH / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "ms_per_step_median": float(np.median(per_step)), "ms_per_step_max": max(per_step),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32" if dt == torch.float32 else "bf16",
        "data": "synthetic",
        "config": {"workload": f"decode_{w.dtype}_B{w.B}H{w.H}d{w.d}m{w.m}", "form": "streaming decode step",
                   "features": w.kind, "B": w.B, "H": w.H, "d": w.d, "m": w.m,
                   "l2": "flushed before every timed step (512 MB write)" if flush else "state larger than L2",
                   "timing": timing},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": None, "kernel": "decode", "kernel_ms": k_ms,
                     "duration_source": dur_src, "kernel_ms_eager": eager_ms,
                     "peak_source": f"HBM copy, {peak_kind}", "algorithmic_bytes": nbytes},
        "gpu_launches": args.steps, "clocks": sampler.summary(),
    }
    print(json.dumps(line))


def omega_flops(m: int, d: int) -> float:
    """fp64 flops of one Omega build: per block of r rows, the projections (a dot product and an
    update, 4d each, for every pair of rows) and the normalisations and chi lengths (5d per row).
    The Box-Muller draws (2 d^2 logarithms and cosines per block) are not counted."""
    total = 0.0
    for b in range(-(-m // d)):
        r = min(d, m - b * d)
        total += 2.0 * d * r * (r - 1) + 5.0 * d * r
    return total


def run_omega(args, w):
    """On-device Omega builder: one favor_omega per timed step for the workload's m and d, the
    steps captured in one CUDA graph with the L2 flush between them."""
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import kernelized_linear_attention_04_b300 as favor

    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    Om = torch.empty(w.m, w.d, dtype=dt, device=dev)
    fbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(i):
        favor.favor_omega(w.omega_seed + i, w.m, w.d, dtype=dt, out=Om)

    sampler = ClockSampler(0)
    with sampler:
        for i in range(args.warmup):
            fbuf.zero_()
            step(i)
        torch.cuda.synchronize()
        assert favor.last_device_error() == 0
        evs = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(args.steps)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i, (a, b) in enumerate(evs):
                fbuf.zero_()
                a.record()
                step(args.warmup + i)
                b.record()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        per_step = [a.elapsed_time(b) for a, b in evs]
    ms = sum(per_step) / len(per_step)
    flops = omega_flops(w.m, w.d)
    ach = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": "FAVOR+ random projection rows built per s (orthogonal, on device)", "value": w.m / (ms * 1e-3),
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "ms_per_step_median": float(np.median(per_step)), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"omega_{w.dtype}_m{w.m}d{w.d}", "form": "orthogonal random features",
                   "m": w.m, "d": w.d, "output": w.dtype, "l2": "flushed before every timed step (512 MB write)",
                   "timing": "one CUDA graph of the timed steps"},
        "roofline": {"bound": "alu", "achieved": ach, "peak": FP64_PEAK_TFLOPS, "unit": "TFLOP/s",
                     "frac": ach / FP64_PEAK_TFLOPS, "traffic": None, "kernel": "omega", "kernel_ms": ms,
                     "duration_source": "graph-timed step (the step is this one launch)",
                     "peak_source": "nominal dense FP64 of a B300", "algorithmic_flops": flops},
        "gpu_launches": args.steps, "clocks": sampler.summary(),
    }
    print(json.dumps(line))


# ------------------------------------------------------------------------------------------------
# FAVOR+ against exact softmax attention: wall clock and divergence over n and m ("Linear
# Attention and the Performer", *Exercise*: the (1, 8, n, 64) shape against the exact operator;
# the "Performer" paper note's checklist: n large enough, wall clock, m, the comparator).
# Context, not a bench line: one JSON object per point on stdout.
# ------------------------------------------------------------------------------------------------

SWEEP_N = (256, 1024, 4096, 16384, 65536)
SWEEP_M = (64, 128, 256, 512)  # the library's range (m <= 512)


def run_sweep(args):
    import torch

    import kernelized_linear_attention_04_b300 as favor

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    ns = [int(x) for x in args.sweep_n.split(",")] if args.sweep_n else list(SWEEP_N)
    ms = [int(x) for x in args.sweep_m.split(",")] if args.sweep_m else list(SWEEP_M)

    def to_dev(a):
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
        return t.to(dev)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a, b in evs:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in evs]))

    forms = {"both": (False, True), "noncausal": (False,), "causal": (True,)}[args.sweep_form]
    for causal in forms:
        for n in ns:
            base = si.Workload("sweep", 1, 8, n, 64, ms[0], "bf16", causal, kind="exp", seed=101 + n, omega_seed=7)
            full = si.full_inputs(base)
            Q, K, V = (to_dev(full[k]) for k in ("Q", "K", "V"))
            del full
            reps = max(3, min(20, int(2e9 / (4.0 * n * n * 64 * 8))))
            Ye = favor.favor_softmax_attn(Q, K, V, causal=causal)
            t_exact = timed(lambda: favor.favor_softmax_attn(Q, K, V, causal=causal, out=Ye), reps)
            ye = Ye.float()
            for m in ms:
                w = base.with_(m=m)
                om, _ = si.omega_for(w)
                Om = to_dev(om)
                op = "causal" if causal else "noncausal"
                ws = torch.empty(max(favor.workspace_bytes(op, 1, 8, n, 64, m, torch.bfloat16, kind="exp"), 1),
                                 dtype=torch.uint8, device=dev)
                call = (lambda: favor.favor_attn_causal(Q, K, V, Om, kind="exp", out=Yf, workspace=ws)) if causal else \
                       (lambda: favor.favor_attn_noncausal(Q, K, V, Om, kind="exp", out=Yf, workspace=ws))
                Yf = torch.empty_like(Q)
                call()
                t_favor = timed(call, max(reps, 10))
                diff = Yf.float() - ye
                print(json.dumps({
                    "sweep": "favor_vs_exact", "form": op, "B": 1, "H": 8, "n": n, "d": 64, "m": m,
                    "features": "exp", "dtype": "bf16", "favor_ms": t_favor, "exact_ms": t_exact,
                    "exact_over_favor": t_exact / t_favor,
                    "rel_l2": float(diff.norm() / ye.norm()), "max_abs": float(diff.abs().max()),
                    "timing": "CUDA events, median, L2 warm", "data": "synthetic iid N(0, 1)"}), flush=True)
            del Q, K, V, Ye
            torch.cuda.empty_cache()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=si.workloads.WORKLOAD_ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the host-core oracle timing")
    ap.add_argument("--decode", action="store_true",
                    help="time the streaming decode step at the workload's B, H, d, m instead of the full call")
    ap.add_argument("--omega", action="store_true",
                    help="time the on-device Omega builder at the workload's m and d instead of the full call")
    ap.add_argument("--n", type=int, default=None,
                    help="override the sequence length (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--H", type=int, default=None,
                    help="override the heads per batch entry (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--sweep", action="store_true",
                    help="FAVOR+ (exp features) against the exact softmax kernel over n and m: time and divergence")
    ap.add_argument("--sweep-n", default=None, help="comma-separated sequence lengths for --sweep")
    ap.add_argument("--sweep-m", default=None, help="comma-separated feature counts for --sweep")
    ap.add_argument("--sweep-form", default="both", choices=["both", "noncausal", "causal"],
                    help="the attention forms --sweep covers")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and ws != args.gpus:
        ap.error("--gpus N > 1 runs under torchrun with N processes")
    w = si.get_workload(args.workload)
    if args.n is not None:
        w = w.with_(n=args.n, name=f"{w.name}@n={args.n}")
    if args.H is not None:
        w = w.with_(H=args.H, name=f"{w.name}@H={args.H}")
    if args.sweep:
        return run_sweep(args)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.decode:
        return run_decode(args, w)
    if args.omega:
        return run_omega(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
