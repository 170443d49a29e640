#!/usr/bin/env python3
"""Benchmark of the block-scaled FP8 weight GEMM (libbsf8) on one GB300 per rank.

Workload (the wo_a decode layer of the page "recipes/docker-images/mia-tp4/adapter/
wo_a_w8.py"): G = 2 groups of W[1024, 4096] as e4m3 twins with 32x32 exponents, M = 6
token rows, split_k = 8 summed in a fixed order, 43 distinct seeded weight copies (one
per layer) cycled so the L2 is cold.  One step = the 43 layer calls of one decode step,
captured once in a CUDA graph and replayed.  Inputs are seeded synthetic tensors (there
is no model checkpoint here).

Prints ONE JSON line on rank 0.  `value` is the weight-stream bandwidth (e4m3 codes +
exponent bytes per call / time per call) summed over all ranks; `e2e` is the same metric
measured through the public Python API with the activations copied from pinned host
memory and the outputs copied back inside the timed region.  `configs` times every other
config of the hot path (make_twin, dequant, pad-K, the GEMM at the tiny, wo_a, down_proj,
mid-row and gate_up/head sweep shapes, per-row scales, fp32 output, prefill-sized rows),
each over enough weight copies to stream at least twice the L2, as us/call (median over
graph replays, p10/p90), weight GB/s, fraction of the measured HBM peak, the kernel that
ran and the split it used.  The SM clock is sampled inside the timed region (each SM's
cycle counter against the global timer) as well as by nvidia-smi.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bsf8|reference]

`--impl reference` times the CPU oracle (oracle/, a plain C restatement of the pages)
on a bounded sample of the same workload: the baseline this library is compared with.
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the op has no
exchange step, so no collective runs on the data path; only the timing is combined
(max over ranks) and the bytes summed.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "weight-stream HBM GB/s (frac of GB300 peak) and us/call at M=6, L2 cold"
LAYERS = 43
# The kernel this workload runs (the decode-ahead kernel: M <= 8, one group per block).
KERNEL_SOURCES = ("block_scaled_fp8_weight_gb300/csrc/bsf8_lowm.cu",
                  "block_scaled_fp8_weight_gb300/csrc/bsf8_device.cuh")
KERNEL_NAME = "lowm_kernel"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_wo_a_m6_dram_traffic.txt")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=("bsf8", "reference"), default="bsf8")
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU time budget of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-calls", type=int, default=0,
                   help="profiling mode: run this many eager layer calls and exit (no JSON)")
    p.add_argument("--split-k", type=int, default=None, help="override the workload's split_k")
    p.add_argument("--workload", choices=("wo_a", "down_proj", "mid", "gate_up", "head",
                                          "make_twin", "dequant", "pad_k"),
                   default="wo_a", help="profiling mode only: which workload to run (a GEMM shape, "
                                        "or make_twin / dequant on the wo_a shape, pad_k on down_proj)")
    p.add_argument("--m", type=int, default=None, help="profiling mode only: token rows")
    p.add_argument("--copies", type=int, default=None,
                   help="profiling mode only: distinct weight copies cycled (default 43, 3 for head)")
    p.add_argument("--suite", action="store_true",
                   help="time every hot-path row (make_twin, dequant, pad-K, the GEMM at every "
                        "config) and print one JSON line per row instead of the headline line")
    p.add_argument("--no-configs", action="store_true",
                   help="leave the per-config map out of the headline line")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, device_is_cuda):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("nccl" if device_is_cuda else "gloo")
    return dist


def barrier(dist, device):
    if dist is None:
        return
    import torch
    if device.type == "cuda":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


def aggregate(dist, elapsed_s: float, units: float, device):
    """Replicas: the job's time is the slowest rank's, its work the sum of all ranks'."""
    if dist is None:
        return elapsed_s, units
    import torch
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ environment

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor throughput to compare large-M GEMMs with (burst, measured)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


def kernel_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    vals = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every ~50 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []   # (t, sm_mhz, max_mhz, reasons)
        self._stop = threading.Event()
        self._thr = None

    def _poll(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                      "--format=csv,noheader,nounits"], capture_output=True,
                                     text=True, timeout=5).stdout.strip()
                f = [x.strip() for x in out.split(",")]
                reasons = []
                for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                      "sw_power_cap"), f[5:9]):
                    if val.lower().startswith("active"):
                        reasons.append(name)
                self.samples.append((time.time(), float(f[1]), float(f[2]), reasons))
            except Exception:
                pass
            self._stop.wait(0.05)

    def start(self):
        self._thr = threading.Thread(target=self._poll, daemon=True)
        self._thr.start()

    def stop(self):
        self._stop.set()
        if self._thr:
            self._thr.join(timeout=10)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside:
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest samples to a timed region shorter than the sampling period"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------------------ workload

def workload():
    from block_scaled_fp8_weight_gb300 import workloads as wl
    return wl.WO_A


def config_dict(wk, pdl=True):
    return {
        "workload": f"wo_a decode step: G={wk.G} x W[{wk.N},{wk.K}] e4m3 + 32x32 ue8m0 exponents, "
                    f"M={wk.M}, split_k={wk.split_k}, {LAYERS} distinct layer copies per step",
        "G": wk.G, "N": wk.N, "K": wk.K, "M": wk.M, "split_k": wk.split_k, "layers": LAYERS,
        "l2": f"inputs larger than L2: {LAYERS} weight copies x {wk.weight_bytes / 1e6:.2f} MB "
              f"= {LAYERS * wk.weight_bytes / 1e6:.0f} MB streamed per step (L2 129 MB)",
        "launch": "one CUDA graph per step" + (", programmatic dependent launch" if pdl else ""),
    }


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_slices(wk, x, w8, ex, parts: int):
    """The layer's weight rows cut into `parts` contiguous slices of whole 32-row blocks
    (each output keeps its own index-order sum, so the slices give the layer's bits)."""
    import numpy as np
    nb = wk.N // 32
    bounds = [round(i * nb / parts) * 32 for i in range(parts + 1)]
    return [(np.ascontiguousarray(w8[:, a:b]), np.ascontiguousarray(ex[:, a // 32:b // 32]))
            for a, b in zip(bounds[:-1], bounds[1:]) if b > a]


def oracle_layer_time(x, slices, threads: int, seconds: float):
    """Seconds per whole-layer call of the oracle with the slices run on `threads` threads
    (the oracle's C function runs without the interpreter lock)."""
    import concurrent.futures as cf
    import oracle
    run = lambda sl: oracle.gemm(x, sl[0], sl[1])
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, slices))                       # load + first touch
        calls, t0 = 0, time.perf_counter()
        while True:
            list(ex.map(run, slices))
            calls += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return el / calls


def cpu_oracle_baseline(wk, seconds: float):
    """The oracle, as it stands, on the host cores: whole wo_a layer calls at M=6, on one
    thread and on one thread per core (the layer's rows split across them), each the
    median of 3 runs."""
    w8, ex = wk.weights(copy=0)
    x = wk.x(copy=0)
    cores = host_cores()
    one = oracle_slices(wk, x, w8, ex, 1)
    many = oracle_slices(wk, x, w8, ex, 4 * cores)
    per = max(0.5, seconds / 6.0)
    t1 = statistics.median(oracle_layer_time(x, one, 1, per) for _ in range(3))
    tn = statistics.median(oracle_layer_time(x, many, cores, per) for _ in range(3))
    return {"value": wk.weight_bytes / tn / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "us_per_call": tn * 1e6,
            "one_thread": {"value": wk.weight_bytes / t1 / 1e9, "us_per_call": t1 * 1e6},
            "sample": f"whole wo_a layer calls (G=2, N=1024, K=4096, M=6), median of 3 runs of "
                      f"~{per:.1f} s: one thread per host core ({cores} cores, the layer's weight rows "
                      f"split into {len(many)} slices), and one thread"}


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm, on all host cores: each step is a bounded slice
    of one layer call (a contiguous range of weight rows, split across one thread per core)."""
    if rank != 0:
        return None
    import oracle
    wk = workload()
    w8, ex = wk.weights(copy=0)
    x = wk.x(copy=0)
    cores = host_cores()
    budget = 90.0
    probe_rows = 32
    t0 = time.perf_counter()
    oracle.gemm(x, w8[:, :probe_rows], ex[:, :probe_rows // 32])
    t_probe = max(time.perf_counter() - t0, 1e-6)
    per_step = budget / max(1, args.steps + args.warmup)
    rows = int(min(wk.N, max(probe_rows, (per_step / t_probe) * probe_rows * cores)) // 32 * 32)
    rows = max(32, rows)
    sub = dataclasses.replace(wk, N=rows)
    slices = oracle_slices(sub, x, w8[:, :rows], ex[:, :rows // 32], min(rows // 32, 4 * cores))
    import concurrent.futures as cf
    run = lambda sl: oracle.gemm(x, sl[0], sl[1])
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        for _ in range(args.warmup):
            list(pool.map(run, slices))
        t0 = time.perf_counter()
        for _ in range(args.steps):
            list(pool.map(run, slices))
        el = time.perf_counter() - t0
    bytes_step = wk.G * rows * wk.K + wk.G * (rows // 32) * (wk.K // 32)
    value = bytes_step * args.steps / el / 1e9
    sample = (f"each step: rows [0, {rows}) of both groups of one wo_a layer (M=6), "
              f"{rows / wk.N:.4f} of a layer call, on {cores} host cores (one thread per core)")
    cfg = config_dict(wk, pdl=False)
    cfg["launch"] = "CPU oracle (plain C, binary32 index-order sum), one thread per host core"
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": cfg, "impl": "reference",
        "us_per_call": el / args.steps * 1e6 * wk.N / rows,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def build_layers(wk, device, copies=LAYERS):
    import torch
    layers = []
    for c in range(copies):
        w8, ex = wk.weights(copy=c)
        x = wk.x(copy=c)
        layers.append((torch.from_numpy(w8).to(device), torch.from_numpy(ex).to(device),
                       torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(device)))
    return layers


def time_graph(layers, wk, steps, warmup, pdl, stream, per_step=False, clock_probe=None):
    """Captures the 43 calls of one step in a CUDA graph; replays `warmup` untimed then
    `steps` timed steps between one pair of CUDA events; returns (seconds, wall t0, wall t1,
    per-step seconds or None).  per_step adds an event between steps (same stream, nothing
    else changes); clock_probe (an int64 [nsm, 2] tensor pair) samples every SM's cycle
    counter right before and right after the timed region."""
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    bsf8.set_option(bsf8.OPT_PDL, 1 if pdl else 0)
    outs = [torch.empty((wk.M, wk.G, wk.N), dtype=torch.bfloat16, device=stream.device) for _ in layers]
    steps_s = None
    try:
        with torch.cuda.stream(stream):
            for (w8, ex, x), y in zip(layers, outs):          # eager warm call (module load)
                bsf8.gemm(x, w8, ex, split_k=wk.split_k, out=y)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for (w8, ex, x), y in zip(layers, outs):
                    bsf8.gemm(x, w8, ex, split_k=wk.split_k, out=y)
            for _ in range(warmup):
                g.replay()
            stream.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1 if per_step else 2)]
            w0 = time.time()
            if clock_probe is not None:
                bsf8.sm_clock_sample(clock_probe[0], stream=stream)
            ev[0].record(stream)
            for i in range(steps):
                g.replay()
                if per_step:
                    ev[i + 1].record(stream)
            ev[-1].record(stream)
            if clock_probe is not None:
                bsf8.sm_clock_sample(clock_probe[1], stream=stream)
            stream.synchronize()
            w1 = time.time()
            if per_step:
                steps_s = [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(steps)]
    finally:
        bsf8.set_option(bsf8.OPT_PDL, 1)
    return ev[0].elapsed_time(ev[-1]) / 1e3, w0, w1, steps_s


def region_clock(probe):
    """Median over SMs of each SM's average clock (MHz) between the two samples."""
    a = probe[0].cpu().numpy().astype("float64")
    b = probe[1].cpu().numpy().astype("float64")
    ok = (a[:, 0] > 0) & (b[:, 0] > a[:, 0])
    if not ok.any():
        return None
    mhz = (b[ok, 1] - a[ok, 1]) / (b[ok, 0] - a[ok, 0]) * 1e3
    return {"sm_mhz_median": float(statistics.median(mhz)), "sm_mhz_min": float(mhz.min()),
            "sm_mhz_max": float(mhz.max()), "sms": int(ok.sum()),
            "how": "each SM's cycle counter against the global ns timer, sampled by a one-warp "
                   "block per SM right before and right after the timed region (bsf8_sm_clock_sample)"}


def time_broken_chain(layers, wk, steps, stream, mode, sleep_cycles=20000):
    """Each layer's GEMM after a kernel that is not this library's (a spin of sleep_cycles
    standing in for a collective or another op; it does not let the GEMM start early), in a
    CUDA graph of the 43 layers.  mode "sleep": the spins alone; "plain": spin + GEMM;
    "prefetch": spin + GEMM with bsf8_prefetch_l2 of the layer's twin on a side stream,
    issued as the spin starts.  Returns seconds per layer."""
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    outs = [torch.empty((wk.M, wk.G, wk.N), dtype=torch.bfloat16, device=stream.device) for _ in layers]
    side = torch.cuda.Stream(device=stream.device)

    def step():
        for (w8, ex, x), y in zip(layers, outs):
            if mode == "prefetch":
                ev = torch.cuda.Event()
                ev.record(stream)
                side.wait_event(ev)
                bsf8.prefetch_l2(w8, ex, stream=side)
            torch.cuda._sleep(sleep_cycles)
            if mode != "sleep":
                bsf8.gemm(x, w8, ex, split_k=wk.split_k, out=y)
        if mode == "prefetch":
            stream.wait_stream(side)

    with torch.cuda.stream(stream):
        step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(3):
            g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
    return e0.elapsed_time(e1) / 1e3 / (steps * len(layers))


def time_eager(layers, wk, steps, stream):
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    outs = [torch.empty((wk.M, wk.G, wk.N), dtype=torch.bfloat16, device=stream.device) for _ in layers]
    with torch.cuda.stream(stream):
        for _ in range(3):
            for (w8, ex, x), y in zip(layers, outs):
                bsf8.gemm(x, w8, ex, split_k=wk.split_k, out=y)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            for (w8, ex, x), y in zip(layers, outs):
                bsf8.gemm(x, w8, ex, split_k=wk.split_k, out=y)
        e1.record(stream)
        stream.synchronize()
    return e0.elapsed_time(e1) / 1e3


def time_isolated(layers, wk, reps, stream):
    """Mean duration of one launch with nothing before or after it on the stream and the L2
    flushed (a 256 MB write) before each, timed by CUDA events around the launch."""
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=stream.device)
    y = torch.empty((wk.M, wk.G, wk.N), dtype=torch.bfloat16, device=stream.device)
    total = 0.0
    with torch.cuda.stream(stream):
        for i in range(reps + 2):
            w8, ex, x = layers[i % len(layers)]
            flush.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bsf8.gemm(x, w8, ex, split_k=wk.split_k, out=y)
            e1.record(stream)
            stream.synchronize()
            if i >= 2:
                total += e0.elapsed_time(e1) / 1e3
    del flush
    return total / reps


def time_e2e(layers, wk, steps, stream):
    """End to end through the public API: every step copies each layer's activations
    from pinned host memory, runs bsf8.gemm, and copies the outputs back."""
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    dev = stream.device
    xh = [x.cpu().pin_memory() for (_, _, x) in layers]
    yh = [torch.empty((wk.M, wk.G, wk.N), dtype=torch.bfloat16).pin_memory() for _ in layers]
    xd = [torch.empty_like(x, device=dev) for x in xh]
    yd = [torch.empty((wk.M, wk.G, wk.N), dtype=torch.bfloat16, device=dev) for _ in layers]

    def step():
        for (w8, ex, _), a, b, xa, yb in zip(layers, xh, yh, xd, yd):
            xa.copy_(a, non_blocking=True)
            bsf8.gemm(xa, w8, ex, split_k=wk.split_k, out=yb)
            b.copy_(yb, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        stream.synchronize()
    h2d = sum(x.numel() * x.element_size() for x in xh)
    d2h = sum(y.numel() * y.element_size() for y in yh)
    return e0.elapsed_time(e1) / 1e3, h2d, d2h


def profile_load_time(which, calls, device):
    """Profiling mode for the load-time rows: `calls` eager calls over distinct copies."""
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    from block_scaled_fp8_weight_gb300 import workloads as wl
    wk = wl.DOWN_PROJ if which == "pad_k" else wl.WO_A
    copies = min(calls, 8)
    twins = [wk.weights(copy=c) for c in range(copies)]
    w8s = [torch.from_numpy(a).to(device) for a, _ in twins]
    exs = [torch.from_numpy(b).to(device) for _, b in twins]
    wbf = [bsf8.dequant(a, b) for a, b in zip(w8s, exs)] if which == "make_twin" else None
    torch.cuda.synchronize(device)
    for i in range(calls):
        c = i % copies
        if which == "make_twin":
            bsf8.make_twin(wbf[c])
        elif which == "dequant":
            bsf8.dequant(w8s[c], exs[c])
        else:
            bsf8.pad_k(w8s[c], exs[c], 640, pad_exp=127)
    torch.cuda.synchronize(device)
    return 0


L2_BYTES = 129e6   # GB300 L2; weight copies are cycled so that each config streams >= 2x this


def copies_for(nbytes: int, least: int = 43, most: int = 2048) -> int:
    """Distinct input copies a config cycles through: at least 43 (one per layer, as on the
    pages) and enough that a pass streams at least twice the L2."""
    return int(max(least, min(most, -(-int(2 * L2_BYTES) // max(1, int(nbytes))))))


def configs_map(device, peak, verbose=False):
    """Every config of the hot path timed on the GPU: each row's calls in a CUDA graph of a
    dependent chain (PDL on) over enough distinct seeded copies that a pass streams at
    least twice the L2, replayed `reps` times with an event pair per replay; us/call is the
    median over replays (p10/p90 beside it).  GB/s counts the weight stream (codes +
    exponent bytes) for the GEMM rows and all bytes moved for make_twin, dequant and pad-K."""
    import ctypes
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    from block_scaled_fp8_weight_gb300 import workloads as wl
    lib = bsf8.load()
    stream = torch.cuda.Stream(device=device)
    out = {}
    t_start = time.time()

    def graph_time(calls, reps):
        with torch.cuda.stream(stream):
            for c in calls:
                c()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in calls:
                    c()
            for _ in range(3):
                g.replay()
            stream.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
            ev[0].record(stream)
            for i in range(reps):
                g.replay()
                ev[i + 1].record(stream)
            stream.synchronize()
        if bsf8.device_status() != 0:
            raise RuntimeError("a kernel reported a timeout")
        per = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e-3 / len(calls) for i in range(reps))
        q = lambda f: per[min(len(per) - 1, int(f * len(per)))]
        return q(0.5), q(0.1), q(0.9)

    def emit(row, t, nbytes, copies, **extra):
        t50, t10, t90 = t
        e = {"us": round(t50 * 1e6, 3), "us_p10": round(t10 * 1e6, 3), "us_p90": round(t90 * 1e6, 3),
             "GBps": round(nbytes / t50 / 1e9, 1), "frac": round(nbytes / t50 / 1e9 / peak, 4),
             "copies": copies}
        e.update(extra)
        out[row] = e
        if verbose:
            print(json.dumps({"row": row, **e}), flush=True)

    sp = lambda: ctypes.c_void_p(stream.cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    reps_for = lambda per_call_s, ncalls: int(min(200, max(5, 0.03 / max(1e-7, per_call_s * ncalls))))

    # a1 make_twin and a2' dequant on the wo_a shape; a7 pad-K on down_proj
    wk = wl.WO_A
    G, N, K = wk.G, wk.N, wk.K
    n = copies_for(3 * G * N * K)
    twins = [wk.weights(copy=c) for c in range(n)]
    w8s = [torch.from_numpy(a).to(device) for a, _ in twins]
    exs = [torch.from_numpy(b).to(device) for _, b in twins]
    wbf = [bsf8.dequant(a, b) for a, b in zip(w8s, exs)]
    o8 = [torch.empty_like(a) for a in w8s]
    oe = [torch.empty_like(b) for b in exs]
    ok = [torch.empty_like(b) for b in exs]
    acc = torch.empty((n,), dtype=torch.int32, device=device)
    calls = [lambda i=i: lib.bsf8_make_twin(ptr(wbf[i]), ptr(o8[i]), ptr(oe[i]), ptr(ok[i]),
                                            ctypes.c_void_p(acc.data_ptr() + 4 * i), G, N, K, sp())
             for i in range(n)]
    emit("a1 make_twin wo_a", graph_time(calls, 10), 3 * G * N * K + 2 * G * (N // 32) * (K // 32), n)
    outs = [torch.empty((G, N, K), dtype=torch.bfloat16, device=device) for _ in range(n)]
    calls = [lambda i=i: lib.bsf8_dequant(ptr(w8s[i]), ptr(exs[i]), ptr(outs[i]), G, N, K, sp())
             for i in range(n)]
    emit("a2' dequant wo_a", graph_time(calls, 10), 3 * G * N * K + G * (N // 32) * (K // 32), n)
    del wbf, o8, oe, ok, outs, w8s, exs, twins
    dk = wl.DOWN_PROJ
    Kp = 640
    n = copies_for(dk.N * (dk.K + Kp))
    dt = [dk.weights(copy=c) for c in range(n)]
    dw = [torch.from_numpy(a).to(device) for a, _ in dt]
    de = [torch.from_numpy(b).to(device) for _, b in dt]
    pw = [torch.empty((1, dk.N, Kp), dtype=torch.uint8, device=device) for _ in range(n)]
    pe = [torch.empty((1, dk.N // 32, Kp // 32), dtype=torch.uint8, device=device) for _ in range(n)]
    calls = [lambda i=i: lib.bsf8_pad_k(ptr(dw[i]), ptr(de[i]), ptr(pw[i]), ptr(pe[i]), 1, dk.N, dk.K,
                                        Kp, 127, sp()) for i in range(n)]
    emit("a7 pad_k down_proj 576->640", graph_time(calls, 20),
         dk.N * dk.K + dk.N * Kp + (dk.N // 32) * (dk.K // 32 + Kp // 32), n)
    del dt, dw, de, pw, pe

    cache = {}

    def weights_of(wk, copies):
        key = (wk.name, wk.K, copies)
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[key] = [tuple(torch.from_numpy(a).to(device) for a in wk.weights(copy=c))
                          for c in range(copies)]
        return cache[key]

    def gemm_time(wk, M, S, copies=None):
        copies = copies or copies_for(wk.weight_bytes)
        layers = []
        for c, (w8, ex) in enumerate(weights_of(wk, copies)):
            x = wk.x(copy=c, M=M)
            layers.append((w8, ex, torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(device)))
        ys = [torch.empty((M, wk.G, wk.N), dtype=torch.bfloat16, device=device) for _ in layers]
        need = bsf8.workspace_bytes(M, wk.N, wk.K, wk.G, S)
        wss = [torch.empty(max(16, need), dtype=torch.uint8, device=device) for _ in layers] if need else [None] * copies
        calls = [lambda l=l, y=y, w=w: bsf8.gemm(l[2], l[0], l[1], split_k=S, out=y, workspace=w)
                 for l, y, w in zip(layers, ys, wss)]
        t = graph_time(calls, reps_for(wk.weight_bytes / 2e12, copies))
        S_used = S or bsf8.auto_split(M, wk.N, wk.K, wk.G)
        kern = bsf8.KERNELS[bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, S)]
        return t, {"M": M, "S": S_used, "kernel": kern, "launches_per_call": 2 if need else 1}, copies

    def gemm_row(row, wk, M, S, copies=None):
        t, info, copies = gemm_time(wk, M, S, copies)
        emit(row, t, wk.weight_bytes, copies, **info)

    gemm_row("C1 tiny M=4 S=1", wl.TINY, 4, 1)
    gemm_row("C1 tiny M=4 S=4", wl.TINY, 4, 4)
    for M in wl.WO_A_ROWS:
        gemm_row(f"C2 wo_a M={M} S=8", wl.WO_A, M, 8)
    gemm_row("C3 down_proj K=576 M=6", wl.DOWN_PROJ, 6, 0)
    gemm_row("C3 down_proj K=640 M=6", dataclasses.replace(wl.DOWN_PROJ, K=640), 6, 0)
    for M in wl.MID_ROWS:                      # each split of the sweep, the best reported
        per_s = {}
        for S in wl.MID_SPLITS:
            per_s[S] = gemm_time(wl.MID, M, S)
        best = min(per_s, key=lambda S: per_s[S][0][0])
        t, info, copies = per_s[best]
        emit(f"C4 mid M={M}", t, wl.MID.weight_bytes, copies, **info,
             us_by_split={str(S): round(v[0][0] * 1e6, 3) for S, v in per_s.items()},
             kernel_by_split={str(S): v[1]["kernel"] for S, v in per_s.items()})
    for M in wl.SWEEP_ROWS:
        gemm_row(f"C5 gate_up N=1152 K=5120 M={M}", wl.GATE_UP, M, 0)
    for M in wl.SWEEP_ROWS:
        gemm_row(f"C5 head N=32768 K=5120 M={M}", wl.HEAD, M, 0, copies=3)

    # f3: per-(row, 32-column) scales at the draft main_proj shape (1280 x 5120)
    N1, K1 = 1280, 5120
    n = copies_for(N1 * K1 + N1 * K1 // 32, least=40)
    rng = wl.rng(90)
    rw8 = [torch.from_numpy(wl.codes(rng, (1, N1, K1))).to(device) for _ in range(n)]
    rex = [torch.from_numpy(wl.exponents(rng, (1, N1, K1 // 32), 110, 130)).to(device) for _ in range(n)]
    rbf = [bsf8.dequant_rows(a, b) for a, b in zip(rw8, rex)]
    o8 = [torch.empty_like(a) for a in rw8]
    oe = [torch.empty_like(b) for b in rex]
    okr = [torch.empty_like(b) for b in rex]
    acc = torch.empty((n,), dtype=torch.int32, device=device)
    calls = [lambda i=i: lib.bsf8_make_twin_rows(ptr(rbf[i]), ptr(o8[i]), ptr(oe[i]), ptr(okr[i]),
                                                 ctypes.c_void_p(acc.data_ptr() + 4 * i), 1, N1, K1, sp())
             for i in range(n)]
    emit("f3 rows make_twin 1280x5120", graph_time(calls, 20), N1 * K1 * 3 + 2 * N1 * K1 // 32, n)
    calls = [lambda i=i: lib.bsf8_dequant_rows(ptr(rw8[i]), ptr(rex[i]), ptr(rbf[i]), 1, N1, K1, sp())
             for i in range(n)]
    emit("f3 rows dequant 1280x5120", graph_time(calls, 20), N1 * K1 * 3 + N1 * K1 // 32, n)
    wbytes = N1 * K1 + N1 * K1 // 32
    for M in (1, 6, 16):
        xs = [torch.from_numpy(wl.activations(rng, M, K1).view("int16")).view(torch.bfloat16).to(device)
              for _ in range(n)]
        ys = [torch.empty((M, 1, N1), dtype=torch.bfloat16, device=device) for _ in range(n)]
        calls = [lambda i=i: bsf8.gemm_rows(xs[i], rw8[i], rex[i], out=ys[i]) for i in range(n)]
        emit(f"f3 rows gemm 1280x5120 M={M}", graph_time(calls, 50), wbytes, n, M=M)
        del xs, ys
    del rw8, rex, rbf, o8, oe, okr

    # f2: fp32 output on the head-like weight (partials of the kernel the shape selects,
    # summed over the splits in fp32)
    for M in (6, 64, 128):
        wk = wl.HEAD
        layers = []
        for c, (w8, ex) in enumerate(weights_of(wk, 3)):
            x = wk.x(copy=c, M=M)
            layers.append((w8, ex, torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(device)))
        S = bsf8.auto_split(M, wk.N, wk.K, wk.G)
        Ps = [torch.empty((S, M, wk.G, wk.N), dtype=torch.float32, device=device) for _ in layers]
        ys = [torch.empty((M, wk.G, wk.N), dtype=torch.float32, device=device) for _ in layers]
        calls = [lambda l=l, P=P, y=y: (bsf8.gemm_partials(l[2], l[0], l[1], S, out=P),
                                        bsf8.splitk_reduce_f32(P, out=y) if S > 1 else None)
                 for l, P, y in zip(layers, Ps, ys)]
        emit(f"f2 fp32 out head M={M}", graph_time(calls, 10), wk.weight_bytes, 3, M=M, S=S,
             kernel=bsf8.KERNELS[bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, S)])
        del layers, Ps, ys

    # f1: past 192 rows (prefill-sized calls from the twin), also against the bf16 peak
    bf16_peak = measured_bf16_tflops()
    for wk, M, copies in ((wl.MID, 1024, 16), (wl.MID, 4096, 4), (wl.HEAD, 512, 2), (wl.HEAD, 2048, 2)):
        layers = []
        for c, (w8, ex) in enumerate(weights_of(wk, copies)):
            x = wk.x(copy=c, M=M)
            layers.append((w8, ex, torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(device)))
        ys = [torch.empty((M, wk.G, wk.N), dtype=torch.bfloat16, device=device) for _ in layers]
        need = bsf8.workspace_bytes(M, wk.N, wk.K, wk.G, 0)
        ws = torch.empty(max(16, need), dtype=torch.uint8, device=device)
        calls = [lambda l=l, y=y: bsf8.gemm(l[2], l[0], l[1], split_k=0, out=y, workspace=ws)
                 for l, y in zip(layers, ys)]
        t = graph_time(calls, 5)
        tf = 2.0 * M * wk.G * wk.N * wk.K / t[0] / 1e12
        emit(f"f1 large-M {'mid G=4 1024x4096' if wk is wl.MID else 'head 32768x5120'} M={M}", t,
             wk.weight_bytes, copies, M=M, S=bsf8.auto_split(M, wk.N, wk.K, wk.G),
             kernel=bsf8.KERNELS[bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, 0)],
             TFLOPs=round(tf, 1), frac_bf16=round(tf / bf16_peak, 4))
        del layers, ys, ws
    cache.clear()
    torch.cuda.empty_cache()
    out["_seconds"] = round(time.time() - t_start, 1)
    return out


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    from block_scaled_fp8_weight_gb300 import build as bsf8_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libbsf8 has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, True)
    bsf8_build.build()
    bsf8.load()
    if args.suite:
        configs_map(device, measured_peaks()[0], verbose=True)
        return 0
    wk = workload()
    if args.profile_calls and args.workload in ("make_twin", "dequant", "pad_k"):
        return profile_load_time(args.workload, args.profile_calls, device)
    if args.profile_calls:
        from block_scaled_fp8_weight_gb300 import workloads as wl
        wk = {"wo_a": wl.WO_A, "down_proj": wl.DOWN_PROJ, "mid": wl.MID, "gate_up": wl.GATE_UP,
              "head": wl.HEAD}[args.workload]
    import dataclasses
    if args.split_k is not None:
        wk = dataclasses.replace(wk, split_k=args.split_k)
    if args.m is not None:
        wk = dataclasses.replace(wk, M=args.m)
    copies = LAYERS if wk.copies > 1 else 3
    if args.profile_calls and args.copies:
        copies = args.copies
    layers = build_layers(wk, device, copies=copies)
    stream = torch.cuda.Stream(device=device)
    if args.profile_calls:
        with torch.cuda.stream(stream):
            for i in range(args.profile_calls):
                w8, ex, x = layers[i % len(layers)]
                bsf8.gemm(x, w8, ex, split_k=wk.split_k)
        torch.cuda.synchronize(device)
        return 0

    # Variants first (untimed for the headline): eager launches, graph without PDL, and one
    # launch on its own (L2 flushed before each) for the launch duration in isolation.
    t_eager = time_eager(layers, wk, max(1, args.steps // 20), stream)
    t_iso = time_isolated(layers, wk, 20, stream)
    t_nopdl, _, _, _ = time_graph(layers, wk, max(1, args.steps // 4), max(3, args.warmup), False, stream)
    broken = {m: time_broken_chain(layers, wk, max(2, args.steps // 4), stream, m) * 1e6
              for m in ("sleep", "plain", "prefetch")}

    nsm = torch.cuda.get_device_properties(device).multi_processor_count
    probe = [torch.zeros((nsm, 2), dtype=torch.int64, device=device) for _ in range(2)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    elapsed, w0, w1, steps_s = time_graph(layers, wk, args.steps, max(3, args.warmup), True, stream,
                                          per_step=True, clock_probe=probe)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(w0, w1)
    clocks["in_region"] = region_clock(probe)

    calls = LAYERS * args.steps
    t_job, bytes_job = aggregate(dist, elapsed, float(wk.weight_bytes) * calls, device)
    value = bytes_job / t_job / 1e9
    us_call = elapsed / calls * 1e6
    per_call = sorted(t / LAYERS * 1e6 for t in steps_s)
    q = lambda f: per_call[min(len(per_call) - 1, int(f * len(per_call)))]

    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    t_e2e, h2d, d2h = time_e2e(layers, wk, e2e_steps, stream)
    t_e2e_job, bytes_e2e = aggregate(dist, t_e2e, float(wk.weight_bytes) * LAYERS * e2e_steps, device)

    peak, peak_kind = measured_peaks()
    achieved = wk.algorithmic_bytes / (elapsed / calls) / 1e9
    traffic = recorded_traffic()
    import block_scaled_fp8_weight_gb300 as bsf8
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_job / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(wk), "us_per_call": us_call,
        "us_per_call_by_step": {"median": q(0.5), "p10": q(0.1), "p90": q(0.9), "steps": len(per_call)},
        "frac_of_peak": {"measured": value / world / peak, "nominal_7900": value / world / 7900.0},
        "gpu_launches": calls,
        "kernel": bsf8.KERNELS[bsf8.gemm_kernel(wk.M, wk.N, wk.K, wk.G, wk.split_k)],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": KERNEL_NAME,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json, burst copy)",
                     "algorithmic_bytes_per_launch": wk.algorithmic_bytes,
                     "launch_time": "timed-region time / launches: consecutive launches overlap "
                                    "(programmatic dependent launch), so the per-launch time is "
                                    "the interval between launch completions",
                     "isolated_launch_us": t_iso * 1e6},
        "e2e": {"value": bytes_e2e / t_e2e_job / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_call": t_e2e / (LAYERS * e2e_steps) * 1e6,
                "steps": e2e_steps, "path": "bsf8.gemm, eager, pinned host x -> device -> host y"},
        "clocks": clocks,
        "variants": {
            "graph_no_pdl_us_per_call": t_nopdl / (LAYERS * max(1, args.steps // 4)) * 1e6,
            "eager_us_per_call": t_eager / (LAYERS * max(1, args.steps // 20)) * 1e6,
            "chain_broken_by_a_foreign_kernel": {
                "what": "each layer's GEMM after a ~10 us spin kernel that is not this library's "
                        "(it does not let the GEMM start early); us per layer",
                "spin_alone_us": broken["sleep"], "spin_then_gemm_us": broken["plain"],
                "spin_then_gemm_with_l2_prefetch_us": broken["prefetch"],
                "gemm_us_without_prefetch": broken["plain"] - broken["sleep"],
                "gemm_us_with_prefetch": broken["prefetch"] - broken["sleep"]},
        },
    }
    if rank == 0 and world == 1 and not args.no_configs:
        line["configs"] = configs_map(device, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_baseline(wk, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
