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
memory and the outputs copied back inside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bsf8|reference]

`--impl reference` times the CPU oracle (oracle/, a plain C restatement of the pages)
on a bounded sample of the same workload: the baseline this library is compared with.
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the op has no
exchange step, so no collective runs on the data path; only the timing is combined
(max over ranks) and the bytes summed.
"""
from __future__ import annotations

import argparse
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
    p.add_argument("--suite", action="store_true",
                   help="time every hot-path row (make_twin, dequant, pad-K, the GEMM at every "
                        "config) and print one JSON line per row instead of the headline line")
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
    """Samples nvidia-smi SM clocks and throttle reasons every 100 ms in the background."""

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
            self._stop.wait(0.1)

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


def cpu_oracle_baseline(wk, seconds: float):
    """The oracle, as it stands, on one host core: whole wo_a layer calls at M=6."""
    import oracle
    w8, ex = wk.weights(copy=0)
    x = wk.x(copy=0)
    oracle.gemm(x, w8, ex)                       # load + first touch
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.gemm(x, w8, ex)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": wk.weight_bytes * calls / el / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle", "us_per_call": el / calls * 1e6,
            "sample": f"{calls} whole wo_a layer calls (G=2, N=1024, K=4096, M=6), "
                      f"{el:.1f} s on one host core"}


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step is a bounded slice of one layer
    call (a contiguous range of weight rows), timed on one host core."""
    if rank != 0:
        return None
    import oracle
    wk = workload()
    w8, ex = wk.weights(copy=0)
    x = wk.x(copy=0)
    budget = 90.0
    probe_rows = 32
    t0 = time.perf_counter()
    oracle.gemm(x, w8[:, :probe_rows], ex[:, :probe_rows // 32])
    t_probe = max(time.perf_counter() - t0, 1e-6)
    per_step = budget / max(1, args.steps + args.warmup)
    rows = int(min(wk.N, max(probe_rows, (per_step / t_probe) * probe_rows)) // 32 * 32)
    rows = max(32, rows)
    ws, es = w8[:, :rows], ex[:, :rows // 32]
    for _ in range(args.warmup):
        oracle.gemm(x, ws, es)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm(x, ws, es)
    el = time.perf_counter() - t0
    bytes_step = wk.G * rows * wk.K + wk.G * (rows // 32) * (wk.K // 32)
    value = bytes_step * args.steps / el / 1e9
    sample = (f"each step: rows [0, {rows}) of both groups of one wo_a layer (M=6), "
              f"{rows / wk.N:.4f} of a layer call, one host core")
    cfg = config_dict(wk, pdl=False)
    cfg["launch"] = "CPU oracle (plain C, binary32 index-order sum), single thread"
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": cfg, "impl": "reference",
        "us_per_call": el / args.steps * 1e6 * wk.N / rows,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
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


def time_graph(layers, wk, steps, warmup, pdl, stream, sampler=None):
    """Captures the 43 calls of one step in a CUDA graph; replays `warmup` untimed then
    `steps` timed steps; returns (seconds, wall t0, wall t1)."""
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    bsf8.set_option(bsf8.OPT_PDL, 1 if pdl else 0)
    outs = [torch.empty((wk.M, wk.G, wk.N), dtype=torch.bfloat16, device=stream.device) for _ in layers]
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
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            w0 = time.time()
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
            stream.synchronize()
            w1 = time.time()
    finally:
        bsf8.set_option(bsf8.OPT_PDL, 1)
    return e0.elapsed_time(e1) / 1e3, w0, w1


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


def run_suite(device, peak):
    """Every hot-path row timed on the GPU: each call of a row in a CUDA graph over enough
    distinct seeded copies that the inputs exceed the L2 (PDL on), reported as us/call and
    as bytes moved per call (the row's algorithmic bytes) over time, against the HBM peak."""
    import ctypes
    import torch
    import block_scaled_fp8_weight_gb300 as bsf8
    from block_scaled_fp8_weight_gb300 import workloads as wl
    lib = bsf8.load()
    stream = torch.cuda.Stream(device=device)
    out = []

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
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            stream.synchronize()
        if bsf8.device_status() != 0:
            raise RuntimeError("a kernel reported a timeout")
        return e0.elapsed_time(e1) * 1e-3 / (reps * len(calls))

    def emit(row, config, t, nbytes, weight_bytes=None):
        line = {"row": row, "config": config, "us_per_call": t * 1e6,
                "GBps": nbytes / t / 1e9, "frac_of_hbm_peak": nbytes / t / 1e9 / peak,
                "bytes_per_call": nbytes}
        if weight_bytes is not None:
            line["weight_stream_GBps"] = weight_bytes / t / 1e9
            line["weight_frac"] = weight_bytes / t / 1e9 / peak
        out.append(line)
        print(json.dumps(line), flush=True)

    sp = lambda: ctypes.c_void_p(stream.cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    # make_twin and dequant on the wo_a shape, 43 copies (cold)
    wk = wl.WO_A
    G, N, K = wk.G, wk.N, wk.K
    twins = [wk.weights(copy=c) for c in range(LAYERS)]
    w8s = [torch.from_numpy(a).to(device) for a, _ in twins]
    exs = [torch.from_numpy(b).to(device) for _, b in twins]
    wbf = [bsf8.dequant(a, b) for a, b in zip(w8s, exs)]
    o8 = [torch.empty_like(a) for a in w8s]
    oe = [torch.empty_like(b) for b in exs]
    ok = [torch.empty_like(b) for b in exs]
    acc = torch.empty((LAYERS,), dtype=torch.int32, device=device)
    calls = [lambda i=i: lib.bsf8_make_twin(ptr(wbf[i]), ptr(o8[i]), ptr(oe[i]), ptr(ok[i]),
                                            ctypes.c_void_p(acc.data_ptr() + 4 * i), G, N, K, sp())
             for i in range(LAYERS)]
    t = graph_time(calls, 20)
    emit("a1 make_twin", f"G={G} N={N} K={K} bf16 -> twin, {LAYERS} copies", t,
         2 * G * N * K + G * N * K + 2 * G * (N // 32) * (K // 32))
    outs = [torch.empty((G, N, K), dtype=torch.bfloat16, device=device) for _ in range(LAYERS)]
    calls = [lambda i=i: lib.bsf8_dequant(ptr(w8s[i]), ptr(exs[i]), ptr(outs[i]), G, N, K, sp())
             for i in range(LAYERS)]
    t = graph_time(calls, 20)
    emit("a2' dequant", f"G={G} N={N} K={K} twin -> bf16, {LAYERS} copies", t,
         G * N * K + G * (N // 32) * (K // 32) + 2 * G * N * K)
    del wbf, o8, oe, ok, outs
    # pad-K on the down_proj twin (576 -> 640), 43 copies
    dk = wl.DOWN_PROJ
    dt = [dk.weights(copy=c) for c in range(LAYERS)]
    dw = [torch.from_numpy(a).to(device) for a, _ in dt]
    de = [torch.from_numpy(b).to(device) for _, b in dt]
    Kp = 640
    pw = [torch.empty((1, dk.N, Kp), dtype=torch.uint8, device=device) for _ in range(LAYERS)]
    pe = [torch.empty((1, dk.N // 32, Kp // 32), dtype=torch.uint8, device=device) for _ in range(LAYERS)]
    calls = [lambda i=i: lib.bsf8_pad_k(ptr(dw[i]), ptr(de[i]), ptr(pw[i]), ptr(pe[i]), 1, dk.N, dk.K,
                                        Kp, 127, sp()) for i in range(LAYERS)]
    t = graph_time(calls, 50)
    emit("a7 pad_k", f"N={dk.N} K={dk.K} -> {Kp}, {LAYERS} copies", t,
         dk.N * dk.K + dk.N * Kp + (dk.N // 32) * (dk.K // 32 + Kp // 32))
    del w8s, exs, twins

    cache = {}

    def weights_of(wk, copies):
        key = (wk.name, wk.K, copies)
        if key not in cache:
            cache.clear()
            cache[key] = [tuple(torch.from_numpy(a).to(device) for a in wk.weights(copy=c))
                          for c in range(copies)]
        return cache[key]

    def gemm_row(name, wk, M, S, copies):
        layers = []
        for c, (w8, ex) in enumerate(weights_of(wk, copies)):
            x = wk.x(copy=c, M=M)
            layers.append((w8, ex, torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(device)))
        ys = [torch.empty((M, wk.G, wk.N), dtype=torch.bfloat16, device=device) for _ in layers]
        need = bsf8.workspace_bytes(M, wk.N, wk.K, wk.G, S)
        wss = [torch.empty(max(16, need), dtype=torch.uint8, device=device) for _ in layers] if need else [None] * copies
        calls = [lambda l=l, y=y, w=w: bsf8.gemm(l[2], l[0], l[1], split_k=S, out=y, workspace=w)
                 for l, y, w in zip(layers, ys, wss)]
        t = graph_time(calls, min(200, max(3, int(2e-3 / max(1e-6, wk.weight_bytes / 4e12)))))
        xy = M * wk.G * wk.K * 2 + M * wk.G * wk.N * 2
        emit(name, f"G={wk.G} N={wk.N} K={wk.K} M={M} split_k={S or 'auto'}, {copies} copies", t,
             wk.weight_bytes + xy, wk.weight_bytes)

    gemm_row("a3-a6 gemm tiny", wl.TINY, 4, 1, LAYERS)
    gemm_row("a3-a6 gemm tiny", wl.TINY, 4, 4, LAYERS)
    for M in (2, 4, 6, 8):
        gemm_row("a3-a6 gemm wo_a", wl.WO_A, M, 8, LAYERS)
    gemm_row("a3-a6 gemm down_proj K=576", wl.DOWN_PROJ, 6, 0, LAYERS)
    import dataclasses
    gemm_row("a3-a6 gemm down_proj K=640", dataclasses.replace(wl.DOWN_PROJ, K=640), 6, 0, LAYERS)
    for M in (9, 16, 32, 64, 96, 128, 192):
        for S in (1, 2, 4, 8):
            gemm_row("a3-a6 gemm mid", wl.MID, M, S, LAYERS)
    for M in (1, 2, 6, 16, 64, 128):
        gemm_row("a3-a6 gemm gate_up", wl.GATE_UP, M, 0, LAYERS)
    for M in (1, 2, 6, 16, 64, 128):
        gemm_row("a3-a6 gemm head", wl.HEAD, M, 0, 3)

    # per-(row, 32-column) scales (the draft main_proj's layout): twin, dequant and GEMM at
    # its shape (1280 output rows, K = 5120), 43 copies
    N1, K1 = 1280, 5120
    rng = wl.rng(90)
    rw8 = [torch.from_numpy(wl.codes(rng, (1, N1, K1))).to(device) for _ in range(LAYERS)]
    rex = [torch.from_numpy(wl.exponents(rng, (1, N1, K1 // 32), 110, 130)).to(device) for _ in range(LAYERS)]
    rbf = [bsf8.dequant_rows(a, b) for a, b in zip(rw8, rex)]
    o8 = [torch.empty_like(a) for a in rw8]
    oe = [torch.empty_like(b) for b in rex]
    ok = [torch.empty_like(b) for b in rex]
    acc = torch.empty((LAYERS,), dtype=torch.int32, device=device)
    calls = [lambda i=i: lib.bsf8_make_twin_rows(ptr(rbf[i]), ptr(o8[i]), ptr(oe[i]), ptr(ok[i]),
                                                 ctypes.c_void_p(acc.data_ptr() + 4 * i), 1, N1, K1, sp())
             for i in range(LAYERS)]
    t = graph_time(calls, 50)
    emit("f3 rows make_twin", f"N={N1} K={K1} bf16 -> twin, {LAYERS} copies", t, N1 * K1 * 3 + 2 * N1 * K1 // 32)
    calls = [lambda i=i: lib.bsf8_dequant_rows(ptr(rw8[i]), ptr(rex[i]), ptr(rbf[i]), 1, N1, K1, sp())
             for i in range(LAYERS)]
    t = graph_time(calls, 50)
    emit("f3 rows dequant", f"N={N1} K={K1} twin -> bf16, {LAYERS} copies", t, N1 * K1 * 3 + N1 * K1 // 32)
    wbytes = N1 * K1 + N1 * K1 // 32
    for M in (1, 6, 16):
        xs = [torch.from_numpy(wl.activations(rng, M, K1).view("int16")).view(torch.bfloat16).to(device)
              for _ in range(LAYERS)]
        ys = [torch.empty((M, 1, N1), dtype=torch.bfloat16, device=device) for _ in range(LAYERS)]
        calls = [lambda i=i: bsf8.gemm_rows(xs[i], rw8[i], rex[i], out=ys[i]) for i in range(LAYERS)]
        t = graph_time(calls, 100)
        emit("f3 rows gemm", f"N={N1} K={K1} M={M} split_k=auto, {LAYERS} copies", t,
             wbytes + M * K1 * 2 + M * N1 * 2, wbytes)
        del xs, ys
    del rw8, rex, rbf, o8, oe, ok

    # fp32 output (the draft head's fp32 logits): partials of the kernel the shape selects,
    # summed over the splits in fp32
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
        t = graph_time(calls, 20)
        xy = M * wk.G * wk.K * 2 + M * wk.G * wk.N * 4
        emit("f2 gemm fp32 out", f"G={wk.G} N={wk.N} K={wk.K} M={M} split_k={S}, 3 copies", t,
             wk.weight_bytes + xy, wk.weight_bytes)
        del layers, Ps, ys

    # Past 192 rows (prefill-sized calls, the pages' drop mode served from the twin): bound by
    # the tensor cores, so reported against the measured dense bf16 peak too.  The calls of a
    # row share one workspace: they run one after another on the stream.
    bf16_peak = measured_bf16_tflops()
    for wk, M, copies in ((wl.MID, 1024, 8), (wl.MID, 4096, 4), (wl.HEAD, 512, 2), (wl.HEAD, 2048, 2)):
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
        flops = 2.0 * M * wk.G * wk.N * wk.K
        xy = M * wk.G * wk.K * 2 + M * wk.G * wk.N * 2
        emit("f1 gemm large-M", f"G={wk.G} N={wk.N} K={wk.K} M={M} split_k=auto, {copies} copies", t,
             wk.weight_bytes + xy, wk.weight_bytes)
        out[-1]["TFLOPs"] = flops / t / 1e12
        out[-1]["frac_of_bf16_peak"] = flops / t / 1e12 / bf16_peak
        print(json.dumps({"row": "f1 gemm large-M", "M": M, "TFLOPs": out[-1]["TFLOPs"],
                          "frac_of_bf16_peak": out[-1]["frac_of_bf16_peak"]}), flush=True)
        del layers, ys, ws
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
        run_suite(device, measured_peaks()[0])
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
    layers = build_layers(wk, device, copies=LAYERS if wk.copies > 1 else 3)
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
    t_nopdl, _, _ = time_graph(layers, wk, max(1, args.steps // 4), max(3, args.warmup), False, stream)

    sampler = ClockSampler(local)
    sampler.start()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    elapsed, w0, w1 = time_graph(layers, wk, args.steps, max(3, args.warmup), True, stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(w0, w1)

    calls = LAYERS * args.steps
    t_job, bytes_job = aggregate(dist, elapsed, float(wk.weight_bytes) * calls, device)
    value = bytes_job / t_job / 1e9
    us_call = elapsed / calls * 1e6

    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    t_e2e, h2d, d2h = time_e2e(layers, wk, e2e_steps, stream)
    t_e2e_job, bytes_e2e = aggregate(dist, t_e2e, float(wk.weight_bytes) * LAYERS * e2e_steps, device)

    peak, peak_kind = measured_peaks()
    achieved = wk.algorithmic_bytes / (elapsed / calls) / 1e9
    traffic = recorded_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_job / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(wk), "us_per_call": us_call,
        "frac_of_peak": {"measured": value / world / peak, "nominal_7900": value / world / 7900.0},
        "gpu_launches": calls,
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
        },
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_baseline(wk, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
