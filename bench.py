#!/usr/bin/env python3
"""Benchmark of the GB300 LiSA forward layer.

One step = one LiSA forward (every kernel of the chain) over one batch of the
PVT-T stage-1 shaped layer: B=32, heads=1, 56x56 grid (n=3136), d_h=d_v=64,
bf16, T=3, geometric beta=0.5, alpha=0.5, seeded synthetic N(0,1) inputs.

Prints one JSON line (rank 0):
  value      tokens*heads per second over the timed K steps, inputs resident
             in HBM, 8 rotating input sets (> 3x the 129 MB L2) so no step
             reads its inputs from L2 left by the previous one;
  e2e        the same metric through lisa_forward_host: pinned host inputs
             copied in and the output copied back inside every step;
  roofline   the dominant kernel's algorithmic bytes per launch over its mean
             launch time (CUDA events between the kernels of a separate pass),
             against the measured HBM copy bandwidth;
  cpu_baseline  the double-precision oracle on the host cores, one slice of
             the same workload per repetition.

--impl reference times that oracle as the reference arm (each step = one
slice of the workload on all host cores).

Multi-GPU: slices are independent (no collective on the path), so every rank
runs its own batch (weak scaling); value = all ranks' tokens*heads over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LiSA fwd tokens·heads/s at n=3136 bf16; % of HBM roofline (ncu GB/s)"
UNIT = "tokens·heads/s"
DEFAULT_WORKLOAD = "pvt_t_s1_56x56_T3"
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--pass", dest="direction", choices=["forward", "backward"], default="forward",
                    help="forward (the headline) or the backward pass (lisa_backward)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=16.0,
                    help="wall-time budget of the cpu_baseline sample (half on all cores, half on one)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's value (a collective over the default process group
    when world > 1; identity otherwise)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_throughput(world: int, units_per_rank: int, steps: int, ms_max: float) -> float:
    """Whole-job units per second: every rank processed its own batch of
    `units_per_rank` per step; the job took the slowest rank's time."""
    return world * units_per_rank * steps / (ms_max / 1e3)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# -- clocks during the timed region ---------------------------------------------------

class ClockSampler:
    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = bus_id
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv",
                                          "-lms", "20"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        text = self.tmp.read()
        self.tmp.close()
        os.unlink(self.tmp.name)
        rows = []
        for row in csv.reader(io.StringIO(text)):
            if len(row) < 9 or row[0].strip().startswith("pci"):
                continue
            rows.append([c.strip() for c in row])
        mine = [r for r in rows if self.bus_id and self.bus_id.lower() in r[0].lower()] or rows
        def num(x):
            try:
                return float(x.split()[0])
            except (ValueError, IndexError):
                return None
        sm = [num(r[1]) for r in mine if num(r[1]) is not None]
        mx = [num(r[2]) for r in mine if num(r[2]) is not None]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in mine:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        loaded = [x for x in sm if mx and x > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(mine)}


# -- peaks, traffic ---------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# The files the forward kernels are built from (the kernels whose DRAM
# traffic profiles/traffic.json records): a change to their code voids
# the recorded counters; comments and other kernels' sources do not.
TRAFFIC_SOURCES = ("hop_stochastic_vision_gb300/csrc/lisa_tc.cu", "hop_stochastic_vision_gb300/csrc/lisa_tc_common.cuh",
                   "hop_stochastic_vision_gb300/csrc/lisa_sm100.cuh",
                   "hop_stochastic_vision_gb300/csrc/lisa_solve.cuh", "hop_stochastic_vision_gb300/csrc/lisa_simt.cu",
                   "hop_stochastic_vision_gb300/csrc/lisa_internal.h", "include/lisa.h")


def _code_only(text: str) -> str:
    """The source with its comments and blank space removed: what the compiler
    sees of it, so an edit to a comment does not void the recorded counters."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash() -> str:
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(os.path.basename(rel).encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, only
    if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    if data.get("source_hash") != source_hash():
        return None
    ent = data.get("kernels", {}).get(workload, {}).get(kernel)
    return None if ent is None else ent.get("dram_bytes_per_launch")


# -- oracle timing (cpu_baseline and the reference arm) --------------------------------------

def oracle_slice_runner(shape, seed=0, threads=None):
    import numpy as np  # noqa: F401
    import oracle
    from lisa_synth import make_inputs, to_f64
    inp = make_inputs(shape, seed=seed, B=1, heads=1)
    xq, xk, v = to_f64(inp["xq"]), to_f64(inp["xk"]), to_f64(inp["v"])
    alpha = inp["alpha"].double().numpy()
    kw = {"beta": shape.beta} if shape.weights == "geometric" else \
        {"mlp": tuple(inp[k].double().numpy() for k in ("W1", "b1", "W2", "b2"))}
    threads = host_cores() if threads is None else threads

    def run():
        oracle.forward(xq, xk, v, (shape.H, shape.W), shape.T, alpha=alpha, mode=oracle.LOWRANK,
                       nthreads=threads, **kw)
    return run, threads


def _time_oracle(shape, seconds: float, threads=None):
    run, threads = oracle_slice_runner(shape, threads=threads)
    run()  # warm
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    sample = ("%d repetitions of one (batch, head) slice of the workload (%dx%d grid, n=%d, d=%d, T=%d), "
              "double-precision LOWRANK oracle on %d thread%s, %.1f s" %
              (reps, shape.H, shape.W, shape.n, shape.d, shape.T, threads, "" if threads == 1 else "s", el))
    return reps * shape.n / el, threads, sample


def cpu_baseline(shape, seconds: float):
    """The oracle on all host cores (the line's value) and on one thread,
    the budget split evenly between the two."""
    value, threads, sample = _time_oracle(shape, seconds / 2)
    one, _, one_sample = _time_oracle(shape, seconds / 2, threads=1)
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
            "single_thread": {"value": one, "unit": UNIT, "cores": 1, "sample": one_sample}}


def reference_arm(args, shape):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    run, threads = oracle_slice_runner(shape)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = args.steps * shape.n / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16-quantised inputs widened to double)",
        "config": config_of(shape, reference=True),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "each step: one (batch, head) slice of the workload "
                                   "(n=%d), LOWRANK oracle on %d threads" % (shape.n, threads)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(shape, reference=False, sets=None):
    depth = "T=%d" % shape.T if shape.T else "untruncated walk (T=0)"
    cfg = {"workload": "%s: LiSA forward layer, B=%d heads=%d grid %dx%d (n=%d) d_h=d_v=%d %s %s "
                       "weights%s, alpha %s, eps=1e-6" %
                       (shape.name, shape.B, shape.heads, shape.H, shape.W, shape.n, shape.d, depth,
                        shape.weights, " beta=%.2f" % shape.beta if shape.weights == "geometric" else "",
                        shape.alpha),
           "B": shape.B, "heads": shape.heads, "grid": [shape.H, shape.W], "n": shape.n,
           "d_h": shape.d, "d_v": shape.d, "T": shape.T, "weights": shape.weights}
    if reference:
        cfg["step"] = "one (batch, head) slice of the workload per step"
    else:
        cfg["l2"] = "inputs rotate over %d device sets (%.0f MB) > 3x L2" % (sets[0], sets[1] / 1e6)
    return cfg


# -- the GPU arm ----------------------------------------------------------------------------

STAGE_BYTES_PER_TOKEN = {
    # algorithmic bytes each kernel must move per token*head (bf16, d = 64):
    # what it has to read of Q, K, V and write of O.  Workspace traffic of the
    # split-K partials is per chunk, not per token, and is left out.
    "stats_kv": 2 * 64 * 2,       # SIMT chain: K, V
    "stats_kq": 2 * 64 * 2,       # SIMT chain: Q, K
    "recur": 0,
    "epilogue": 4 * 64 * 2,       # Q, K, V in, O out
    "tc_keysum": 64 * 2,          # tensor-core chain: K
    "tc_stats": 3 * 64 * 2,       # V, Q, K
    "tc_recur": 0,
    "tc_epilogue": 4 * 64 * 2,    # Q, K, V in (halo rows counted once), O out
    "tc_stats_fused": 3 * 64 * 2, # V, Q, K (K once: it stays resident)
}


def stage_bytes(name: str, units: int, d: int, dtype: str) -> int:
    """Algorithmic bytes one launch of kernel `name` moves for `units`
    token*heads at width d: the table is per token*head at bf16, d = 64, so
    it scales with the width and the element size."""
    esz = 2 if dtype == "bf16" else 4
    return STAGE_BYTES_PER_TOKEN.get(name, 0) * units * d * esz // (64 * 2)


def ours_arm(args, shape):
    import torch
    import torch.distributed as dist

    from hop_stochastic_vision_gb300 import build as lisa_build
    from hop_stochastic_vision_gb300 import lisa
    from lisa_synth import make_inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        lisa_build.build()
    if world > 1:
        dist.barrier()
    lib = lisa.load()

    inp = make_inputs(shape, seed=rank)
    B, heads, n, D, T = shape.B, shape.heads, shape.n, shape.d, shape.T
    units = B * heads * n
    set_bytes = 4 * inp["xq"].numel() * inp["xq"].element_size()
    R = max(2, -(-3 * L2_BYTES // set_bytes))
    sets = []
    for r in range(R):
        sets.append({k: inp[k].to(dev).contiguous() for k in ("xq", "xk", "v")})
        sets[-1]["o"] = torch.empty_like(sets[-1]["v"])
    alpha = inp["alpha"].to(dev)
    keep = []
    if shape.weights == "mlp":
        mlp = tuple(inp[k].to(dev) for k in ("W1", "b1", "W2", "b2"))
        wt, keep = lisa.make_weights(T, mlp=mlp)
        wmode = lisa.LISA_W_MLP
    else:
        wt, keep = lisa.make_weights(T, beta=shape.beta)
        wmode = lisa.LISA_W_GEOMETRIC
    dt = lisa.LISA_BF16 if shape.dtype == "bf16" else lisa.LISA_F32
    nbytes = lisa.lisa_workspace_bytes(B, heads, shape.H, shape.W, D, D, T, dt)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    wref = __import__("ctypes").byref(wt)
    call_args = [(s["xq"].data_ptr(), s["xk"].data_ptr(), s["v"].data_ptr(), s["o"].data_ptr(), B, heads,
                  shape.H, shape.W, D, D, T, wref, alpha.data_ptr(), 1e-6, 1, dt, ws.data_ptr(), nbytes, sh)
                 for s in sets]
    fwd = lib.lisa_forward

    def step(i):
        rc = fwd(*call_args[i % R])
        if rc != 0:
            raise RuntimeError("lisa_forward: " + lisa.lisa_status_string(rc))

    nstages = lisa.lisa_num_stages(B, heads, shape.H, shape.W, D, T, dt, wt)
    # warm-up (also loads the kernels before graph capture)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i)
    torch.cuda.synchronize(dev)

    # graphs of G steps cycling through the input sets
    G = min(args.steps, 100)
    reps, rem = divmod(args.steps, G)

    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                step(i)
        return g
    g_main = capture(G) if reps else None
    g_rem = capture(rem) if rem else None
    with torch.cuda.stream(stream):
        if g_main is not None:
            g_main.replay()
    torch.cuda.synchronize(dev)

    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        if hasattr(props, "pci_bus_id"):
            bus = "%08x:%02x:%02x" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                      props.pci_device_id)
    except Exception:
        bus = None
    sampler = ClockSampler(bus)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_max = max_over_ranks(start.elapsed_time(end), world, dev)
    value = weak_throughput(world, units, args.steps, ms_max)

    # per-kernel pass: events between the kernels of each step; the stream is
    # held by a short bounded sleep while the host enqueues, so the kernels
    # run back to back
    Ks = min(args.steps, 100)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nstages + 1)] for _ in range(Ks)]
    stage_fn = lib.lisa_forward_stage
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(2e8))
        for i in range(Ks):
            a = call_args[i % R]
            for stg in range(nstages):
                evs[i][stg].record(stream)
                rc = stage_fn(stg, *a)
                if rc != 0:
                    raise RuntimeError("lisa_forward_stage: " + lisa.lisa_status_string(rc))
            evs[i][nstages].record(stream)
    torch.cuda.synchronize(dev)
    names = [lisa.lisa_stage_name(B, heads, shape.H, shape.W, D, T, dt, wt, s) for s in range(nstages)]
    stage_us = [1e3 * sum(evs[i][s].elapsed_time(evs[i][s + 1]) for i in range(Ks)) / Ks
                for s in range(nstages)]
    dom = max(range(nstages), key=lambda s: stage_us[s])
    peak, peak_src = hbm_peak()
    esz = 2 if shape.dtype == "bf16" else 4
    dom_bytes = stage_bytes(names[dom], units, shape.d, shape.dtype)
    achieved = dom_bytes / (stage_us[dom] * 1e-6) / 1e9
    traffic = ncu_traffic(names[dom], shape.name)
    path_bytes = 4 * shape.d * esz * units
    step_s = ms_max / 1e3 / args.steps

    # end to end through the C ABI with pinned host buffers
    hq, hk, hv = (inp[k].pin_memory() for k in ("xq", "xk", "v"))
    ho = torch.empty_like(hv).pin_memory()
    s0 = sets[0]
    host_args = (hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), s0["xq"].data_ptr(),
                 s0["xk"].data_ptr(), s0["v"].data_ptr(), s0["o"].data_ptr(), B, heads, shape.H, shape.W,
                 D, D, T, wref, alpha.data_ptr(), 1e-6, 1, dt, ws.data_ptr(), nbytes, sh)
    Ke = min(args.steps, 200)
    host_fn = lib.lisa_forward_host
    with torch.cuda.stream(stream):
        for _ in range(3):
            host_fn(*host_args)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke):
            rc = host_fn(*host_args)
            if rc != 0:
                raise RuntimeError("lisa_forward_host: " + lisa.lisa_status_string(rc))
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_value = weak_throughput(world, units, Ke, max_over_ranks(e0.elapsed_time(e1), world, dev))
    io_bytes = inp["xq"].numel() * inp["xq"].element_size()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(shape, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype,
            "data": "synthetic (seeded N(0,1) projections in the layer's shape; no dataset or weights)",
            "config": config_of(shape, sets=(R, R * set_bytes)),
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 3 * io_bytes,
                    "d2h_bytes_per_step": io_bytes, "steps": Ke,
                    "path": "lisa_forward_host (pinned host in, device forward, host out)"},
            "gpu_launches": args.steps * nstages,
            "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_src if peak_src == "measured"
                         else "fallback 6.8 TB/s",
                         "bytes_per_launch": dom_bytes, "launch_us": stage_us[dom],
                         "stage_us": dict(zip(names, stage_us)),
                         "whole_forward": {"bytes_per_step": path_bytes, "step_us": step_s * 1e6,
                                           "achieved_gbs": path_bytes / step_s / 1e9,
                                           "frac": path_bytes / step_s / 1e9 / peak}},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    del keep


# -- the backward pass ------------------------------------------------------------------

BWD_METRIC = "LiSA bwd tokens·heads/s (gradients of Xq, Xk, V, alpha%s); %% of HBM roofline"
# algorithmic bytes per token*head: read Q, K, V, dO, write dQ, dK, dV (d = 64, bf16)
BWD_BYTES_PER_TOKEN = 7 * 64 * 2


def oracle_backward_runner(shape, seed=0):
    import oracle
    from lisa_synth import make_inputs, to_f64
    inp = make_inputs(shape, seed=seed, B=1, heads=1)
    xq, xk, v = to_f64(inp["xq"]), to_f64(inp["xk"]), to_f64(inp["v"])
    import numpy as np
    dO = np.random.default_rng(seed).standard_normal(v.shape)
    alpha = inp["alpha"].double().numpy()

    kw = {"beta": shape.beta} if shape.weights == "geometric" else \
        {"mlp": tuple(inp[k].double().numpy() for k in ("W1", "b1", "W2", "b2"))}

    def run():
        oracle.backward(xq, xk, v, dO, (shape.H, shape.W), shape.T, alpha=alpha, **kw)
    return run


def backward_arm(args, shape):
    """One step = one lisa_backward over the workload's batch (inputs and
    upstream gradient resident in HBM, rotated over sets larger than 3x L2)."""
    import ctypes

    import torch

    from hop_stochastic_vision_gb300 import build as lisa_build
    from hop_stochastic_vision_gb300 import lisa
    from lisa_synth import make_inputs

    rank, world, local = dist_env()
    if rank != 0:
        return
    mlp = shape.weights == "mlp"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lisa_build.build()
    lib = lisa.load()
    inp = make_inputs(shape)
    B, heads, n, D, T = shape.B, shape.heads, shape.n, shape.d, shape.T
    units = B * heads * n
    set_bytes = 7 * inp["xq"].numel() * inp["xq"].element_size()
    R = max(2, -(-3 * L2_BYTES // set_bytes))
    g = torch.Generator("cpu").manual_seed(1)
    sets = []
    for _ in range(R):
        st = {k: inp[k].to(dev).contiguous() for k in ("xq", "xk", "v")}
        st["dO"] = torch.randn(inp["v"].shape, generator=g).to(inp["v"].dtype).to(dev)
        st["dq"], st["dk"], st["dv"] = (torch.empty_like(st["v"]) for _ in range(3))
        sets.append(st)
    alpha = inp["alpha"].to(dev)
    dalpha = torch.empty(heads, dtype=torch.float32, device=dev)
    dt = lisa.LISA_BF16 if shape.dtype == "bf16" else lisa.LISA_F32
    stream = torch.cuda.Stream(dev)
    if mlp:   # adaptive weights: lisa_backward_mlp, with the parameters' gradients
        params = tuple(inp[k].to(dev) for k in ("W1", "b1", "W2", "b2"))
        pgrads = tuple(torch.empty_like(x) for x in params)
        wt, keep = lisa.make_weights(T, mlp=params)
        mg = lisa.lisa_mlp_grads(*(x.data_ptr() for x in pgrads))
        nbytes = lisa.lisa_backward_mlp_workspace_bytes(B, heads, shape.H, shape.W, D, D, T, shape.hidden, dt)
        fn = lib.lisa_backward_mlp
    else:
        wt, keep = lisa.make_weights(T, beta=shape.beta)
        nbytes = lisa.lisa_backward_workspace_bytes(B, heads, shape.H, shape.W, D, D, T, dt)
        fn = lib.lisa_backward
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def args_of(s_):
        head = (s_["xq"].data_ptr(), s_["xk"].data_ptr(), s_["v"].data_ptr(), s_["dO"].data_ptr(), s_["dq"].data_ptr(),
                s_["dk"].data_ptr(), s_["dv"].data_ptr(), dalpha.data_ptr())
        tail = (B, heads, shape.H, shape.W, D, D, T, ctypes.byref(wt), alpha.data_ptr(), 1e-6, 1, dt, ws.data_ptr(),
                nbytes, stream.cuda_stream)
        return head + ((ctypes.byref(mg),) if mlp else ()) + tail
    call = [args_of(s_) for s_ in sets]

    def step(i):
        rc = fn(*call[i % R])
        if rc != 0:
            raise RuntimeError("lisa_backward: " + lisa.lisa_status_string(rc))

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i)
    torch.cuda.synchronize(dev)
    G = min(args.steps, 50)
    reps, rem = divmod(args.steps, G)
    graphs = []
    for count in ([G] if reps else []) + ([rem] if rem else []):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(count):
                step(i)
        graphs.append(gr)
    with torch.cuda.stream(stream):
        graphs[0].replay()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(None)
    sampler.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            graphs[0].replay()
        if rem:
            graphs[-1].replay()
        end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = start.elapsed_time(end)
    value = units * args.steps / (ms / 1e3)
    # kernels per backward: 2 statistics + 7 (recurrence, dUbar, window statistics, reverse
    # recurrence, token pass, per-slice reduction, dK finish with dalpha), plus the bf16 operand
    # image at d = 64; adaptive weights: the MLP pass replaces two, one dU_k pass if T > 1, two
    # for the parameters, and at bf16, d = 64 the MLP operand images
    tc = 1 if (shape.dtype == "bf16" and D == 64) else 0
    nk = 9 + tc + ((1 + (1 if T > 1 else 0) + tc) if mlp else 0)
    peak, peak_src = hbm_peak()
    esz = 2 if shape.dtype == "bf16" else 4
    bytes_step = 7 * D * esz * units
    achieved = bytes_step / (ms / 1e3 / args.steps) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        run = oracle_backward_runner(shape)
        run()
        reps_c, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds:
            run()
            reps_c += 1
        el = time.perf_counter() - t0
        cpu = {"value": reps_c * n / el, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "%d repetitions of one (batch, head) slice (n=%d), double-precision oracle backward, "
                         "%.1f s" % (reps_c, n, el)}
    line = {
        "metric": BWD_METRIC % (" and the MLP parameters" if mlp else ""), "value": value, "unit": UNIT,
        "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": shape.dtype,
        "data": "synthetic (seeded N(0,1) inputs and upstream gradient; no dataset or weights)",
        "config": dict(config_of(shape, sets=(R, R * set_bytes)), direction="backward"),
        "clocks": clocks,
        "gpu_launches": args.steps * nk,
        "roofline": {"bound": "hbm", "kernel": "whole backward (%d kernels)" % nk, "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": peak_src, "bytes_per_step": bytes_step},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    del keep


def main():
    args = parse_args()
    from lisa_synth import SHAPES
    shape = SHAPES[args.workload]
    if args.impl == "reference":
        reference_arm(args, shape)
    elif args.direction == "backward":
        backward_arm(args, shape)
    else:
        ours_arm(args, shape)


if __name__ == "__main__":
    main()
