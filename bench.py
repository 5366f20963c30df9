#!/usr/bin/env python
"""Benchmark of the dropless MoE expert layer on GB300: one step = route +
forward + backward (down to d(logits) of the router) of one layer over one
batch of synthetic tokens.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 235b]
  python bench.py --impl reference ...      # the float64 CPU oracle arm

Metric: per-layer training-step throughput in algorithmic TFLOP/s
(18 * T * top_k * H * I per step: 6 forward + 12 backward), plus per-pass
forward / backward ms.  Prints ONE JSON line on rank 0.

Default workload: the Qwen3-235B-A22B layer shape (T=16384, H=4096, E=128,
top_k=8, I=1536, bf16), the shape at which the tensor-roofline target is
stated.  Inputs are seeded synthetic draws (``workloads``); the per-step
working set (4.8 GB of weights, 0.1 GB of tokens) is far larger than the
129 MB L2, so no L2 flush is needed between steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import CONFIGS, make_inputs  # noqa: E402

# Kernels of this library per timed step (route 3: router, scan, scatter;
# router backward 1).  bf16: forward gather, 2 GEMMs, combine; backward
# gather of dY, 2 co-scheduled GEMM launches, combine, d(gate) reduction.
# mxfp8: forward gather+quantise, W13 / W2 dual quantise, 2 GEMMs (the
# gate/up epilogue writes A's encodings), combine; backward dY
# gather+quantise, 2 GEMM launches (the dSwiGLU epilogue writes dh13's
# encodings), combine, d(gate) reduction.  fp8_bwd: the bf16-precision
# forward (gate after W2), and the mxfp8 backward plus 4 quantise passes of
# W2, A, W13, X_perm.
LAUNCHES_PER_STEP = {"bf16": 13, "mxfp8": 15, "fp8_bwd": 17}
CPU_SAMPLE_EXPERTS = 16   # cpu_baseline: all assignments of 16 experts
REF_SAMPLE_EXPERTS = 1    # reference arm: one expert per step (rotating)


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="235b", choices=[k for k in CONFIGS if k != "tiny"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the shorter runs of the other workloads and modes")
    # smaller variants of the workload, for profiler captures
    p.add_argument("--tokens", type=int, default=None, help="override T")
    p.add_argument("--experts", type=int, default=None, help="override E")
    p.add_argument("--mode", default="bf16", choices=["bf16", "mxfp8", "fp8_bwd"],
                   help="GEMM precision (bf16; MXFP8 forward+backward; bf16 forward + MXFP8 backward)")
    p.add_argument("--clocks-dir", default=tempfile.gettempdir(),
                   help="where the raw nvidia-smi clock samples of the timed region are kept")
    p.add_argument("--debug-flags", type=int, default=0,
                   help="library debug flags (diagnosis runs only, e.g. 4 = split backward)")
    return p.parse_args()


def _config(args):
    import dataclasses
    cfg = CONFIGS[args.workload]
    kw = {}
    if args.tokens:
        kw["T"] = args.tokens
    if args.experts:
        kw["E"] = args.experts
    if kw:
        cfg = dataclasses.replace(cfg, name=cfg.name + "-variant", **kw)
    return cfg


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _host_cores():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = [i["num_threads"] for i in info if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def _workload_desc(cfg):
    return (f"{cfg.name}: MoE expert layer T={cfg.T} H={cfg.H} E={cfg.E} top_k={cfg.k} "
            f"I={cfg.I}" + (" (Zipf-skewed routing, 8 empty experts)" if cfg.skew else ""))


def _oracle_sample(cfg, inp, experts):
    """The float64 oracle on a bounded sample of the workload: routing of the
    whole batch, then forward + backward of every assignment of the given
    experts (each expert's assignments form a k=1 sub-batch with their own
    gates and the expert's weights).  Returns (seconds, algorithmic flops)."""
    from oracle import moe_oracle as O
    from workloads import bf16_bits_to_f32

    def f32(a):
        return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a

    t0 = time.perf_counter()
    idx, gate = O.route(inp["logits"], cfg.k)
    n_total = 0
    for e in experts:
        t, j = np.nonzero(idx == e)
        if t.size == 0:
            continue
        n_total += t.size
        sub_idx = np.zeros((t.size, 1), np.int32)
        sub_gate = gate[t, j][:, None]
        X = f32(inp["X"][t])
        dY = f32(inp["dY"][t])
        W13 = f32(inp["W13"][e:e + 1])
        W2 = f32(inp["W2"][e:e + 1])
        O.forward(X, W13, W2, sub_idx, sub_gate)
        O.backward(X, W13, W2, sub_idx, sub_gate, dY)
    dt = time.perf_counter() - t0
    return dt, 18.0 * n_total * cfg.H * cfg.I


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, directory):
        self.index = index
        self.proc = None
        self.path = os.path.join(directory, f"clocks_bench_{os.getpid()}.csv")
        self.t0 = self.t1 = None   # host wall clock at the start / end of the timed region

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
                except ValueError:
                    continue
        # samples taken inside the timed region (all of them if none fell inside)
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        sm = [r[1] for r in use]
        mx = [r[2] for r in use]
        power = [r[3] for r in use]
        reasons = set()
        for r in use:
            for n, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_timed_region": len(inside),
                "power_w_median": statistics.median(power) if power else None}


def _traffic(kernel, src_files):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in src_files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    with open(path) as f:
        for line in f:
            m = re.match(r"\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*([0-9.eE+]+)\s*\|", line)
            if m and m.group(1) == kernel and m.group(2) == digest:
                return float(m.group(3))
    return None


def max_over_ranks(values, world, device):
    """Element-wise maximum of per-rank timings (the slowest replica sets the
    whole job's time); the identity for a single process."""
    import torch
    if world <= 1:
        return list(values)
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(flops_per_step, world, ms_step):
    """Whole-job TFLOP/s: every replica runs one step of flops_per_step in the
    (max over ranks) step time."""
    return world * flops_per_step / (ms_step * 1e-3) / 1e12


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = _config(args)
    inp = make_inputs(cfg)
    times, flops = [], []
    for i in range(args.warmup + args.steps):
        experts = [(i * REF_SAMPLE_EXPERTS + q) % cfg.E for q in range(REF_SAMPLE_EXPERTS)]
        dt, fl = _oracle_sample(cfg, inp, experts)
        if i >= args.warmup:
            times.append(dt)
            flops.append(fl)
    ms = 1e3 * statistics.mean(times)
    value = sum(flops) / sum(times) / 1e12
    cores = _host_cores()
    sample = (f"float64 oracle: routing of the whole batch, then forward+backward of all "
              f"assignments of {REF_SAMPLE_EXPERTS} expert(s) per step (rotating experts)")
    print(json.dumps({
        "impl": "reference", "metric": "moe_layer_step_tflops", "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_desc(cfg), "sample_experts": REF_SAMPLE_EXPERTS},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def _per_config(cfg, mode, d, steps, warmup, peaks):
    """fwd / bwd / step ms of one workload and mode on already-resident inputs
    ``d`` (device tensors), with the grouped-GEMM launch times from the
    library's event hooks: the bracket from the first to the last GEMM launch
    of a call (in the MXFP8 modes it also holds the quantise passes between
    the launches) and the sum of the GEMM launches alone."""
    import torch

    import mixture_experts_layer_18_gb300 as M
    from mixture_experts_layer_18_gb300.layer import MoELayer
    L = MoELayer(cfg.T, cfg.H, cfg.E, cfg.I, cfg.k, mode=mode)
    io = L.empty_io()
    dl = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")

    def fwd():
        L.route(d["logits"])
        L.forward(d["X"], d["W13"], d["W2"], io["Y"])

    def bwd():
        L.backward(d["dY"], d["W13"], d["W2"], io["dX"], io["dW13"], io["dW2"], io["dgate"])
        L.route_backward(io["dgate"], dl)

    for _ in range(warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    pf = [(ev(), ev()) for _ in range(steps)]
    pb = [(ev(), ev()) for _ in range(steps)]
    lf = [[(ev(), ev()) for _ in range(2)] for _ in range(steps)]   # per GEMM launch
    lb = [[(ev(), ev()) for _ in range(2)] for _ in range(steps)]
    for a, b in pf + pb + [x for row in lf + lb for x in row]:
        a.record()             # materialise the event handles (torch creates them lazily)
        b.record()
    t0, t1 = ev(), ev()
    torch.cuda.synchronize()
    t0.record()
    for i in range(steps):
        M.moe_set_gemm_events(M.MOE_WS_FORWARD, pf[i][0].cuda_event, pf[i][1].cuda_event)
        M.moe_set_gemm_launch_events(M.MOE_WS_FORWARD, [a.cuda_event for a, _ in lf[i]],
                                     [b.cuda_event for _, b in lf[i]])
        fwd()
        M.moe_set_gemm_events(M.MOE_WS_BACKWARD, pb[i][0].cuda_event, pb[i][1].cuda_event)
        M.moe_set_gemm_launch_events(M.MOE_WS_BACKWARD, [a.cuda_event for a, _ in lb[i]],
                                     [b.cuda_event for _, b in lb[i]])
        bwd()
    t1.record()
    torch.cuda.synchronize()
    if L.device_status() != 0:
        raise RuntimeError(f"{cfg.name} {mode}: device status {L.device_status()}")
    step = t0.elapsed_time(t1) / steps

    def timed(fn):
        a, b = ev(), ev()
        torch.cuda.synchronize()
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    fwd_ms, bwd_ms = timed(fwd), timed(bwd)
    gf = statistics.mean(a.elapsed_time(b) for a, b in pf)
    gb = statistics.mean(a.elapsed_time(b) for a, b in pb)
    gf1 = statistics.mean(sum(a.elapsed_time(b) for a, b in row) for row in lf)
    gb1 = statistics.mean(sum(a.elapsed_time(b) for a, b in row) for row in lb)
    out = {"workload": _workload_desc(cfg), "mode": mode, "steps": steps, "warmup": warmup,
           "ms_per_step": step, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
           "tflops": (cfg.fwd_flops() + cfg.bwd_flops()) / (step * 1e-3) / 1e12,
           "fwd_tflops": cfg.fwd_flops() / (fwd_ms * 1e-3) / 1e12,
           "bwd_tflops": cfg.bwd_flops() / (bwd_ms * 1e-3) / 1e12}
    if mode != "f32":
        peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
        pk_f = peak * (2 if mode == "mxfp8" else 1)
        pk_b = peak * (2 if mode in ("mxfp8", "fp8_bwd") else 1)
        out["gemm"] = {
            "fwd_launch_ms": gf, "bwd_launch_ms": gb,
            "fwd_frac": cfg.fwd_flops() / (gf * 1e-3) / 1e12 / pk_f,
            "bwd_frac": cfg.bwd_flops() / (gb * 1e-3) / 1e12 / pk_b,
            "fwd_gemm_only_ms": gf1, "bwd_gemm_only_ms": gb1,
            "fwd_gemm_only_frac": cfg.fwd_flops() / (gf1 * 1e-3) / 1e12 / pk_f,
            "bwd_gemm_only_frac": cfg.bwd_flops() / (gb1 * 1e-3) / 1e12 / pk_b,
            "peak_tflops_fwd": pk_f, "peak_tflops_bwd": pk_b,
            "note": ("bf16 sustained measured peak" + (" x 2 (nominal fp8/bf16 ratio) where MXFP8"
                     if mode != "bf16" else "")
                     + ("; the bracket includes the quantise passes between the GEMM launches, "
                        "gemm_only sums the two GEMM launches of each call"
                        if mode != "bf16" else ""))}
    del L, io
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import mixture_experts_layer_18_gb300 as M
    from mixture_experts_layer_18_gb300.layer import MoELayer

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group(backend="nccl")
    torch.cuda.set_device(local)
    cfg = _config(args)
    inp = make_inputs(cfg, seed=rank)

    def dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    d = {k: dev(v) for k, v in inp.items()}
    M.moe_set_debug(args.debug_flags, 0)
    L = MoELayer(cfg.T, cfg.H, cfg.E, cfg.I, cfg.k, mode=args.mode)
    io = L.empty_io()

    def fwd():
        L.route(d["logits"])
        L.forward(d["X"], d["W13"], d["W2"], io["Y"])

    dlogits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")

    def bwd():
        L.backward(d["dY"], d["W13"], d["W2"], io["dX"], io["dW13"], io["dW2"], io["dgate"])
        L.route_backward(io["dgate"], dlogits)

    def step():
        fwd()
        bwd()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if L.device_status() != 0:
        raise RuntimeError(f"device status {L.device_status()} after warm-up")

    def barrier():
        if world > 1:
            dist.barrier()

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        return e

    # ---- timed steps (kernel-level events around the backward GEMM launch)
    K = args.steps
    pairs_b = [(ev(), ev()) for _ in range(K)]
    pairs_f = [(ev(), ev()) for _ in range(K)]
    lb = [[(ev(), ev()) for _ in range(2)] for _ in range(K)]   # per GEMM launch
    lf = [[(ev(), ev()) for _ in range(2)] for _ in range(K)]
    for a, b in pairs_b + pairs_f + [x for row in lb + lf for x in row]:   # materialise handles
        a.record()
        b.record()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, args.clocks_dir)
    clocks.start()
    time.sleep(0.4)
    barrier()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    clocks.t0 = time.time()
    t0.record()
    for i in range(K):
        M.moe_set_gemm_events(M.MOE_WS_FORWARD, pairs_f[i][0].cuda_event, pairs_f[i][1].cuda_event)
        M.moe_set_gemm_launch_events(M.MOE_WS_FORWARD, [a.cuda_event for a, _ in lf[i]],
                                     [b.cuda_event for _, b in lf[i]])
        fwd()
        M.moe_set_gemm_events(M.MOE_WS_BACKWARD, pairs_b[i][0].cuda_event, pairs_b[i][1].cuda_event)
        M.moe_set_gemm_launch_events(M.MOE_WS_BACKWARD, [a.cuda_event for a, _ in lb[i]],
                                     [b.cuda_event for _, b in lb[i]])
        bwd()
    t1.record()
    torch.cuda.synchronize()
    clocks.t1 = time.time()
    barrier()
    clk = clocks.stop()
    ms_step = t0.elapsed_time(t1) / K
    # the GEMM launches alone (summed per call), and the bracket from the
    # first to the last of them (MXFP8: with the quantise passes in between)
    gemm_b = statistics.mean(sum(a.elapsed_time(b) for a, b in row) for row in lb)
    gemm_f = statistics.mean(sum(a.elapsed_time(b) for a, b in row) for row in lf)
    bracket_b = statistics.mean(a.elapsed_time(b) for a, b in pairs_b)
    bracket_f = statistics.mean(a.elapsed_time(b) for a, b in pairs_f)
    if L.device_status() != 0:
        raise RuntimeError(f"device status {L.device_status()} after timed steps")

    # ---- per-pass timings
    def timed(fn, n):
        a, b = ev(), ev()
        torch.cuda.synchronize()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    fwd_ms = timed(fwd, K)
    bwd_ms = timed(bwd, K)

    # ---- the pages' full-layer measure: 2 x forward + backward with full
    # activation checkpointing (a forward that keeps nothing, then the
    # recomputing forward and the backward), captured as one CUDA graph
    def full_layer():
        L.route(d["logits"])
        L.forward(d["X"], d["W13"], d["W2"], io["Y"], save=False)
        L.forward(d["X"], d["W13"], d["W2"], io["Y"], save=True)
        bwd()

    full_layer()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        full_layer()
    graph.replay()
    torch.cuda.synchronize()
    full_ms = timed(graph.replay, K)
    if L.device_status() != 0:
        raise RuntimeError(f"device status {L.device_status()} after graph replays")

    # ---- end to end: pinned host inputs in, results out, every step.  The
    # copies run on a second stream into and out of double-buffered device
    # sets, so one step's transfers overlap its neighbours' compute (a
    # prefetching input pipeline); every step still moves its own inputs in
    # and its own results out inside the timed region.
    h_in = {k: d[k].cpu().pin_memory() for k in ("logits", "X", "dY")}
    h_out = {k: torch.empty(io[k].shape, dtype=io[k].dtype, pin_memory=True)
             for k in ("Y", "dX", "dgate")}
    din = [{k: d[k] for k in h_in}, {k: torch.empty_like(d[k]) for k in h_in}]
    dout = [{k: io[k] for k in h_out}, {k: torch.empty_like(io[k]) for k in h_out}]
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()

    def e2e_run(n):
        """n steps; returns ms per step from the first copy in to the last copy out."""
        in_ready = [torch.cuda.Event(), torch.cuda.Event()]
        in_free = [torch.cuda.Event(), torch.cuda.Event()]
        out_ready = [torch.cuda.Event(), torch.cuda.Event()]
        out_free = [torch.cuda.Event(), torch.cuda.Event()]

        def h2d(b):
            with torch.cuda.stream(copy):
                copy.wait_event(in_free[b])          # the step that last read set b is done
                for k, h in h_in.items():
                    din[b][k].copy_(h, non_blocking=True)
                in_ready[b].record(copy)

        def d2h(b):
            with torch.cuda.stream(copy):
                copy.wait_event(out_ready[b])
                for k, h in h_out.items():
                    h.copy_(dout[b][k], non_blocking=True)
                out_free[b].record(copy)

        torch.cuda.synchronize()
        start, end = ev(), ev()
        start.record(comp)
        copy.wait_stream(comp)
        h2d(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                h2d(b ^ 1)
            comp.wait_event(in_ready[b])
            comp.wait_event(out_free[b])             # step i-2's results are out
            x, o = din[b], dout[b]
            L.route(x["logits"])
            L.forward(x["X"], d["W13"], d["W2"], o["Y"])
            L.backward(x["dY"], d["W13"], d["W2"], o["dX"], io["dW13"], io["dW2"], o["dgate"])
            L.route_backward(o["dgate"], dlogits)
            in_free[b].record(comp)
            out_ready[b].record(comp)
            d2h(b)
        comp.wait_stream(copy)
        end.record(comp)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / n

    e2e_run(2)
    e2e_ms = e2e_run(K)
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())

    # ---- max over ranks
    ms_step, e2e_ms, fwd_ms, bwd_ms, gemm_b, gemm_f, full_ms, bracket_b, bracket_f = max_over_ranks(
        [ms_step, e2e_ms, fwd_ms, bwd_ms, gemm_b, gemm_f, full_ms, bracket_b, bracket_f], world,
        "cuda")

    flops_step = cfg.fwd_flops() + cfg.bwd_flops()
    value = job_throughput(flops_step, world, ms_step)
    peaks, src = _peaks()
    # The GEMM launches are timed inside the step loop, which runs
    # power-capped (SM cycles / globaltimer over the bf16 GEMM launches:
    # ~1.57 GHz against 2.07 GHz max), so the denominator is the sustained
    # measured peak; the burst fraction is reported beside it.
    peak_burst = float(peaks["bf16_tflops"])
    peak = float(peaks.get("bf16_tflops_sustained", peak_burst))
    # MXFP8 contractions: measured bf16 peak x the nominal fp8 / bf16 ratio (2)
    mx_b = args.mode in ("mxfp8", "fp8_bwd")
    mx_f = args.mode == "mxfp8"
    peak_b = peak * (2 if mx_b else 1)
    peak_f = peak * (2 if mx_f else 1)
    peak_note = (f"{src} bf16_tflops_sustained" if "bf16_tflops_sustained" in peaks
                 else f"{src} bf16_tflops (burst)") + (" x 2 (nominal fp8/bf16 ratio)" if mx_b else "")
    ach_b = cfg.bwd_flops() / (gemm_b * 1e-3) / 1e12
    ach_f = cfg.fwd_flops() / (gemm_f * 1e-3) / 1e12
    traffic = None if mx_b else _traffic(
        "moe_gemm_kernel<bf16,256,2>/backward",
        ["mixture_experts_layer_18_gb300/csrc/gemm.cu",
         "mixture_experts_layer_18_gb300/csrc/common.cuh"])
    kname = ("moe_gemm_kernel<bf16,256,2>: the backward's two co-scheduled GEMM launches "
             "({D, dW2}, {dX, dW13})" if not mx_b
             else "moe_gemm_kernel<e4m3,192,2>: the MXFP8 backward's two co-scheduled GEMM "
             "launches ({D, dW2}, {dX, dW13})")
    out = {
        "metric": "moe_layer_step_tflops", "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.mode,
        "data": "synthetic",
        "config": {"workload": _workload_desc(cfg), "T": cfg.T, "H": cfg.H, "E": cfg.E,
                   "top_k": cfg.k, "I": cfg.I, "mode": args.mode,
                   "flops_per_step": flops_step, "parallelism": "replicas",
                   "l2": "inputs larger than L2 (no flush)"},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "full_layer": {"ms": full_ms, "what": "2 x forward + backward (full activation "
                       "checkpointing), replayed as one CUDA graph",
                       "tflops": world * (2 * cfg.fwd_flops() + cfg.bwd_flops()) /
                       (full_ms * 1e-3) / 1e12},
        "fwd_tflops": cfg.fwd_flops() / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": cfg.bwd_flops() / (bwd_ms * 1e-3) / 1e12,
        "roofline": {"kernel": kname,
                     "bound": "tensor", "achieved": ach_b, "peak": peak_b, "unit": "TFLOP/s",
                     "frac": ach_b / peak_b, "traffic": traffic,
                     "peak_source": peak_note, "launch_ms": gemm_b,
                     "launch_ms_how": "sum of the two launches' CUDA-event times per step",
                     "bracket_ms": bracket_b,
                     "frac_of_burst_peak": ach_b / (peak_burst * peak_b / peak)},
        "roofline_forward_gemms": {"achieved": ach_f, "peak": peak_f, "frac": ach_f / peak_f,
                                   "unit": "TFLOP/s", "launch_ms": gemm_f,
                                   "bracket_ms": bracket_f,
                                   "frac_of_burst_peak": ach_f / (peak_burst * peak_f / peak)},
        "e2e": {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": "pinned host inputs (logits, X, dY) in and results (Y, dX, d(gate)) out "
                       "every step on a second stream, double-buffered device sets, first copy in "
                       "to last copy out"},
        "gpu_launches": LAUNCHES_PER_STEP[args.mode] * K,
        "clocks": clk,
    }
    # ---- the other workloads of the metric (shorter runs; the headline value
    # above stays the 235B bf16 step)
    if world == 1 and not args.no_per_config and not (args.tokens or args.experts):
        pc = []
        if args.workload == "235b" and args.mode == "bf16":
            for m in ("mxfp8", "fp8_bwd"):
                pc.append(_per_config(CONFIGS["235b_mxfp8"], m, d, 10, 3, peaks))
        del d
        torch.cuda.empty_cache()
        c30 = CONFIGS["30b"]
        i30 = make_inputs(c30)
        d30 = {k: dev(v) for k, v in i30.items()}
        pc.append(_per_config(c30, "bf16", d30, 10, 3, peaks))
        d30["logits"] = dev(make_inputs(CONFIGS["30b_zipf"], parts=("logits",))["logits"])
        pc.append(_per_config(CONFIGS["30b_zipf"], "bf16", d30, 10, 3, peaks))
        del d30
        ct = CONFIGS["tiny"]
        dt_ = {k: dev(v) for k, v in make_inputs(ct).items()}
        pc.append(_per_config(ct, "f32", dt_, 10, 3, peaks))
        out["per_config"] = pc

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        experts = list(range(CPU_SAMPLE_EXPERTS))
        dt, fl = _oracle_sample(cfg, inp, experts)
        out["cpu_baseline"] = {
            "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": _host_cores(), "kind": "oracle",
            "sample": (f"float64 oracle: routing of the whole batch, then forward+backward of all "
                       f"assignments of experts 0..{CPU_SAMPLE_EXPERTS - 1} "
                       f"({fl / (18.0 * cfg.H * cfg.I):.0f} assignments), {dt:.1f} s")}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
