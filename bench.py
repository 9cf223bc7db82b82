#!/usr/bin/env python
"""KDA RecoverSSM verify + commit throughput on GB300.

One step = every layer's speculative verify (one launch per layer) followed by
one commit launch that folds the accepted tokens of all layers, on seeded
synthetic inputs already resident in HBM.  Default workload: B=256 requests,
H=32 heads, K=V=128, window Q=4, 24 KDA layers, 512-slot fp32 state pools
(dim-first conv state, bf16 conv weight).

Prints one JSON line (rank 0).  Metric: verified tokens/s (sum over live
requests of min(query_len, Q) per step, all ranks) and the achieved HBM
bandwidth of the algorithmic bytes.  ``--impl reference`` times the CPU
oracle instead (bounded sample, host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify+commit tokens/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- workload accounting

def step_accounting(cfg, meta) -> dict:
    """Tokens and algorithmic HBM bytes of one step (every layer's verify plus
    the commit), from the drawn arrays: state read once per live (request,
    head) by the verify, read and written once by the commit when it folds
    at least one token; activations, outputs, records, conv taps and gate
    parameters at their stored sizes."""
    H, K, V, Q, W, L = cfg.H, cfg.K, cfg.V, cfg.Q, cfg.W, cfg.L
    qsl = meta.query_start_loc.astype(np.int64)
    lens = np.clip(np.diff(qsl), 0, Q)
    live = meta.state_indices > 0
    acc = np.minimum(np.maximum(meta.num_accepted.astype(np.int64), 0), lens)
    w_bytes = 4 if cfg.conv_weight_fp32 else 2
    params = 3 * H * K * W * w_bytes + 4 * H + 4 * H * K
    item_fixed = 4 * V * K + (W - 1) * 3 * K * 2 + (W - 2) * 3 * K * 2
    item_per_token = (3 * K * 2 + K * 2 + 2 + V * 2) + (4 * V + 4 * K) + 3 * K * 2
    verify_layer = (H * (live.sum() * item_fixed + item_per_token * lens[live].sum())
                    + lens[~live].sum() * H * V * 2 + params)
    m = acc[live & (acc > 0)]
    commit = L * H * (m.size * 2 * 4 * V * K + (4 * V + 4 * K) * m.sum())
    # the deferred schedule folds inside the verify, which reads the state once
    # for both: one state read fewer per folded (layer, request, head)
    deferred = L * verify_layer + commit - L * H * m.size * 4 * V * K
    return dict(tokens=int(lens[live].sum()), verify_layer_bytes=int(verify_layer),
                verify_bytes=int(L * verify_layer), commit_bytes=int(commit),
                step_bytes=int(L * verify_layer + commit), commit_items=int(L * H * m.size),
                deferred_step_bytes=int(deferred))


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kind: str) -> str:
    csrc = os.path.join(ROOT, "linear_attention_ssm_kda_gb300", "csrc")
    files = {"verify": ["kda_verify.cu", "kda_device.cuh", "kda_params.h"],
             "commit": ["kda_commit.cu", "kda_device.cuh", "kda_params.h"]}[kind]
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary
    (``profiles/traffic.txt``: kernel, source hash, workload, bytes per launch),
    if it was taken on the current source of the kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split("#", 1)[0].split()
                if len(parts) >= 4 and parts[0] == kind:
                    if parts[1] == kernel_source_hash(kind) and parts[2] == workload:
                        return int(parts[3])
    except (OSError, ValueError):
        return None
    return None


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device):
        self.proc = None
        self.target = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.target = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.target = vis.split(",")[0] if vis else "0"

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", self.target],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------- distributed plumbing

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world == 1:
        return 0, 0, 1
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank runs an independent shard of requests (its own seeded draw)."""
    return base_seed + 1000 * rank


def workload_config(c, acct) -> dict:
    """The ``config`` object of the JSON line (both arms)."""
    return {
        "workload": (f"{c.name}: verify then commit, B={c.B} requests, H={c.H} heads, K=V={c.K}, "
                     f"window Q={c.Q}, conv width {c.W}, {c.L} layers, {c.slots}-slot fp32 state pools, "
                     f"{'dim' if c.conv_dim_first else 'seq'}-first conv state, "
                     f"{'fp32' if c.conv_weight_fp32 else 'bf16'} conv weight, "
                     f"{'lower_bound' if c.lower_bound is not None else 'softplus'} gate"),
        "tokens_per_step": acct["tokens"],
        "algorithmic_bytes_per_step": acct["step_bytes"],
        "l2": "inputs larger than L2 (each step streams every layer's live state, ~GBs)",
        "activations": "bf16", "state": "fp32",
    }


# --------------------------------------------------------------------------- oracle timing (CPU)

def time_oracle(cfg_name: str, steps: int, warmup: int, threads: int | None = None, layers: int | None = None):
    """The CPU oracle as it stands, timed on full steps of the workload: per
    step, the full request batch's verify and commit, L times (one layer's
    inputs, re-used for every layer: the oracle's work does not depend on the
    values, and L distinct C2 layers would need about 24 GiB of host memory).
    Returns (tokens/s, seconds per step, sample description, threads, accounting)."""
    tests = os.path.join(ROOT, "tests")
    if tests not in sys.path:
        sys.path.insert(0, tests)
    from oracle_io import host_layer, run_commit, run_verify
    from workloads import CONFIGS, make_problem

    cfg = CONFIGS[cfg_name]
    if layers:
        cfg = cfg.replace(L=layers)
    threads = threads or len(os.sched_getaffinity(0))
    prob = make_problem(cfg, "cpu", L=1)
    acct = step_accounting(cfg, prob.meta)
    hl = host_layer(prob, 0)

    def one_step():
        # a decode step: every layer's verify rolls the conv state and writes
        # records in place, its commit advances the state in place
        for _ in range(cfg.L):
            run_verify(prob, hl, num_threads=threads)
            run_commit(prob, hl, num_threads=threads)

    for _ in range(warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    per_step = (time.perf_counter() - t0) / steps
    sample = (f"{cfg_name} full steps: the request batch (B={cfg.B}, H={cfg.H}), verify + commit of {cfg.L} "
              f"layers per step (one layer's inputs re-used), {steps} timed steps after {warmup}")
    return acct["tokens"] / per_step, per_step, sample, threads, acct


# --------------------------------------------------------------------------- GPU arm

def run_e2e(args, prob, ctx, stream, dev, world):
    """End to end through the public API with host buffers: every step copies
    its inputs from pinned host memory, runs, and reads its outputs back
    (``workloads.drive.HostPipeline``: each layer's copies overlap the other
    layers' kernels)."""
    from workloads.drive import HostPipeline, pinned_meta

    host_fused = torch.empty(prob.fused.shape, dtype=prob.fused.dtype, pin_memory=True)
    host_fused.copy_(prob.fused)
    host_meta = pinned_meta(prob.meta)
    host_out = torch.empty(prob.out.shape, dtype=prob.out.dtype, pin_memory=True)
    h2d = host_fused.numel() * 2 + sum(t.numel() * 4 for t in host_meta.values())
    d2h = host_out.numel() * 2
    pipe = HostPipeline(prob, ctx, stream)

    for _ in range(max(1, args.warmup // 2)):
        pipe.step(host_fused, host_meta, host_out)
    pipe.drain()
    torch.cuda.synchronize(dev)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, args.steps // 2)
    barrier(world)
    e_start.record(stream)
    for _ in range(e2e_steps):
        pipe.step(host_fused, host_meta, host_out)
    pipe.drain()
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end)
    return e2e_ms, e2e_steps, h2d, d2h


def run_deferred(args, prob, dm, stream, dev, world):
    """The deferred schedule of the same workload (``kda_verify_fold``): each
    layer's verify first folds the previous step's accepted records into the
    checkpoint, so a step is L launches and no commit launch.  Every step uses
    the same request metadata, so each folds what the step before accepted."""
    from workloads.drive import verify_layer

    L = prob.cfg.L

    def step():
        for l in range(L):
            verify_layer(prob, l, dm, stream=stream, fold=dm)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    d_start = torch.cuda.Event(enable_timing=True)
    d_end = torch.cuda.Event(enable_timing=True)
    steps = max(3, args.steps // 2)
    barrier(world)
    d_start.record(stream)
    for _ in range(steps):
        step()
    d_end.record(stream)
    torch.cuda.synchronize(dev)
    return d_start.elapsed_time(d_end), steps


def verify_tail(prob, dm, stream, dev):
    """The verify kernel's schedule on one layer of the workload, after the
    timed region: kda_verify_debug's timer hook gives each CTA's start and
    finish on the GPU's global timer; reported is the kernel's span and the
    spread between the first and the last CTA to finish."""
    import linear_attention_ssm_kda_gb300 as kda
    from workloads.drive import verify_layer

    cfg = prob.cfg
    items = cfg.B * cfg.H
    grid = min(items, torch.cuda.get_device_properties(dev).multi_processor_count)
    times = torch.zeros(2 * items, dtype=torch.int64, device=dev)
    ws = kda.new_workspace(dev)
    spans, spreads = [], []
    for _ in range(5):
        verify_layer(prob, 0, dm, workspace=ws, stream=stream, debug=(-1, 1_000_000_000, times))
        torch.cuda.synchronize(dev)
        t = times[: 2 * grid].view(grid, 2).cpu()
        spans.append(float(t[:, 1].max() - t[:, 0].min()) / 1e3)
        spreads.append(float(t[:, 1].max() - t[:, 1].min()) / 1e3)
    span, spread = statistics.median(spans), statistics.median(spreads)
    return {"ctas": grid, "kernel_span_us": span, "finish_spread_us": spread,
            "finish_spread_frac": spread / span if span > 0 else None,
            "how": "median of 5 launches of one layer with per-CTA global-timer stamps (kda_verify_debug)"}


def run_long_window(args, dev):
    """The long-window workload (C3: B=512, H=32, Q=8, one layer) on both
    schedules, one GPU: verify then commit (the tensor-core verify, the
    default at Q = 8, and the commit launch) against the deferred schedule
    (kda_verify_fold on the CUDA cores, no commit launch).  Every step uses
    the same request metadata, so each step's fold folds what the step before
    accepted."""
    from workloads import CONFIGS, make_problem
    from workloads.drive import commit_all, commit_context, device_meta, verify_layer

    cfg = CONFIGS["C3"]
    prob = make_problem(cfg, dev)
    acct = step_accounting(cfg, prob.meta)
    dm = device_meta(prob.meta, dev)
    ctx = commit_context(prob)
    stream = torch.cuda.current_stream(dev)

    def plain():
        for l in range(cfg.L):
            verify_layer(prob, l, dm, stream=stream)
        commit_all(ctx, dm, stream=stream)

    def deferred():
        for l in range(cfg.L):
            verify_layer(prob, l, dm, stream=stream, fold=dm)

    out = {}
    steps = max(5, args.steps // 2)
    for name, fn in (("verify_then_commit", plain), ("deferred", deferred)):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"ms_per_step": ms, "tokens_per_s": acct["tokens"] / (ms / 1e3)}
    out["workload"] = "C3: B=512, H=32, K=V=128, Q=8, 1 layer, lower-bound gate"
    out["steps"] = steps
    return out


def run_gpu(args, rank, local, world):
    import linear_attention_ssm_kda_gb300 as kda
    from linear_attention_ssm_kda_gb300 import _build
    from workloads import CONFIGS, make_problem
    from workloads.drive import commit_all, commit_context, device_meta, verify_layer

    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    barrier(world)
    kda.load_library()
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    cfg = CONFIGS[args.config]
    if args.layers:
        cfg = cfg.replace(L=args.layers)
    prob = make_problem(cfg, dev, seed=shard_seed(cfg.seed, rank))
    meta = prob.meta
    acct = step_accounting(cfg, meta)
    dm = device_meta(meta, dev)
    ctx = commit_context(prob)
    stream = torch.cuda.current_stream(dev)
    L = cfg.L

    def step(evs=None):
        for l in range(L):
            if evs is not None:
                evs[l].record(stream)
            verify_layer(prob, l, dm, stream=stream)
        if evs is not None:
            evs[L].record(stream)
        commit_all(ctx, dm, stream=stream)
        if evs is not None:
            evs[L + 1].record(stream)

    ws = kda.new_workspace(dev)
    for l in range(L):  # one checked pass: the device reports no error on this workload
        verify_layer(prob, l, dm, workspace=ws, stream=stream)
    commit_all(ctx, dm, workspace=ws, stream=stream)
    flags = kda.read_device_error(ws, stream)
    if flags:
        raise RuntimeError(f"device error bits 0x{flags:x} on the benchmark workload")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # per-launch events over the timed region
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(L + 2)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)  # let the sampler attach before the region starts
    t_start.record(stream)
    for k in range(args.steps):
        step(events[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    verify_ms = [events[k][l].elapsed_time(events[k][l + 1]) for k in range(args.steps) for l in range(L)]
    commit_ms = [events[k][L].elapsed_time(events[k][L + 1]) for k in range(args.steps)]

    e2e_ms, e2e_steps, h2d, d2h = None, 0, 0, 0
    if not args.no_e2e:
        e2e_ms, e2e_steps, h2d, d2h = run_e2e(args, prob, ctx, stream, dev, world)
    tail = verify_tail(prob, dm, stream, dev) if world == 1 else None
    d_ms, d_steps = None, 0
    if not args.no_deferred:
        d_ms, d_steps = run_deferred(args, prob, dm, stream, dev, world)
    long_window = None
    if not args.no_deferred and world == 1 and args.config != "C3":
        long_window = run_long_window(args, dev)

    # aggregate over ranks: units of all ranks / the slowest rank's time
    t_max = max_over_ranks(elapsed_ms, world)
    e_max = max_over_ranks(e2e_ms, world) if e2e_ms is not None else None
    tokens_all = sum_over_ranks(acct["tokens"] * args.steps, world)
    tokens_e2e = sum_over_ranks(acct["tokens"] * e2e_steps, world)
    bytes_all = sum_over_ranks(acct["step_bytes"] * args.steps, world)
    d_max = max_over_ranks(d_ms, world) if d_ms is not None else None
    tokens_d = sum_over_ranks(acct["tokens"] * d_steps, world)
    bytes_d = sum_over_ranks(acct["deferred_step_bytes"] * d_steps, world)
    if rank != 0:
        return None
    ms_per_step = t_max / args.steps
    value = tokens_all / (t_max / 1e3)
    achieved = bytes_all / (t_max / 1e3) / 1e9
    peak, peak_kind = measured_peak_gbs()
    v_avg = statistics.mean(verify_ms)
    c_avg = statistics.mean(commit_ms)
    v_gbs = acct["verify_layer_bytes"] / (v_avg / 1e3) / 1e9
    c_gbs = acct["commit_bytes"] / (c_avg / 1e3) / 1e9
    v_share = L * v_avg / (L * v_avg + c_avg)
    workload = f"{args.config}"
    if v_share >= 0.5:
        dom, dom_gbs, dom_bytes, dom_ms = "kda_verify", v_gbs, acct["verify_layer_bytes"], v_avg
    else:
        dom, dom_gbs, dom_bytes, dom_ms = "kda_commit", c_gbs, acct["commit_bytes"], c_avg
    traffic = profiled_traffic("verify" if dom == "kda_verify" else "commit", workload)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cv, cstep, sample, threads, _ = time_oracle(args.config, steps=args.cpu_steps, warmup=1,
                                                    layers=args.layers)  # bounded: ~10-20 s
        cpu = {"value": cv, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample,
               "s_per_full_step": cstep}
        # the same oracle on one thread, one layer of the step (about a second)
        _, one_layer, _, _, _ = time_oracle(args.config, steps=1, warmup=0, threads=1, layers=1)
        cpu["one_thread"] = {"s_per_layer": one_layer, "s_per_layer_all_cores": cstep / cfg.L,
                             "sample": f"{args.config}: the request batch, verify + commit of one layer, 1 step"}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; inputs resident in HBM)",
        "config": workload_config(cfg, acct),
        "achieved_hbm_gbs": achieved,
        "pct_of_8tbs": 100.0 * achieved / NOMINAL_HBM_GBS,
        "pct_of_measured_hbm": 100.0 * achieved / peak,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": peak, "unit": "GB/s",
                     "frac": dom_gbs / peak, "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms},
        "kernels": {
            "kda_verify": {"launches_per_step": L, "avg_ms": v_avg, "bytes_per_launch": acct["verify_layer_bytes"],
                           "gbs": v_gbs, "share": v_share},
            "kda_commit": {"launches_per_step": 1, "avg_ms": c_avg, "bytes_per_launch": acct["commit_bytes"],
                           "gbs": c_gbs, "share": 1 - v_share, "items": acct["commit_items"]},
        },
        "e2e": None if e_max is None else {
            "value": tokens_e2e / (e_max / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
            "copies": "per layer on two copy streams, overlapping the other layers' kernels"},
        "deferred": None if d_max is None else {
            "value": tokens_d / (d_max / 1e3), "unit": "tokens/s", "ms_per_step": d_max / d_steps,
            "achieved_hbm_gbs": bytes_d / (d_max / 1e3) / 1e9,
            "algorithmic_bytes_per_step": acct["deferred_step_bytes"], "steps": d_steps,
            "schedule": "each layer's verify first folds the previous step's accepted records into the "
                        "checkpoint (kda_verify_fold), no commit launch"},
        "long_window": long_window,
        "verify_schedule": tail,
        # each kda_verify is two launches (the conv pass, then the verify kernel)
        "gpu_launches": args.steps * (2 * L + 1),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    return line


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    from workloads import CONFIGS
    cfg = CONFIGS[args.config]
    if args.layers:
        cfg = cfg.replace(L=args.layers)
    steps = args.steps
    value, per_step, sample, threads, acct = time_oracle(args.config, steps=steps, warmup=args.warmup,
                                                         layers=args.layers)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": workload_config(cfg, acct),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="C2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-steps", type=int, default=8, help="full oracle steps of the cpu_baseline sample")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the layer count (small cases for profiling; not a bench line)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-deferred", action="store_true", help="skip the deferred-schedule timing")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    launched = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and launched == 1:
        ap.error(f"--gpus {args.gpus}: one process per GPU; launch with "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus} ...")
    if launched > 1 and launched != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {launched}")
    rank, local, world = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_gpu(args, rank, local, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
