#!/usr/bin/env python3
"""Benchmark of the context-parallel ring-attention forward on GB300.

One step = one pass of the whole path over the 128K-token Llama-3-70B-shaped causal GQA workload
(B=1, T=131072, h=64, n_kv=8, d_k=128, n_cp=16, zigzag): token placement (gather of Q, K, V and
position ids), every virtual rank over every ring step with block skipping and the online
softmax, and the write-back of O and lse in natural order. Inputs stay resident in HBM; they
are 2.7 GB, larger than L2, so no flush is needed between steps.

Prints one JSON line. ``--impl reference`` times the fp64 CPU oracle instead (the reference
arm of this benchmark), on a bounded sample of rows of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "ring-attn fwd effective TFLOP/s on 1 GB300; % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "llama70b_zigzag_T128k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one attention launch on a workload and how they were taken, keyed by
# the sha256 prefix of the attention kernel source they were measured on: a changed kernel reports
# null until it is measured again. The 70B-shaped 128K launch is too large for a capture with more
# than the launch time, so its figure is a one-launch capture of the same kernel at T = 32768,
# scaled by the work units to the 128K launch (4 times): a lower bound there, where K/V tiles start
# to be re-read once two KV heads in flight fill L2.
MEASURED_TRAFFIC = {"d3d05013087c7b18": {"llama70b_zigzag_T128k": (4593913600 + 2132709888,
                                                        "one-launch ncu capture of the 128K launch itself, a single "
                                                        "pass (4,593,913,600 B read + 2,132,709,888 B written); the "
                                                        "reads exceed Q, K and V once by the K/V tiles L2 could not "
                                                        "keep between the units that share them")}}


def source_key(text: str) -> str:
    """sha256 of C++ source with its comments and blank space taken out, so that a comment edit
    does not orphan counters taken on the same code."""
    import hashlib
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)      # block comments
    text = re.sub(r"//[^\n]*", " ", text)                   # line comments
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def attention_source_hash() -> str:
    path = os.path.join(ROOT, "context_ring_attention_blockwise_gb300", "csrc", "attention.cu")
    with open(path, encoding="utf-8") as f:
        return source_key(f.read())


def measured_traffic(workload_name: str):
    """(bytes per launch, how it was measured) or (None, None)."""
    return MEASURED_TRAFFIC.get(attention_source_hash(), {}).get(workload_name, (None, None))


def reduce_max(value: float, dist, device=None) -> float:
    """The maximum of `value` over all ranks (the slowest rank sets the job's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank: float, world: int, max_ms_per_step: float) -> float:
    """Aggregate throughput: the work every rank did in one step over the slowest rank's step time."""
    return work_per_rank * world / (max_ms_per_step * 1e-3)


def flops_eff(w) -> float:
    """4*B*h*d per visible pair; causal pairs counted as T^2/2 (a diagonal block as half)."""
    pairs = w.T * w.T / 2 if w.causal else float(w.T) * w.T
    return 4.0 * w.B * w.h * w.d * pairs


def clock_adjusted(achieved: float, peak_tf: float, peaks: dict, clocks):
    """The achieved rate per GHz of the median SM clock during the timed region, and the fraction of
    the sustained peak scaled to that clock (the peak was measured at the median SM clock the peak
    file records under load): how close the kernel is to the tensor pipe clock for clock."""
    peak_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    mhz = clocks.get("sm_mhz") if clocks else None
    if not peak_mhz or not mhz:
        return None
    return {"tflops_per_ghz": achieved / (mhz / 1000.0), "peak_sm_mhz": peak_mhz, "run_sm_mhz": mhz,
            "frac_at_run_clock": achieved / (peak_tf * mhz / peak_mhz)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clock and throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# Reference arm and CPU baseline: the fp64 oracle on sampled rows
# ---------------------------------------------------------------------------------------------

def oracle_sample_rate(w, q, k, v, n_rows: int, seed: int):
    """Time the oracle on n_rows sampled query rows (all heads, whole batch); returns
    (effective TFLOP/s, seconds, sample description). Work counted as 4*d per visible pair."""
    import oracle
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.T, size=n_rows, replace=False)).astype(np.int64)
    pairs = float(np.sum(rows + 1)) if w.causal else float(n_rows) * w.T
    t0 = time.perf_counter()
    oracle.get().attention(q, k, v, causal=w.causal, rows=rows)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.d * w.h * w.B * pairs
    return flops / dt / 1e12, dt, f"{n_rows} uniformly drawn query rows x {w.h} heads x B={w.B} (seed {seed})"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_model() -> str:
    """The host CPU's model name (x86: "model name"; Arm: implementer and part numbers)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    key, val = (x.strip() for x in line.split(":", 1))
                    fields.setdefault(key, val)
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU implementer" in fields:
        return f"{platform.machine()} implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return platform.machine()


def cpu_baseline_entry(w, rate: float, seconds: float, sample: str) -> dict:
    """The oracle's rate with its per-core figure and the full workload's time extrapolated
    linearly in visible pairs (the oracle's cost per pair does not depend on the row)."""
    cores = host_cores()
    return {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
            "seconds": seconds, "per_core_gflops": rate * 1e3 / cores, "cpu": host_cpu_model(),
            "full_workload_s_extrapolated": flops_eff(w) / (rate * 1e12) if rate > 0 else None}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v = synth.make_qkv(w)
    import oracle
    oracle.build()
    rows_per_step = args.ref_rows
    for i in range(args.warmup):
        oracle_sample_rate(w, q, k, v, rows_per_step, seed=1000 + i)
    rates, times = [], []
    for i in range(args.steps):
        r, dt, desc = oracle_sample_rate(w, q, k, v, rows_per_step, seed=2000 + i)
        rates.append(r)
        times.append(dt)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": cpu_baseline_entry(w, value, float(np.sum(times)),
                                           f"per step: {rows_per_step} query rows x {w.h} heads of the workload"),
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, args):
    if args.path == "ring":
        par = (f"ring over {args.gpus} processes, {w.n_cp // args.gpus} ranks each" if args.gpus > 1
               else "single GPU, one process holding all ranks")
    elif args.path == "steps":
        par = "replicas of the ring-step path" if args.gpus > 1 else "single GPU, one launch per ring step"
    else:
        par = "replicas" if args.gpus > 1 else "single GPU"
    return {"workload": w.name, "B": w.B, "T": w.T, "h": w.h, "n_kv": w.n_kv, "d_k": w.d, "n_cp": w.n_cp,
            "layout": synth.LAYOUT_NAMES[args.layout], "causal": w.causal, "path": args.path,
            "l2": "inputs larger than L2 (no flush)" if w.T >= 65536 else "L2 flushed between steps",
            "parallelism": par}


# ---------------------------------------------------------------------------------------------
# The GPU arm
# ---------------------------------------------------------------------------------------------

def run_gpu_ring(args, w):
    """The multi-process ring: process p (one per GPU) holds ranks p R .. p R + R - 1 of the n_cp
    (R = n_cp / processes) and passes the block that crosses to the next process over NCCL; one
    process holds the whole ring and passes blocks between its own ranks. The work is the whole
    sequence's once, whatever the number of processes (strong scaling)."""
    import torch
    import context_ring_attention_blockwise_gb300 as cp
    from context_ring_attention_blockwise_gb300 import _build
    from context_ring_attention_blockwise_gb300.ring import NcclTransport, RingProcess, local_tokens

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if w.n_cp % world:
        raise SystemExit(f"n_cp = {w.n_cp} is not a multiple of {world} processes")
    _build.build()
    dev = torch.device("cuda", local)
    R = w.n_cp // world
    toks = local_tokens(w.T, w.n_cp, args.layout, rank * R, R)
    q_full, k_full, v_full = synth.make_qkv(w)
    q_h, k_h, v_h = (np.ascontiguousarray(x[:, toks]) for x in (q_full, k_full, v_full))
    del q_full, k_full, v_full

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v = to_dev(q_h), to_dev(k_h), to_dev(v_h)
    plan = cp.Plan(w.T, w.h, w.n_kv, w.d, w.n_cp, args.layout, w.causal)
    ring = RingProcess(plan, w.B, rank=rank, world=world, transport=NcclTransport(rank, world) if world > 1 else None,
                       device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.h, R * plan.T // w.n_cp), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=dev, priority=-1)   # ring hops: ahead of the e2e uploads
    for _ in range(args.warmup):
        ring.forward(q, k, v, out=o, lse=lse, stream=stream, copy_stream=copy)
    torch.cuda.synchronize()
    cp.check(plan, ring.backend.ws)
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        ring.forward(q, k, v, out=o, lse=lse, stream=stream, copy_stream=copy)
    b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    cp.check(plan, ring.backend.ws)
    ms_per_step = reduce_max(a.elapsed_time(b) / args.steps, dist, dev)
    value = flops_eff(w) / (ms_per_step * 1e-3) / 1e12

    # end to end: this process's shard from pinned host memory and its outputs back, every step,
    # double-buffered as in the fused path's e2e (upload of step i+1 and readback of step i-1 beside
    # the forward of step i)
    qp, kp, vp = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (q_h, k_h, v_h))
    bufs = [(q, k, v, o, lse),
            (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o), torch.empty_like(lse))]
    outs = [(torch.empty(o.shape, dtype=torch.bfloat16).pin_memory(),
             torch.empty(lse.shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_steps = max(3, args.steps)          # the same K steps as the device-timed region

    def e2e_run(n):
        computed, read = [None, None], [None, None]
        for i in range(n):
            sl = i % 2
            qb, kb, vb, ob, lb = bufs[sl]
            with torch.cuda.stream(up):
                if computed[sl] is not None:
                    up.wait_event(computed[sl])
                qb.copy_(qp, non_blocking=True)
                kb.copy_(kp, non_blocking=True)
                vb.copy_(vp, non_blocking=True)
                uploaded = torch.cuda.Event()
                uploaded.record(up)
            stream.wait_event(uploaded)
            if read[sl] is not None:
                stream.wait_event(read[sl])
            ring.forward(qb, kb, vb, out=ob, lse=lb, stream=stream, copy_stream=copy)
            computed[sl] = torch.cuda.Event()
            computed[sl].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[sl])
                outs[sl][0].copy_(ob, non_blocking=True)
                outs[sl][1].copy_(lb, non_blocking=True)
                read[sl] = torch.cuda.Event()
                read[sl].record(down)
        for r in read:
            if r is not None:
                stream.wait_event(r)

    e2e_run(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    a.record(stream)
    up.wait_stream(stream)
    e2e_run(e2e_steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(b) / e2e_steps, dist, dev)
    del bufs, outs
    # one more pass with an event timeline: does each hop end before the step beside it does?
    marks = []
    kv_before = ring.counters.kv[0]
    t0 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    ring.forward(q, k, v, out=o, lse=lse, stream=stream, copy_stream=copy, timeline=marks)
    torch.cuda.synchronize()
    timeline = hop_summary([t0.elapsed_time(ce) for ce, _ in marks], [t0.elapsed_time(xe) for _, xe in marks], False)
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    plan_counts = plan.counts(w.B)
    uploads = -(-(R * ((w.T // w.n_cp + 127) // 128)) // 960)
    result = None
    if rank == 0:
        result = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(w, args),
            "frac_of_peak": value / world / peak_tf,
            "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": value / world / peak_tf, "traffic": None,
                         "kernel": "whole ring path (placement, n_cp steps of ring_attention_kernel, finalize)",
                         "peak_kind": f"bf16 dense, sustained, {peak_src}",
                         "peak_burst": float(peaks.get("bf16_tflops", 0.0))},
            "e2e": {"value": flops_eff(w) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": int(q_h.nbytes + k_h.nbytes + v_h.nbytes),
                    "d2h_bytes_per_step": int(o.numel() * 2 + lse.numel() * 4)},
            "ring": {"processes": world, "ranks_per_process": R,
                     "kv_bytes_recv_per_rank": int(ring.counters.kv[0] - kv_before),
                     "timeline": timeline,
                     "kv_bytes_recv_per_rank_pages": int(plan_counts["kv_bytes_recv"][0]),
                     "transport": "NCCL send/recv" if world > 1 else "none (one process holds the ring)"},
            # per step: the order upload, placement (pos_tiles, tile_suffix, permute), per ring step
            # the tile counts and the attention kernel, and the write-back
            "gpu_launches": (uploads + 3 + 2 * w.n_cp + 1) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_gpu(args, w):
    import torch
    import context_ring_attention_blockwise_gb300 as cp
    from context_ring_attention_blockwise_gb300 import _build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    dev = torch.device("cuda", local)

    q_h, k_h, v_h = synth.make_qkv(w)
    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v = to_dev(q_h), to_dev(k_h), to_dev(v_h)
    plan = cp.Plan(w.T, w.h, w.n_kv, w.d, w.n_cp, args.layout, w.causal)
    ring = args.path == "steps"           # the ring-step path: permute, n_cp ring steps, finalize
    ws = cp.alloc_workspace(plan.ring_workspace_size(w.B) if ring else plan.workspace_size(w.B), dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.h, w.T), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=dev, priority=-1)   # ring hops: the next step waits on them
    flush = None
    if w.T < 65536:   # inputs below L2 size: flush between steps
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(evs=None):
        if flush is not None:
            flush.zero_()
        if evs:
            evs[0].record(stream)
        if ring:
            cp.ring_forward(q, k, v, plan, ws=ws, out=o, lse=lse, stream=stream)
        else:
            cp.permute(q, k, v, plan, ws, stream=stream)
            if evs:
                evs[1].record(stream)
            cp.attend(plan, w.B, ws, o, lse, stream=stream)
        if evs:
            evs[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    cp.check(plan, ws)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if dist is not None:
        dist.barrier()
    cp.check(plan, ws)
    total_ms = reduce_max(t_start.elapsed_time(t_end), dist, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(flops_eff(w), world, ms_per_step) / 1e12
    if ring:
        attn_ms = None
        perm_ms = None
    else:
        perm_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
        attn_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))

    # e2e through the public API with host buffers: every step copies its inputs from pinned host
    # memory and reads O and lse back into pinned host memory, inside the timed region. Two device
    # buffer sets and two copy streams double-buffer the steps, as a caller streaming batches
    # would: the upload of step i+1 and the readback of step i-1 overlap the forward of step i.
    qp = torch.from_numpy(q_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    kp = torch.from_numpy(k_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    vp = torch.from_numpy(v_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    bufs = [(q, k, v, o, lse),
            (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o), torch.empty_like(lse))]
    outs = [(torch.empty(o.shape, dtype=torch.bfloat16).pin_memory(),
             torch.empty(lse.shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_steps = max(3, args.steps)          # the same K steps as the device-timed region

    def e2e_run(n):
        computed = [None, None]   # forward of the last step that used each buffer set
        read = [None, None]       # readback of that step
        for i in range(n):
            s = i % 2
            qb, kb, vb, ob, lb = bufs[s]
            with torch.cuda.stream(up):
                if computed[s] is not None:
                    up.wait_event(computed[s])
                qb.copy_(qp, non_blocking=True)
                kb.copy_(kp, non_blocking=True)
                vb.copy_(vp, non_blocking=True)
                uploaded = torch.cuda.Event()
                uploaded.record(up)
            stream.wait_event(uploaded)
            if read[s] is not None:
                stream.wait_event(read[s])
            if ring:
                cp.ring_forward(qb, kb, vb, plan, ws=ws, out=ob, lse=lb, stream=stream)
            else:
                cp.forward(qb, kb, vb, plan, ws=ws, out=ob, lse=lb, stream=stream)
            computed[s] = torch.cuda.Event()
            computed[s].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[s])
                outs[s][0].copy_(ob, non_blocking=True)
                outs[s][1].copy_(lb, non_blocking=True)
                read[s] = torch.cuda.Event()
                read[s].record(down)
        for r in read:
            if r is not None:
                stream.wait_event(r)

    e2e_run(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    up.wait_stream(stream)
    e2e_run(e2e_steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(b) / e2e_steps, dist, dev)
    for s in range(2):
        assert torch.equal(outs[s][0].view(torch.int16), o.cpu().view(torch.int16)), "e2e readback differs from the device-resident forward"
    h2d = q_h.nbytes + k_h.nbytes + v_h.nbytes
    d2h = o.numel() * 2 + lse.numel() * 4

    peaks, peak_src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    result = None
    if rank == 0:
        kernel_ms = attn_ms if attn_ms is not None else ms_per_step
        achieved = flops_eff(w) / (kernel_ms * 1e-3) / 1e12
        # the library's kernels per step: the unit order's upload (960 entries a launch) and the
        # placement (pos_tiles, tile_suffix, permute), then per attention launch the per-row-group
        # tile counts and the attention kernel; the ring-step path launches attention once per
        # step and finalizes once
        n_qt = -(-(w.T // w.n_cp) // 128)
        n_grp = n_qt if (w.h // w.n_kv) % 2 == 0 else (n_qt + 1) // 2
        uploads = -(-(w.n_cp * n_grp) // 960)
        launches_per_step = (uploads + 3 + 2) if not ring else (uploads + 3 + 2 * w.n_cp + 1)
        result = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(w, args),
            "frac_of_peak": value / world / peak_tf,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": achieved / peak_tf,
                         "frac_of_burst": achieved / float(peaks.get("bf16_tflops", peak_tf)),
                         "clock_adjusted": clock_adjusted(achieved, peak_tf, peaks, clocks),
                         "traffic": args.traffic if args.traffic is not None else (None if ring else measured_traffic(w.name)[0]),
                         "traffic_how": None if ring else measured_traffic(w.name)[1],
                         "kernel": "ring_attention_kernel<128>" if not ring else "whole ring-step path",
                         "peak_kind": f"bf16 dense, sustained, {peak_src}",
                         "peak_burst": float(peaks.get("bf16_tflops", 0.0))},
            "kernels_ms": {"permute_and_placement": perm_ms, "attention": attn_ms},
            "e2e": {"value": whole_job_rate(flops_eff(w), world, e2e_ms) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
    del qp, kp, vp, outs, bufs
    # the secondary measurements and the CPU baseline belong to the single-GPU line: with more
    # ranks they would hold every GPU idle behind rank 0
    if rank == 0 and world == 1 and args.extras and not ring:
        result["extras"] = extras(cp, plan, w, q, k, v, ws, stream, copy, dev, peaks)
    if rank == 0 and world == 1 and args.cpu_baseline:
        rate, dt, desc = oracle_sample_rate(w, q_h, k_h, v_h, args.cpu_rows, seed=7)
        result["cpu_baseline"] = cpu_baseline_entry(w, rate, dt, desc)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def ring_timeline(step_fn, n_cp, stream, copy, next_step_bound):
    """Event timeline of one ring-step pass: timing events on the compute stream after each
    step's work and on the copy stream after that step's hops. A hop is hidden when it ends
    before the compute it must precede does: the same step's (next_step_bound = False: the
    forward's K/V hop for step s + 1 runs beside step s) or the next step's (True: the
    backward's gradient hop of step s is added into at step s + 1)."""
    import torch
    t0 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    marks = []
    for s in range(n_cp):
        step_fn(s)
        ce, xe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ce.record(stream)
        xe.record(copy)
        marks.append((ce, xe))
    torch.cuda.synchronize()
    return hop_summary([t0.elapsed_time(ce) for ce, _ in marks], [t0.elapsed_time(xe) for _, xe in marks],
                       next_step_bound)


def hop_summary(c_end, x_end, next_step_bound: bool) -> dict:
    """From the times (ms from the pass's start) at which each step's compute and its hops
    ended: per-step compute time, and each hop's slack before the compute it must precede
    (negative: exposed). The last step has no hop to hide (forward) or only the return hop,
    with no later step (backward)."""
    n = len(c_end)
    slack = [(c_end[s + 1] if next_step_bound else c_end[s]) - x_end[s] for s in range(n - 1)]
    step_ms = [c_end[0]] + [c_end[s] - c_end[s - 1] for s in range(1, n)]
    return {"steps": n, "step_ms_min": min(step_ms), "step_ms_max": max(step_ms),
            "hops_hidden": all(x >= 0 for x in slack), "min_slack_ms": min(slack) if slack else None,
            "exposed_ms_total": sum(max(0.0, -x) for x in slack)}


def extras(cp, plan, w, q, k, v, ws, stream, copy, dev, peaks):
    """Secondary measurements: the ring-step path at the same workload, and the HBM-bound
    kernels (placement, merge) against the measured copy bandwidth."""
    import torch
    out = {}
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # placement: reads and writes Q, K, V once
    moved = 2 * (q.numel() + k.numel() + v.numel()) * 2
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(2):
        cp.permute(q, k, v, plan, ws, stream=stream)
    a.record(stream)
    for _ in range(5):
        cp.permute(q, k, v, plan, ws, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / 5
    out["placement"] = {"ms": ms, "gbs": moved / ms / 1e6, "frac_of_hbm": moved / ms / 1e6 / hbm}
    # standalone merge of two fp32 partials at the workload's (T, h, d)
    rows = w.B * w.T
    S = 2
    op = torch.randn((S, rows, w.h, w.d), dtype=torch.float32, device=dev)
    lp = torch.randn((S, w.h, rows), dtype=torch.float32, device=dev)
    mo = torch.empty((rows, w.h, w.d), dtype=torch.bfloat16, device=dev)
    ml = torch.empty((w.h, rows), dtype=torch.float32, device=dev)
    for _ in range(2):
        cp.merge(op, lp, mo, ml, stream=stream)
    a.record(stream)
    for _ in range(5):
        cp.merge(op, lp, mo, ml, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / 5
    mb = op.numel() * 4 + lp.numel() * 4 + mo.numel() * 2 + ml.numel() * 4
    out["merge_S2"] = {"ms": ms, "gbs": mb / ms / 1e6, "frac_of_hbm": mb / ms / 1e6 / hbm}
    del op, lp, mo, ml
    # the n_cp-way merge at the GQA 16K shape (8 partials of [16384, 32, 128]): one partial per
    # virtual rank's view of a row, the most partials the ring-step path combines
    ws16 = synth.workload("gqa_zigzag_T16k")
    S, rows = ws16.n_cp, ws16.B * ws16.T
    op = torch.randn((S, rows, ws16.h, ws16.d), dtype=torch.float32, device=dev)
    lp = torch.randn((S, ws16.h, rows), dtype=torch.float32, device=dev)
    mo = torch.empty((rows, ws16.h, ws16.d), dtype=torch.bfloat16, device=dev)
    ml = torch.empty((ws16.h, rows), dtype=torch.float32, device=dev)
    for _ in range(2):
        cp.merge(op, lp, mo, ml, stream=stream)
    a.record(stream)
    for _ in range(5):
        cp.merge(op, lp, mo, ml, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / 5
    mb = op.numel() * 4 + lp.numel() * 4 + mo.numel() * 2 + ml.numel() * 4
    out[f"merge_S{S}_{ws16.name}"] = {"ms": ms, "gbs": mb / ms / 1e6, "frac_of_hbm": mb / ms / 1e6 / hbm}
    del op, lp, mo, ml
    # the ring-faithful path: permute, n_cp steps, finalize. By default each step's kernel moves
    # the blocks for the next step itself (its idle warps copy while the attention runs), so the
    # hop ends with the step; the same path with the hops on a copy stream follows.
    wsr = cp.alloc_workspace(plan.ring_workspace_size(w.B), dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.h, w.T), dtype=torch.float32, device=dev)

    def ring_pass_ms(copy_stream, passes=2):
        cp.ring_forward(q, k, v, plan, ws=wsr, out=o, lse=lse, stream=stream, copy_stream=copy_stream)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(passes):
            cp.ring_forward(q, k, v, plan, ws=wsr, out=o, lse=lse, stream=stream, copy_stream=copy_stream)
        b.record(stream)
        torch.cuda.synchronize()
        cp.check(plan, wsr)
        return a.elapsed_time(b) / passes

    ms = ring_pass_ms(None)
    o2, lse2 = torch.empty_like(q), torch.empty((w.B, w.h, w.T), dtype=torch.float32, device=dev)
    cp.permute(q, k, v, plan, wsr, stream=stream)
    tl = ring_timeline(lambda s: cp.ring_step(plan, w.B, s, wsr, compute=stream, copy=None), plan.n_cp, stream,
                       stream, False)
    cp.finalize(plan, w.B, wsr, o2, lse2, stream=stream)
    torch.cuda.synchronize()
    cp.check(plan, wsr)
    # the hop is part of each step's kernel, so it cannot end after its step: no separate copy
    # to time (the step times above include it)
    tl.update({"hops_hidden": True, "min_slack_ms": None, "exposed_ms_total": 0.0,
               "hop": "in the step's kernel: its two idle warps per CTA copy every rank's block into the next slot"})
    out["ring_step_path"] = {"ms_per_step": ms, "tflops_eff": flops_eff(w) / (ms * 1e-3) / 1e12, "timeline": tl}
    # the hops on a copy stream instead, with an event timeline: does each K/V hop end before the
    # step beside it?
    ms_c = ring_pass_ms(copy)
    cp.permute(q, k, v, plan, wsr, stream=stream)
    tl_c = ring_timeline(lambda s: cp.ring_step(plan, w.B, s, wsr, compute=stream, copy=copy), plan.n_cp, stream, copy,
                         False)
    cp.finalize(plan, w.B, wsr, o2, lse2, stream=stream)
    torch.cuda.synchronize()
    cp.check(plan, wsr)
    out["ring_step_path"]["copy_stream"] = {"ms_per_step": ms_c, "tflops_eff": flops_eff(w) / (ms_c * 1e-3) / 1e12,
                                            "timeline": tl_c}
    # the same with SMs left free during the attention launches, so that the device-to-device hop
    # of the next block can run beside the step instead of in its tail
    for reserve in (4, 8):
        plan.set_reserved_sms(reserve)
        cp.ring_forward(q, k, v, plan, ws=wsr, out=o2, lse=lse2, stream=stream, copy_stream=copy)
        torch.cuda.synchronize()
        a.record(stream)
        cp.ring_forward(q, k, v, plan, ws=wsr, out=o2, lse=lse2, stream=stream, copy_stream=copy)
        b.record(stream)
        torch.cuda.synchronize()
        ms_r = a.elapsed_time(b)
        cp.permute(q, k, v, plan, wsr, stream=stream)
        tl = ring_timeline(lambda s: cp.ring_step(plan, w.B, s, wsr, compute=stream, copy=copy), plan.n_cp, stream,
                           copy, False)
        cp.finalize(plan, w.B, wsr, o2, lse2, stream=stream)
        torch.cuda.synchronize()
        cp.check(plan, wsr)
        out["ring_step_path"]["copy_stream"][f"reserved_sms_{reserve}"] = {"ms_per_step": ms_r,
                                                             "tflops_eff": flops_eff(w) / (ms_r * 1e-3) / 1e12,
                                                             "timeline": tl}
    plan.set_reserved_sms(0)
    del wsr, o2, lse2
    # document masks: the same workload packed with seeded documents of 2K..16K tokens
    rng = np.random.default_rng(w.seed)
    lengths = []
    while sum(lengths) < w.T:
        lengths.append(int(rng.integers(2048, 16385)))
    lengths[-1] -= sum(lengths) - w.T
    lengths = [x for x in lengths if x > 0]
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    lo = torch.from_numpy(np.repeat(starts, lengths).astype(np.int32)).to(dev)
    pairs = sum(x * (x + 1) // 2 for x in lengths)
    flops_docs = 4.0 * w.B * w.h * w.d * pairs
    od, lsed = torch.empty_like(o), torch.empty_like(lse)
    cp.forward_masked(q, k, v, plan, lo, ws=ws, out=od, lse=lsed, stream=stream)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(3):
        cp.forward_masked(q, k, v, plan, lo, ws=ws, out=od, lse=lsed, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    ms = a.elapsed_time(b) / 3
    out["documents"] = {"ms": ms, "documents": len(lengths), "tflops_eff": flops_docs / (ms * 1e-3) / 1e12,
                        "flops": "4 B h d per visible (query, key) pair inside each document"}
    # the same documents given as ids in shuffled order (the document-id mask: tile classes from
    # each tile's id range, a bitmask walk, the id compare in the element mask)
    ids = rng.permutation(len(lengths)).astype(np.int32) * 7 + 1
    docd = torch.from_numpy(np.repeat(ids, lengths).astype(np.int32)).to(dev)
    cp.forward_docs(q, k, v, plan, docd, ws=ws, out=od, lse=lsed, stream=stream)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(3):
        cp.forward_docs(q, k, v, plan, docd, ws=ws, out=od, lse=lsed, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    ms = a.elapsed_time(b) / 3
    out["document_ids"] = {"ms": ms, "documents": len(lengths), "ids": "shuffled", "tflops_eff": flops_docs / (ms * 1e-3) / 1e12}
    # short documents: 64 of 2048 tokens (the unit boundaries dominate)
    lo64 = torch.from_numpy((np.arange(w.T) // 2048 * 2048).astype(np.int32)).to(dev)
    flops64 = 4.0 * w.B * w.h * w.d * (w.T // 2048) * (2048 * 2049 // 2)
    cp.forward_masked(q, k, v, plan, lo64, ws=ws, out=od, lse=lsed, stream=stream)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(3):
        cp.forward_masked(q, k, v, plan, lo64, ws=ws, out=od, lse=lsed, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    ms = a.elapsed_time(b) / 3
    out["documents_64x2k"] = {"ms": ms, "documents": w.T // 2048, "tflops_eff": flops64 / (ms * 1e-3) / 1e12}
    del lo64
    del od, lsed, lo, docd
    # the backward pass: dq, dk, dv from the forward's o and lse and a synthetic output gradient
    wsb = cp.alloc_workspace(plan.backward_workspace_size(w.B), dev)
    dout = torch.randn(q.shape, dtype=torch.bfloat16, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    cp.backward(q, k, v, o, lse, dout, plan, ws=wsb, dq=dq, dk=dk, dv=dv, stream=stream)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(2):
        cp.backward(q, k, v, o, lse, dout, plan, ws=wsb, dq=dq, dk=dk, dv=dv, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    cp.check(plan, wsb)
    ms = a.elapsed_time(b) / 2
    tf = 2.5 * flops_eff(w) / (ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    out["backward"] = {"ms": ms, "tflops_eff": tf, "frac_of_bf16_sustained": tf / peak,
                       "convention": "2.5 x the forward's effective FLOPs (five GEMMs per visible tile pair); "
                                     "the kernels compute seven (dQ recomputes S and dP)",
                       "includes": "placement, D = <dO, O> prep, dK/dV kernel, dQ kernel",
                       "ring_bytes_recv_per_rank": int(plan.backward_counts(w.B)["bytes_recv"][0]),
                       "ring_bytes_note": "K and V blocks (bf16) plus the circulating dK and dV blocks (fp32 partial sums)"}
    del wsb
    # the backward as ring steps: each step's kernels on the compute stream; K/V and the fp32
    # dK/dV partial sums hop between the ranks' slots on the copy stream
    wsr = cp.alloc_workspace(plan.backward_ring_workspace_size(w.B), dev)
    cp.ring_backward(q, k, v, o, lse, dout, plan, ws=wsr, dq=dq, dk=dk, dv=dv, stream=stream, copy_stream=copy)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(2):
        cp.ring_backward(q, k, v, o, lse, dout, plan, ws=wsr, dq=dq, dk=dk, dv=dv, stream=stream, copy_stream=copy)
    b.record(stream)
    torch.cuda.synchronize()
    cp.check(plan, wsr)
    ms = a.elapsed_time(b) / 2
    tf = 2.5 * flops_eff(w) / (ms * 1e-3) / 1e12
    out["backward_ring_step_path"] = {"ms": ms, "tflops_eff": tf, "frac_of_bf16_sustained": tf / peak,
                                      "includes": "placement and prep, n_cp steps of the dQ and dK/dV kernels (the "
                                                  "contributions reduced into the circulating sums) with the K/V and "
                                                  "gradient hops, finalize"}
    # event timeline: does each step's gradient hop end before the next step's work is done? (Its
    # dK/dV kernel waits for that hop; the dQ kernel before it overlaps the hop.)
    cp.backward_begin(q, k, v, o, lse, dout, plan, wsr, stream=stream)
    out["backward_ring_step_path"]["timeline"] = ring_timeline(
        lambda s: cp.backward_ring_step(plan, w.B, s, wsr, compute=stream, copy=copy), plan.n_cp, stream, copy, True)
    cp.backward_finalize(plan, w.B, wsr, dq, dk, dv, stream=stream)
    torch.cuda.synchronize()
    cp.check(plan, wsr)
    del wsr, dout, dq, dk, dv
    # the all-gather variant at the 405B per-TP slice (one KV head per rank, the pages' 63 MB case):
    # the exposed gather beside the attention launch that follows it
    out["allgather"] = allgather_extra(cp, dev, peaks)
    # the head split (Ulysses) as the comparison workload: all-to-all, per-rank attention over
    # every token of h / n_cp heads, all-to-all back; bytes per rank against the ring's
    up = cp.UlyssesPlan(w.T, w.h, w.n_kv, w.d, w.n_cp, w.causal)
    wsu = cp.alloc_workspace(up.workspace_size(w.B), dev)
    ou, lseu = torch.empty_like(o), torch.empty_like(lse)
    cp.ulysses_forward(q, k, v, up, ws=wsu, out=ou, lse=lseu, stream=stream)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(3):
        cp.ulysses_forward(q, k, v, up, ws=wsu, out=ou, lse=lseu, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    cp.check(up, wsu)
    ms = a.elapsed_time(b) / 3
    out["ulysses"] = {"ms": ms, "tflops_eff": flops_eff(w) / (ms * 1e-3) / 1e12, "n_cp": w.n_cp,
                      "heads_per_rank": w.h // w.n_cp, "kv_heads_per_rank": max(w.n_kv // w.n_cp, 1),
                      "a2a_bytes_recv_per_rank": int(up.counts(w.B)["bytes_recv"][0]),
                      "ring_kv_bytes_recv_per_rank": int(plan.counts(w.B)["kv_bytes_recv"][0]),
                      "includes": "both all-to-alls (as on-GPU layout switches) and the per-rank attention"}
    del wsu, ou, lseu, up
    return out


def allgather_extra(cp, dev, peaks):
    """The all-gather variant on the 405B per-TP slice (T = 131072, h = 16, one KV head, 16 ranks):
    placement, the gather of every rank's copy of K and V (timed alone: the exposed phase), and
    the attention launch over the gathered copies; beside it the ring's fused launch on the same
    placement. Bytes per rank from the library's count (the pages' 63 MB)."""
    import torch
    w = synth.workload("llama405b_tp_T128k")
    q_h, k_h, v_h = synth.make_qkv(w)
    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v = to_dev(q_h), to_dev(k_h), to_dev(v_h)
    plan = cp.Plan(w.T, w.h, w.n_kv, w.d, w.n_cp, w.layouts[0], w.causal)
    ws = cp.alloc_workspace(plan.allgather_workspace_size(w.B), dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.h, w.T), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    cp.allgather_forward(q, k, v, plan, ws=ws, out=o, lse=lse, stream=stream)
    torch.cuda.synchronize()
    reps = 3
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    for r in range(reps):
        cp.permute(q, k, v, plan, ws, stream=stream)
        ev[r][0].record(stream)
        cp.allgather_gather(plan, w.B, ws, stream=stream)
        ev[r][1].record(stream)
        cp.allgather_attend(plan, w.B, ws, o, lse, stream=stream)
        ev[r][2].record(stream)
        cp.attend(plan, w.B, ws, o, lse, stream=stream)
        ev[r][3].record(stream)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    gather_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    attend_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    ring_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in ev]))
    recv = int(plan.allgather_counts(w.B)["bytes_recv"][0])
    copied = 2 * w.n_cp * (k_h.nbytes + v_h.nbytes)      # read + write of every rank's copy
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"workload": f"{w.name} {synth.LAYOUT_NAMES[w.layouts[0]]}", "gather_ms": gather_ms,
            "attention_ms": attend_ms, "exposed_frac": gather_ms / (gather_ms + attend_ms),
            "ring_fused_attention_ms": ring_ms, "bytes_recv_per_rank": recv,
            "gather_gbs": copied / gather_ms / 1e6, "gather_frac_of_hbm": copied / gather_ms / 1e6 / hbm,
            "tflops_eff_attention": flops_eff(w) / (attend_ms * 1e-3) / 1e12,
            "pages": "63 MB per GPU per layer, about 1.3 ms over InfiniBand, against about 27 ms of compute"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.CONFIGS))
    ap.add_argument("--layout", default=None, help="contiguous|zigzag|striped (default: the workload's first)")
    ap.add_argument("--path", choices=["fused", "ring", "steps"], default="fused",
                    help="fused: one persistent launch over every rank and step; ring: the ring across "
                         "processes (one per GPU), each holding n_cp / processes ranks; steps: the "
                         "single-process ring-step path (one launch per step, hops inside the step kernels)")
    ap.add_argument("--traffic", type=float, default=None, help="DRAM bytes per attention launch from ncu, if known")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--cpu-rows", type=int, default=256, help="query rows the CPU baseline computes (~13 s on 16 cores)")
    ap.add_argument("--ref-rows", type=int, default=8, help="query rows per step of the reference arm")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="run the workload's shape at a shorter T (for small profiling captures)")
    args = ap.parse_args()
    w = synth.workload(args.workload)
    if args.seq_len is not None:
        import dataclasses
        w = dataclasses.replace(w, T=args.seq_len, name=f"{w.name}@T{args.seq_len}")
    args.layout = w.layouts[0] if args.layout is None else synth.LAYOUT_IDS[args.layout]
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.path == "ring":
        return run_gpu_ring(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
