"""Benchmark: banded + global sparse attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 5] [--impl ours|reference]

One step = one sa_forward call over one batch of the long-context workload
(B=1, H=16, N=131072, D=128, window 1024, globals 0..63, bf16): band tiles,
global-row split-K pass, merge (the global rows are contiguous, so they are read
in place; a scattered set adds a gather).  The metric is useful
(in-mask) attention FLOP/s: 4*D per scored (query, key) pair, pairs counted
exactly by sa_count_pairs.  Inputs (1.6 GB) are larger than the 129 MB L2, so
no flush is needed between steps.  The ``e2e`` key times the same work from
host memory: one sa_forward_host call per step on pinned q, k, v (copies in,
attention, copy of the output back, inside the call and the timed region).

Prints ONE JSON line on rank 0.  Under torchrun each rank runs its own
independent batch (weak scaling) and the time is the max over ranks.
``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample of
rows of the same workload.

``--workload gather`` times the other workload instead: attention over
per-query key lists (sa_forward_gather) on the retrieval shape (B=1, H=16,
4096 queries per head, each attending to 1024 of 131072 keys, D=128, bf16).
Its metric is the key/value bytes the lists name, gathered per second, beside
the useful TFLOP/s (4*D per valid list entry).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_long_context_banded_gb300 import inputs  # noqa: E402

METRIC = "in-mask attention TFLOP/s & % of bf16 TC peak on 1 GB300 (N=4K–128K)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # about a second of timed work at the default workload, so that the 200 ms
    # clock sampler sees the GPU under load several times
    ap.add_argument("--steps", type=int, default=600)  # >= 50: the headline is their median
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="5",
                    help="workload number 1..5, or 'gather' for the list-attention workload")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--oracle-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tf32", action="store_true",
                    help="fp32 workloads: tf32 products on the tensor cores (SA_TF32)")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the workload with this many heads (profiling a smaller case)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one call captured in a CUDA graph (after the eager "
                         "warm-up); the per-stage pass and e2e stay eager")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p.get("bf16_tflops_sustained"),
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def measured_traffic(workload: int):
    """DRAM bytes (read + write) per launch of the attention kernel from an ncu
    capture, if one was taken of the kernel source as it is now: the capture's
    record names the SHA-256 of the kernel source it was taken of, and a record
    of another source gives None."""
    import hashlib
    rec_path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "sparse_long_context_banded_gb300", "csrc", "sa_tc.cu")
    if not os.path.exists(rec_path):
        return None, "no ncu capture recorded"
    with open(rec_path) as f:
        rec = json.load(f)
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    entry = rec.get(str(workload))
    if not entry:
        return None, "no ncu capture of this workload"
    if entry.get("kernel_source_sha256") != digest:
        return None, "ncu capture taken of another kernel source"
    return entry["dram_bytes_per_launch"], entry["source"]


def workload_flops(w, sa):
    """In-mask FLOPs per step: total and the band kernel's share (non-global rows)."""
    per_head, total = sa.count_pairs(w.N, w.window, w.dilation, w.H, w.globals_)
    pairs = w.B * total
    global_pairs = w.B * w.H * len(w.globals_) * w.N
    return 4.0 * w.D * pairs, 4.0 * w.D * (pairs - global_pairs), pairs


def rank_seed(w, rank: int) -> int:
    """Seed of rank `rank`'s batch: rank 0 uses the workload's own seed, other
    ranks independent batches of the same shape (weak scaling)."""
    return 1000 + w.number + (7919 * rank if rank else 0)


def job_value(flops_per_step: float, steps: int, ms_max: float, world: int) -> float:
    """Whole-job TFLOP/s: work of all ranks over the slowest rank's time."""
    return world * flops_per_step * steps / (ms_max * 1e-3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("SA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return rank, world


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file.read().splitlines() if ln.strip()]
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if len(r) > 1 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 2 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        loaded = [x for x in sm if x > 0.5 * (max(mx) if mx else 0)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def oracle_sample_timing(w, qkv, target_seconds: float, seed: int = 0):
    """Time the fp64 oracle on a random sample of rows of the workload.

    Returns (tflops, seconds, rows, threads).  The sample is uniform over all
    B*H*N rows; its FLOPs are counted exactly from each sampled row's mask size.
    """
    import oracle
    from sparse_long_context_banded_gb300 import sa

    o = oracle.default()
    threads = oracle.default_threads()
    q, k, v = qkv
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.H * w.N
    # per-row mask sizes (exact): band length + globals outside it, or N for a global row
    G = np.array(w.globals_, dtype=np.int64)

    def row_pairs(rows):
        i = rows % w.N
        h = (rows // w.N) % w.H
        d = np.array(w.dilation, dtype=np.int64)[h]
        half = w.window // 2
        lo = np.maximum(-half, -(i // d))
        hi = np.minimum(half, (w.N - 1 - i) // d)
        cnt = hi - lo + 1
        for g in G:
            diff = i - g
            inside = (np.abs(diff) <= half * d) & (diff % d == 0)
            cnt += (~inside).astype(np.int64)
        is_g = np.isin(i, G)
        cnt[is_g] = w.N
        return cnt

    n = 256
    while True:
        rows = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False))
        t0 = time.perf_counter()
        o.forward_longformer(q, k, v, w.window, w.dilation, w.globals_, scale=w.scale,
                             rows=rows, threads=threads, want_lse=False)
        dt = time.perf_counter() - t0
        if dt >= target_seconds or n >= total_rows:
            break
        n = int(min(total_rows, max(2 * n, n * target_seconds / max(dt, 1e-3) * 1.1)))
    flops = 4.0 * w.D * float(row_pairs(rows).sum())
    return flops / dt / 1e12, dt, int(rows.size), threads


def run_reference(args):
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    w = inputs.workload(args.workload)
    qkv = inputs.draw_qkv(w)
    # each step is a bounded sample; the whole run stays near two minutes of CPU work
    per_step = max(0.05, min(args.oracle_seconds, 75.0 / max(1, args.steps + args.warmup)))
    vals, secs = [], []
    rows = threads = 0
    for s in range(args.warmup + args.steps):
        tf, dt, rows, threads = oracle_sample_timing(w, qkv, per_step, seed=s)
        if s >= args.warmup:
            vals.append(tf)
            secs.append(dt)
    value = statistics.median(vals)
    sample = (f"{rows} uniformly drawn query rows of {w.B * w.H * w.N} per step "
              f"(~{statistics.median(secs):.1f} s of fp64 CPU work)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.describe(), "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "window": w.window, "n_globals": len(w.globals_)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    from sparse_long_context_banded_gb300 import build, sa

    rank, world = dist_setup()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    sa.load()

    w = inputs.workload(args.workload)
    if args.heads:
        w = dataclasses.replace(w, H=args.heads, dilation=w.dilation[:1] * args.heads)
    # each rank runs its own independent batch of the workload (weak scaling)
    qkv = inputs.draw_qkv(w, seed=rank_seed(w, rank))
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def host_tensor(a):
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
            else torch.from_numpy(a)
        return t

    hq, hk, hv = (host_tensor(a) for a in qkv)
    q, k, v = (t.to(dev) for t in (hq, hk, hv))
    out = torch.empty_like(q)
    flops_step, band_flops, pairs = workload_flops(w, sa)
    stream = torch.cuda.current_stream(dev)

    tf32 = bool(args.tf32) and w.dtype == "fp32"

    def eager_step():
        sa.forward(q, k, v, w.window, w.dilation, w.globals_, scale=w.scale, out=out, stream=stream,
                   tf32=tf32)

    step = eager_step
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sa.sync_status(stream)
    if args.graph:
        # one call captured on a side stream (the first eager calls built the
        # schedule); the timed steps replay it on the launching stream
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                sa.forward(q, k, v, w.window, w.dilation, w.globals_, scale=w.scale, out=out,
                           stream=side, tf32=tf32)
        torch.cuda.synchronize()

        def step():
            graph.replay()

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        sa.sync_status(stream)

    # inputs smaller than L2 (129 MB): write a 512 MB buffer between steps, outside
    # the per-step events, so that no step finds its inputs in L2
    in_bytes = 4 * q.numel() * q.element_size()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if in_bytes < (512 << 20) else None
    # timed region: K steps with no instrumentation but one CUDA event between
    # consecutive steps (the per-step times; their median is the headline)
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    if flush is None:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        evs[0].record(stream)
        for i in range(args.steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    else:
        pairs_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(args.steps)]
        for a, b in pairs_ev:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        step_ms = [a.elapsed_time(b) for a, b in pairs_ev]
    barrier(world)
    clocks = sampler.stop()
    sa.sync_status(stream)
    ms_median_local = statistics.median(step_ms)
    ms_step = max_over_ranks(ms_median_local, world, dev)
    ms_mean = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    value = job_value(flops_step, 1, ms_step, world)

    # per-kernel times from a separate, instrumented pass (CUDA events around
    # every launch on the launching stream)
    prof_steps = max(10, min(50, args.steps))
    sa.profile_begin()
    for _ in range(prof_steps):
        if flush is not None:
            flush.zero_()
        eager_step()
    torch.cuda.synchronize()
    prof = sa.profile_end()
    launches_per_step = sum(p["launches"] for p in prof.values()) / prof_steps

    pk = peaks()
    # the dominant kernel: the band launch, which on the tensor cores also runs
    # the global rows (then its algorithmic work is every in-mask pair)
    fused = prof["global_rows"]["launches"] == 0 and len(w.globals_) > 0
    kern_flops = flops_step if fused else band_flops
    kern_ms = prof["band"]["ms"] / max(1, prof["band"]["launches"])
    kern_tflops = kern_flops / (kern_ms * 1e-3) / 1e12
    traffic, traffic_src = measured_traffic(args.workload) if not args.heads else (None, "")

    # end to end through the C ABI with host buffers: every step is one
    # sa_forward_host call on pinned q, k, v, which copies them in, runs the
    # attention and copies the output back, overlapping the copies of one
    # group of heads with the computation of another; the call returns when
    # the output is in host memory, so the host clock times it
    e2e = None
    if not args.no_e2e:
        pq, pk_, pv = (t.pin_memory() for t in (hq, hk, hv))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def host_step():
            sa.forward_host(pq, pk_, pv, w.window, w.dilation, w.globals_, scale=w.scale,
                            out=hout, tf32=tf32, device=dev)

        for _ in range(2):
            host_step()
        e2e_steps = max(4, min(args.steps, 12))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        ms_e2e = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
        h2d = 3 * q.numel() * q.element_size()
        d2h = out.numel() * out.element_size()
        e2e = {"value": world * flops_step * e2e_steps / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ms_e2e / e2e_steps, "steps": e2e_steps,
               "call": "sa_forward_host on pinned host tensors (copies in, attention, copy "
                       "out; groups of heads pipelined inside the call)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, secs, rows, threads = oracle_sample_timing(w, qkv, args.oracle_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} uniformly drawn query rows of {w.B * w.H * w.N}, "
                         f"{secs:.1f} s of fp64 CPU work"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_stat": f"median of {args.steps} per-step CUDA-event times "
                                f"(max over ranks); mean {ms_mean:.4f} ms",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if w.dtype == "bf16" else ("tf32" if tf32 else "fp32"), "data": "synthetic",
            "config": {"workload": w.describe(), "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                       "window": w.window, "n_globals": len(w.globals_),
                       "in_mask_pairs_per_step": pairs * world,
                       "in_mask_gflop_per_step": flops_step * world / 1e9,
                       "launch": "CUDA graph replay of one captured call" if args.graph
                       else "eager sa.forward calls",
                       "l2": (f"inputs ({in_bytes / 1e9:.2f} GB) larger than L2; no flush"
                              if flush is None else
                              f"inputs ({in_bytes / 1e6:.0f} MB) smaller than L2: a 512 MB "
                              f"buffer written between steps, outside the per-step events"),
                       "pct_of_bf16_peak": 100.0 * value / (world * pk["bf16_tflops"]),
                       "pct_of_bf16_peak_sustained": (100.0 * value / (world * pk["bf16_tflops_sustained"])
                                                      if pk.get("bf16_tflops_sustained") else None)},
            "roofline": {"bound": "tensor",
                         "kernel": "band + global rows (one launch)" if fused else "band",
                         "achieved": kern_tflops,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": kern_tflops / pk["bf16_tflops"],
                         "traffic": traffic, "traffic_source": traffic_src,
                         "peak_source": f"{pk['source']} bf16 dense (burst)",
                         "frac_of_sustained": (kern_tflops / pk["bf16_tflops_sustained"]
                                               if pk.get("bf16_tflops_sustained") else None),
                         "algorithmic_flops_per_launch": kern_flops,
                         "ms_per_launch": kern_ms,
                         "timing": f"CUDA events around each launch, {prof_steps} steps of a "
                                   f"separate pass after the timed region"},
            "stages_ms_per_step": {s: prof[s]["ms"] / prof_steps for s in prof},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_gather(args):
    """One step = one sa_forward_gather call over the retrieval workload."""
    import torch

    from sparse_long_context_banded_gb300 import build, sa

    rank, world = dist_setup()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    sa.load()
    w = inputs.gather_workload()
    q_, k_, v_, idx_ = inputs.draw_gather(w, seed=rank)
    valid = int((idx_ >= 0).sum())
    gathered = valid * 2 * w.D * 2  # key and value row per valid entry, bf16
    flops_step = 4.0 * w.D * valid

    def dev_tensor(a):
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
            else torch.from_numpy(a)
        return t.to(dev)

    q, k, v, idx = (dev_tensor(a) for a in (q_, k_, v_, idx_))
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def step():
        sa.forward_gather(q, k, v, idx, scale=w.scale, out=out, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sa.sync_status(stream)
    steps = max(1, min(args.steps, 200))
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    sa.profile_begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    prof = sa.profile_end()
    barrier(world)
    clocks = sampler.stop()
    sa.sync_status(stream)
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / steps
    kernel_ms = prof["band"]["ms"] / max(1, prof["band"]["launches"])
    pk = peaks()
    if rank == 0:
        gbs = gathered / (kernel_ms * 1e-3) / 1e9
        line = {
            "metric": "list attention: gathered key/value GB/s", "value":
                world * gathered * steps / (ms_total * 1e-3) / 1e9, "unit": "GB/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.describe(), "valid_entries_per_step": valid * world,
                       "useful_tflops": world * flops_step * steps / (ms_total * 1e-3) / 1e12,
                       "l2": "lists name 34 GB of rows per step; repeats across queries "
                             "are served from L2 (head-major order), no flush"},
            "roofline": {"bound": "hbm", "kernel": "gather_attention", "achieved": gbs,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                         "traffic": None, "peak_source": f"{pk['source']} HBM copy",
                         "note": "achieved counts gathered bytes, most of them L2 hits, so "
                                 "frac can exceed 1; unique HBM bytes are ~1.4 GB per step",
                         "ms_per_launch": kernel_ms},
            "cpu_baseline": None, "e2e": None,
            "gpu_launches": sum(p["launches"] for p in prof.values()),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if str(args.workload) == "gather":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the CPU baseline arm covers the default workload only"}))
            return
        run_gather(args)
        return
    args.workload = int(args.workload)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
