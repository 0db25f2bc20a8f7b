#!/usr/bin/env python3
"""Benchmark of the paged-attention forward pass (libpagedattn) on GB300.

One "step" is one pa_forward call over one batch (the split-KV decode kernel
with its log-sum-exp merge, the persistent prefill kernel: whatever the batch
needs), replayed from CUDA graphs captured with a static launch grid.  The
headline workload is the Llama-3.1-8B-shaped single-stream decode at context
32768 (32 query heads, 8 KV heads, head_dim 128, page 16, bf16 N(0,1), pages
scattered in a pool 1.5x the need); --config picks another.  At N = 1 the same
process also measures every other workload of the metric (single-stream decode
at 1024 and 8192, the 64-sequence batched decode, the causal varlen prefill, the
mixed batch), speculative multi-token decode, the paged KV-cache write of the
prefill's new tokens and a 32-layer full-graph decoder step, each as a record
under "sub_records" with its own timing, kernel roofline and clock summary (and
an end-to-end figure for the attention workloads).

Per workload:
  * timed region: `steps` steps replayed from CUDA graphs, after W untimed
    warm-up steps and a short clock-settling replay; value = algorithmic work
    (KV bytes, or causal FLOPs for the prefill) of all steps on all ranks / the
    max over ranks of the region;
  * kernel roofline: the dominant kernel alone (the other kernel of a mixed
    batch is not launched), in runs of consecutive launches bracketed by CUDA
    events on the launching stream, at least 100 runs; achieved = algorithmic
    bytes (or FLOPs) per launch / mean launch duration; peak = the measured HBM
    copy bandwidth, or for the prefill the sustained bf16 rate (its timing runs
    for a second or more under the power cap);
  * e2e: the same metric through the public API with the step's q and metadata
    in pinned host memory and its out brought back to pinned host memory every
    step: copied in and out (eager calls, captured graphs, a captured pipeline),
    or, for shapes without prefill rows, read and written in place by the decode
    kernel over the host link; the best mode, each timed over at least 0.2 s
    after one untimed replay.
L2: each step reads one of R identical copies of the KV pool in rotation, with
R * (KV bytes per step) > 3 * L2, so no step finds its pages in L2.
Every call passes pa_options.early_metadata (the metadata is the same for every
step, so no kernel before a call writes it): a decode grid launched early reads
its metadata and prefetches its first pages while the previous call finishes;
--no-early-metadata measures without it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
"""

from __future__ import annotations

import argparse
import datetime as dt
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "llama_decode_32768"
SUB_CONFIGS = ["llama_decode_1024", "llama_decode_8192", "llama_decode_32768", "batched_decode", "varlen_prefill",
               "mixed", "spec_decode"]
LAYERS_SUB = ("llama_decode_32768", 32)  # the full-graph decoder step of the sub-records
FALLBACK_HBM_GBS = 6800.0      # profiling recipe's fallback, one earlier GB300 measurement
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_SUSTAINED = 1700.0
CSRC = os.path.join(ROOT, "paged_kv_cache_forward_gb300", "csrc")
KERNEL_SOURCES = {
    "decode_splitkv": ["decode.cu", "pa_device.cuh", "pa_internal.h"],
    "prefill": ["prefill_tc.cu", "tc_device.cuh", "pa_device.cuh", "pa_internal.h"],
}
DESCRIPTIONS = {
    "tiny_decode": "batch 1, 1 query token, Hq 4 / Hkv 1, head_dim 64, context 256, page 16, 16 of 64 pages",
    "llama_decode_1024": "batch 1, Hq 32 / Hkv 8, head_dim 128, page 16, context 1024, pool 1.5x",
    "llama_decode_8192": "batch 1, Hq 32 / Hkv 8, head_dim 128, page 16, context 8192, pool 1.5x",
    "llama_decode_32768": "batch 1, Hq 32 / Hkv 8, head_dim 128, page 16, context 32768, pool 1.5x",
    "batched_decode": "batch 64, Hq 32 / Hkv 8, head_dim 128, page 16, context U[512, 8192], K x0.5",
    "varlen_prefill": "batch 8, Hq 32 / Hkv 8, head_dim 128, causal, new U[128, 2048], prefix U[0, 4096]",
    "mixed": "4 prefill x 512 + 60 decode ctx U[1024, 16384] + 1 decode ctx 131072, Hq 32 / Hkv 8, D 128",
    "spec_decode": "batch 16 x 4 new tokens (speculative decoding), ctx U[2048, 8192], Hq 32 / Hkv 8, D 128",
}
KERNEL_RUN = 16            # consecutive launches per timed run of the dominant kernel (at least)
KERNEL_RUN_MAX = 512
KERNEL_RUN_MS = 3.0        # target length of one timed run
KERNEL_MIN_RUNS = 100
KERNEL_MIN_S = 0.25
E2E_MIN_S = 0.2
SETTLE_MS = 300.0
SM_HZ_NOMINAL = 2.07e9     # converts the pre-region spin to cycles


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 2 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kv-chunk", type=int, default=0, help="override the tuned split size (sweeps)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-early-metadata", action="store_true",
                    help="every call waits for the previous kernel before reading its metadata (pa_options)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-records", action="store_true", help="headline workload only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle leg")
    ap.add_argument("--layers", type=int, default=0,
                    help="model-step mode: L layers, each with its own KV cache, one pa_forward per layer; "
                         "times one CUDA graph of all L layers against L one-layer graphs and eager calls")
    ap.add_argument("--kernel-runs", type=int, default=KERNEL_MIN_RUNS,
                    help="timed runs of the dominant kernel alone (profiling runs use fewer)")
    ap.add_argument("--settle-ms", type=float, default=SETTLE_MS,
                    help="graph replays before the timed region so that clocks settle; 0 for profiling runs")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- multi-rank

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(seed: int, rank: int) -> int:
    """Weak scaling: every rank runs its own independent batch of the same shapes."""
    return seed + 1000 * rank


def reduce_max(value: float, world: int, device=None) -> float:
    """Max over ranks (timing is taken as the slowest rank's)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------- workload

def work_of(batch):
    """Algorithmic work of one step: KV bytes, the decode kernel's bytes, causal FLOPs."""
    D, Hq = batch.head_dim, batch.num_q_heads
    kv = batch.kv_bytes()
    q_bytes = batch.num_tokens * Hq * D * 2
    pages = sum((L + batch.page_size - 1) // batch.page_size for L in batch.seq_lens.tolist())
    flops = 4 * D * Hq * batch.causal_pairs()
    q_lens = batch.q_lens()
    qmax = 16 // (Hq // batch.num_kv_heads) if Hq // batch.num_kv_heads <= 16 else 1  # decode-path tokens
    dec = [(n, L) for n, L in zip(q_lens, batch.seq_lens.tolist()) if 1 <= n <= qmax]
    dec_kv = sum(L for _, L in dec) * 2 * batch.num_kv_heads * D * 2
    dec_tokens = sum(n for n, _ in dec)
    dec_pages = sum((L + batch.page_size - 1) // batch.page_size for _, L in dec)
    return dict(kv_bytes=kv, flops=flops, tokens=batch.num_tokens,
                # K and V of the decode sequences, their q and out rows, 4 B per block-table entry
                decode_bytes=dec_kv + 2 * dec_tokens * Hq * D * 2 + dec_pages * 4,
                algorithmic_bytes=kv + 2 * q_bytes + pages * 4)


def metric_of(config: str):
    if config == "varlen_prefill":
        return "prefill attention TFLOP/s", "TFLOP/s", "tensor"
    return "decode KV GB/s", "GB/s", "hbm"


def value_of(config, work, seconds_per_step):
    if config == "varlen_prefill":
        return work["flops"] / seconds_per_step / 1e12
    return work["kv_bytes"] / seconds_per_step / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except (OSError, ValueError):
        j = {}
    hbm = j.get("hbm_gbs")
    bf16 = j.get("bf16_tflops")
    bf16s = j.get("bf16_tflops_sustained")
    return dict(
        hbm=(float(hbm), "measured") if hbm else (FALLBACK_HBM_GBS, "fallback"),
        bf16=(float(bf16), "measured") if bf16 else (FALLBACK_BF16_TFLOPS, "fallback"),
        bf16_sustained=(float(bf16s), "measured") if bf16s else (FALLBACK_BF16_SUSTAINED, "fallback"),
    )


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, config: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source
    is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{config}.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    kv = {}
    for ln in lines:
        if ":" in ln and ln.strip().startswith(("traffic_bytes_per_launch", "kernel_source_sha256")):
            k, v = ln.strip().split(":", 1)
            kv[k.strip()] = v.strip().strip("`")
    if kv.get("kernel_source_sha256") != source_hash(kernel):
        return None
    try:
        return float(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def stats_ms(xs):
    qs = statistics.quantiles(xs, n=10) if len(xs) >= 2 else [xs[0]] * 9
    return {"mean": statistics.mean(xs), "median": statistics.median(xs), "p10": qs[0], "p90": qs[-1],
            "n": len(xs)}


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling (200 ms) running across the warm-up and timed phases."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float, what: str):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        rows = []
        for ln in open(self.path).read().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        note = f"samples inside {what}"
        if not inside:
            inside = rows[-3:]
            note = f"{what} shorter than the sampling period; last samples of the loaded run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "no samples"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3][i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "note": note}


# ------------------------------------------------------------- CPU baseline

def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def _oracle_rate(batch, config, target_s: float, threads: int):
    """Seconds per whole step of the oracle on `threads` host threads (0: all),
    from a bounded sample of (token, head) rows spread over the batch."""
    import oracle
    Hq = batch.num_q_heads
    total_rows = batch.num_tokens * Hq
    rows = [(t, h) for t in range(batch.num_tokens) for h in range(Hq)]
    n = len(rows)
    probe = rows[:: max(1, n // 64)][:64]
    t = time.perf_counter()
    oracle.batch_attention(batch, rows=probe, threads=threads)
    per_row = (time.perf_counter() - t) / len(probe)
    want = max(1, int(target_s / max(per_row, 1e-9)))
    if want >= n:
        sample = rows
        reps = max(1, int(target_s / max(per_row * n, 1e-9)))
    else:
        sample = rows[:: max(1, n // want)][:want]
        reps = 1
    t = time.perf_counter()
    for _ in range(reps):
        oracle.batch_attention(batch, rows=sample, threads=threads)
    elapsed = time.perf_counter() - t
    frac = len(sample) * reps / total_rows
    return elapsed / frac, f"{len(sample)} of {total_rows} (token, head) rows x {reps} repetition(s), " \
                           f"{elapsed:.1f} s; step time scaled by the row fraction"


def cpu_baseline(batch, config, target_s: float):
    """The fp64 oracle, as it stands, on this host's cores (all of them, and one),
    on bounded samples of the workload."""
    import oracle
    work = work_of(batch)
    _, unit, _ = metric_of(config)
    step_s, sample = _oracle_rate(batch, config, target_s, 0)
    step1_s, sample1 = _oracle_rate(batch, config, max(1.0, target_s / 3), 1)
    return {"value": value_of(config, work, step_s), "unit": unit, "cores": oracle.max_threads(),
            "kind": "oracle", "sample": sample, "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "single_thread": {"value": value_of(config, work, step1_s), "unit": unit, "threads": 1,
                              "sample": sample1}}


def run_reference(args):
    """--impl reference: the fp64 CPU oracle timed as the reference arm."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    import oracle
    from paged_kv_cache_forward_gb300 import workloads as W
    torch.manual_seed(0)
    batch = W.CONFIGS[args.config](seed=args.seed)
    metric, unit, _ = metric_of(args.config)
    steps = args.steps or 3
    warm = max(0, min(args.warmup, 1))
    budget = min(120.0 / max(1, steps + warm), args.cpu_seconds)
    for _ in range(warm):
        _oracle_rate(batch, args.config, min(budget, 5.0), 0)
    runs = [_oracle_rate(batch, args.config, budget, 0) for _ in range(steps)]
    step_s = statistics.median(r[0] for r in runs)
    v = value_of(args.config, work_of(batch), step_s)
    line = {
        "impl": "reference", "metric": metric, "value": v, "unit": unit, "n_gpus": args.gpus, "steps": steps,
        "warmup": warm, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.config}: {DESCRIPTIONS.get(args.config, '')}", "seed": args.seed},
        "cpu_baseline": {"value": v, "unit": unit, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": runs[0][1], "cpu_model": cpu_model(), "nproc": os.cpu_count()},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------- ours

class Workload:
    """One workload on the device: the batch, R rotating KV pool copies, the
    output, a stream, the launch plan and the forward call."""

    def __init__(self, config, seed, dev, kv_chunk=0, early=1):
        import torch
        import paged_kv_cache_forward_gb300 as pa
        from paged_kv_cache_forward_gb300 import workloads as W
        self.pa, self.torch, self.config, self.dev, self.kv_chunk = pa, torch, config, dev, kv_chunk
        self.early = early  # pa_options.early_metadata: the metadata is the same for every call
        self.batch = W.CONFIGS[config](seed=seed)
        self.work = work_of(self.batch)
        props = torch.cuda.get_device_properties(dev)
        self.l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
        per_step = max(self.work["kv_bytes"], 1)
        self.R = 1 if per_step > 3 * self.l2 else int(math.ceil(3 * self.l2 / per_step)) + 1
        d = self.batch.to(dev)
        self.d = d
        self.ks = [d.k_cache] + [d.k_cache.clone() for _ in range(self.R - 1)]
        self.vs = [d.v_cache] + [d.v_cache.clone() for _ in range(self.R - 1)]
        self.out = torch.empty_like(d.q)
        self.stream = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize(dev)  # inputs and pool copies were made on the default stream
        self.plan = pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens, kv_chunk=kv_chunk)
        pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, kv_chunk=kv_chunk, stream=self.stream)
        b = self.batch
        G = b.num_q_heads // b.num_kv_heads
        qmax = 16 // G if G <= 16 else 1
        has_decode = any(1 <= n <= qmax for n in b.q_lens())
        self.dominant = "prefill" if (config == "varlen_prefill" or not has_decode) else "decode_splitkv"

    def call(self, i, events=None, launch_only=0, out=None):
        d = self.d
        self.pa.forward(d.q, self.ks[i % self.R], self.vs[i % self.R], d.block_table, d.seq_lens, d.query_start_loc,
                        self.out if out is None else out, scale=self.batch.scale, kv_chunk=self.kv_chunk,
                        events=events, stream=self.stream, launch_only=launch_only, early_metadata=self.early)

    def graph(self, n, fn):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=self.stream):
            for i in range(n):
                fn(i)
        return g


def timing_events(external: bool):
    """A pair of timing events; external ones are recorded as nodes of a graph
    captured around them (None, None if this torch has no external events)."""
    import torch
    if not external:
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    except TypeError:
        return None, None


def time_kernel(wl, world, est_ms, min_runs=KERNEL_MIN_RUNS):
    """Mean, median, p10, p90 launch duration (ms) of the dominant kernel alone:
    a graph of KERNEL_RUN consecutive launches (the pool copies in rotation)
    bracketed by CUDA events recorded on the launching stream, replayed at least
    KERNEL_MIN_RUNS times and for at least KERNEL_MIN_S."""
    torch = wl.torch
    key = "prefill" if wl.dominant == "prefill" else "decode"
    only = (2 if key == "prefill" else 1) if wl.plan["launches"] > 1 else 0
    # a run lasts a few milliseconds (16 to 512 launches): the two event nodes
    # and the graph's own start cost stay small against it
    want = int(min(KERNEL_RUN_MAX, max(KERNEL_RUN, math.ceil(KERNEL_RUN_MS / max(est_ms, 1e-3)))))
    run = max(wl.R, want // wl.R * wl.R)
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # torch creates the CUDA event on its first record(); do that outside the
    # capture so that the library receives real handles to re-record.
    e_a.record(wl.stream)
    e_b.record(wl.stream)
    wl.stream.synchronize()

    def launch(i):
        ev = {}
        if i == 0:
            ev[f"{key}_start_event"] = e_a
        if i == run - 1:
            ev[f"{key}_stop_event"] = e_b
        wl.call(i, events=ev, launch_only=only)

    g = wl.graph(run, launch)
    with torch.cuda.stream(wl.stream):  # a graph replays on the current stream
        g.replay()
    wl.stream.synchronize()
    first = e_a.elapsed_time(e_b) / run
    n_runs = max(min_runs, int(math.ceil(KERNEL_MIN_S / max(first * run / 1e3, 1e-6)))) if min_runs >= \
        KERNEL_MIN_RUNS else max(1, min_runs)
    per = []
    for _ in range(n_runs):
        # two replays back to back: the events keep the second one's times, a
        # run that starts while the GPU is busy (not after an idle gap)
        with torch.cuda.stream(wl.stream):
            g.replay()
            g.replay()
        wl.stream.synchronize()
        per.append(e_a.elapsed_time(e_b) / run)
    del g
    per_max = reduce_max(statistics.mean(per), world, wl.dev)
    st = stats_ms(per)
    st["mean_max_over_ranks"] = per_max
    st["how"] = (f"{'only the ' + key + ' kernel launched' if only else 'the whole step is this kernel'}; "
                 f"CUDA events around runs of {run} consecutive launches, {n_runs} runs, each the second of two "
                 f"back-to-back replays")
    return st


def time_e2e(wl, world, est_ms):
    """The metric through the public API with host buffers: every step brings its
    q and metadata in from pinned host memory and its out back to pinned host
    memory.  Best of eager calls and captured graphs of 64 steps that copy (one
    packed copy in, one out), a captured pipeline whose copies overlap the
    neighbouring steps' forwards, and (shapes without prefill rows) captured
    steps whose decode kernel reads and writes the pinned host buffers in place;
    each mode timed over at least E2E_MIN_S after one untimed pass."""
    torch, pa, b, dev, stream = wl.torch, wl.pa, wl.batch, wl.dev, wl.stream
    parts = [b.q, b.block_table, b.seq_lens, b.query_start_loc]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 15) // 16 * 16
    hbuf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, k):
        t = parts[k]
        return buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for k, t in enumerate(parts):
        view(hbuf, k).copy_(t)
    eq, ebt, esl, eqsl = (view(dbuf, k) for k in range(4))
    out = wl.out
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    R, ks, vs = wl.R, wl.ks, wl.vs
    Me = 64
    n_e2e = max(Me, int(math.ceil(E2E_MIN_S / max(est_ms / 1e3, 1e-7) / Me)) * Me)

    def e2e_step(i):
        dbuf.copy_(hbuf, non_blocking=True)
        pa.forward(eq, ks[i % R], vs[i % R], ebt, esl, eqsl, out, scale=b.scale, kv_chunk=wl.kv_chunk, stream=stream,
                   early_metadata=wl.early)
        hout.copy_(out, non_blocking=True)

    def timed(fn, reps):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        barrier(world)
        with torch.cuda.stream(stream):
            a0.record()
            for r in range(reps):
                fn(r)
            a1.record()
        stream.synchronize()
        barrier(world)
        return a0.elapsed_time(a1)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    # (a) eager: copies and pa_forward launched from the host every step
    eager_ms = reduce_max(timed(e2e_step, n_e2e), world, dev) / n_e2e
    # (b) the same steps captured in CUDA graphs of Me steps, replayed: what a
    # serving loop that captures its decode step sees
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        for i in range(Me):
            e2e_step(i)
    reps = n_e2e // Me
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        ge.replay()
    graph_ms = reduce_max(timed(lambda r: ge.replay(), reps), world, dev) / (reps * Me)
    del ge
    # (c) the same steps pipelined inside a CUDA graph: inputs copied in on one
    # side stream, results copied out on another, two alternating input arenas
    # and output buffers; step i+1's input copy and step i-1's output copy
    # overlap step i's forward.  Every step still copies its own inputs in and
    # its own result out.
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dbufs = [dbuf, torch.empty_like(dbuf)]
    outs2 = [out, torch.empty_like(out)]
    houts = [hout, torch.empty(out.shape, dtype=out.dtype, pin_memory=True)]
    arenas = [[view(db, k) for k in range(4)] for db in dbufs]
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=stream):
        ev_fwd = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        ev_start = torch.cuda.Event()
        ev_start.record(stream)
        cs_in.wait_event(ev_start)
        cs_out.wait_event(ev_start)
        for i in range(Me):
            k = i & 1
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(cs_in):
                if i >= 2:
                    cs_in.wait_event(ev_fwd[k])  # forward(i-2) has read arena k
                dbufs[k].copy_(hbuf, non_blocking=True)
                ev_in.record(cs_in)
            stream.wait_event(ev_in)
            if i >= 2:
                stream.wait_event(ev_out[k])  # out k copied out by step i-2
            qv, btv, slv, qslv = arenas[k]
            pa.forward(qv, ks[i % R], vs[i % R], btv, slv, qslv, outs2[k], scale=b.scale,
                       kv_chunk=wl.kv_chunk, stream=stream, early_metadata=wl.early)
            ev_fwd[k] = torch.cuda.Event()
            ev_fwd[k].record(stream)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(ev_fwd[k])
                houts[k].copy_(outs2[k], non_blocking=True)
                ev_out[k] = torch.cuda.Event()
                ev_out[k].record(cs_out)
        ev_end_in, ev_end_out = torch.cuda.Event(), torch.cuda.Event()
        ev_end_in.record(cs_in)
        ev_end_out.record(cs_out)
        stream.wait_event(ev_end_in)
        stream.wait_event(ev_end_out)
    with torch.cuda.stream(stream):
        gp.replay()
    pipe_ms = reduce_max(timed(lambda r: gp.replay(), reps), world, dev) / (reps * Me)
    del gp
    # (d) shapes without prefill rows: q, the metadata and out stay in pinned host
    # memory, which the decode kernel reads and writes in place over the host
    # link (pa_forward's pointer rules), so a step launches no copies; two
    # alternating input arenas and output buffers, captured like (b).
    zc_ms = None
    if pa.plan_for(b.q, b.k_cache, b.block_table, b.seq_lens, kv_chunk=wl.kv_chunk)["prefill_ctas"] == 0:
        hbufs = [hbuf, torch.empty(total, dtype=torch.uint8, pin_memory=True)]
        hbufs[1].copy_(hbuf)
        harenas = [[view(hb, k) for k in range(4)] for hb in hbufs]
        gz = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gz, stream=stream):
            for i in range(Me):
                qv, btv, slv, qslv = harenas[i & 1]
                pa.forward(qv, ks[i % R], vs[i % R], btv, slv, qslv, houts[i & 1], scale=b.scale,
                           kv_chunk=wl.kv_chunk, stream=stream, early_metadata=wl.early)
        with torch.cuda.stream(stream):
            gz.replay()
        zc_ms = reduce_max(timed(lambda r: gz.replay(), reps), world, dev) / (reps * Me)
        del gz
    h2d = sum(t.numel() * t.element_size() for t in parts)
    what = ("per step: q and metadata copied (one packed copy) from pinned host memory, pa_forward, out "
            "copied to pinned host memory, serial on one stream; KV cache resident")
    modes = {
        "graph_pipelined": (pipe_ms, "per step: q and metadata copied (one packed copy) from pinned host memory "
                                     "on a side stream, pa_forward, out copied to pinned host memory on a second "
                                     "side stream, two alternating input/output buffers so that neighbouring "
                                     f"steps' copies overlap the forward; captured in CUDA graphs of {Me} steps; "
                                     "KV cache resident"),
        "graph": (graph_ms, what + f"; steps captured in CUDA graphs of {Me} and replayed"),
        "eager": (eager_ms, what + "; launched eagerly from the host"),
    }
    if zc_ms is not None:
        modes["graph_host_buffers"] = (
            zc_ms, "per step: pa_forward reads q and the metadata from pinned host memory and writes out to "
                   "pinned host memory in place (over NVLink-C2C; no copy launches), two alternating host "
                   f"input/output buffers; captured in CUDA graphs of {Me} steps; KV cache resident")
    best = min(modes, key=lambda m: modes[m][0])
    return {"ms_per_step": modes[best][0], "steps": n_e2e, "mode": best + ": " + modes[best][1],
            "modes_ms_per_step": {m: v[0] for m, v in modes.items()},
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hout.numel() * hout.element_size()}


def measure(config, args, dev, rank, world, local, steps=None, warmup=None, with_e2e=True, region_s=2.0):
    """One workload's record: timed region, kernel roofline, e2e, clocks."""
    import torch
    torch.cuda.synchronize(dev)
    wl = Workload(config, rank_seed(args.seed, rank), dev, args.kv_chunk, early=0 if args.no_early_metadata else 1)
    work, pa, stream = wl.work, wl.pa, wl.stream
    metric, unit, _ = metric_of(config)
    W_req = args.warmup if warmup is None else warmup

    # W untimed warm-up steps (the first also loads the kernels)
    with torch.cuda.stream(stream):
        for i in range(max(1, W_req)):
            wl.call(i)
    stream.synchronize()
    assert pa.device_error(stream) == 0

    # one eager step's time sizes the default step count and the e2e phase
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for i in range(10):
            wl.call(i)
        e1.record()
    stream.synchronize()
    est_ms = e0.elapsed_time(e1) / 10
    if steps is None:
        steps = int(min(200000, max(200, region_s * 1e3 / max(est_ms, 1e-3))))

    # graphs of M consecutive steps, rotating over the R pool copies
    R = wl.R
    M = min(steps, max(R, 256))
    M = max(R, (M // R) * R) if M >= R else M
    full, rem = divmod(steps, M)
    g_main = wl.graph(M, wl.call)
    g_rem = wl.graph(rem, wl.call) if rem else None

    sampler = ClockSampler(local).start()
    t_load0 = time.time()
    # clock settling: graph replays for about args.settle_ms (not counted as warm-up)
    settle_reps = int(math.ceil(args.settle_ms / max(est_ms * M, 1e-3))) if args.settle_ms > 0 else 0
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        for _ in range(settle_reps):
            g_main.replay()
    stream.synchronize()

    # When the K steps fit one graph, the region's two events are recorded by
    # nodes of that graph, first and last, so the region holds exactly the K
    # steps (not the graph's launch latency); otherwise they bracket the replays.
    start, stop = timing_events(external=True)
    g_timed = None
    if full == 1 and g_rem is None and start is not None:
        # (torch creates the CUDA event on its first record: outside the capture)
        start.record(stream)
        stop.record(stream)
        stream.synchronize()

        def timed_steps(i):
            if i == 0:
                start.record(stream)
            wl.call(i)
            if i == M - 1:
                stop.record(stream)
        g_timed = wl.graph(M, timed_steps)
    else:
        start, stop = timing_events(external=False)
    barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        if g_timed is not None:
            # The GPU is kept busy up to the graph's first node (a ~30 us spin,
            # outside the region), as it is in a serving loop, rather than
            # starting the K steps from idle.
            torch.cuda._sleep(int(30e-6 * SM_HZ_NOMINAL))
            g_timed.replay()
        else:
            start.record()
            for _ in range(full):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            stop.record()
    stream.synchronize()
    torch.cuda.synchronize(dev)
    barrier(world)
    region_ms = start.elapsed_time(stop)
    assert pa.device_error(stream) == 0
    region_how = ("CUDA events recorded by the first and last nodes of one graph of the K steps" if g_timed is not None
                  else f"CUDA events around {full} replay(s) of a {M}-step graph" + (" and one of the rest" if rem else ""))
    del g_main, g_rem, g_timed

    kern = time_kernel(wl, world, est_ms, args.kernel_runs)
    t_load1 = time.time()
    sampler.stop()
    assert pa.device_error(stream) == 0

    region_ms_max = reduce_max(region_ms, world, dev)
    ms_per_step = region_ms_max / steps
    total_kv = reduce_sum(work["kv_bytes"], world, dev)
    total_flops = reduce_sum(work["flops"], world, dev)
    total_tokens = reduce_sum(work["tokens"], world, dev)
    value = value_of(config, {"kv_bytes": total_kv, "flops": total_flops}, region_ms_max / 1e3 / steps)

    peaks = measured_peaks()
    k_ms = kern["mean"]
    if wl.dominant == "prefill":
        # The prefill kernel is timed over a second or more of back-to-back
        # launches, under the power cap: the sustained bf16 rate is its peak.
        peak, src = peaks["bf16_sustained"]
        achieved = work["flops"] / (k_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{src} (sustained bf16)", "frac_of_burst_peak": achieved / peaks["bf16"][0]}
        per_launch = work["flops"]
    else:
        peak, src = peaks["hbm"]
        achieved = work["decode_bytes"] / (k_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{src} (copy bandwidth)"}
        per_launch = work["decode_bytes"]
    roof.update({"traffic": committed_traffic(wl.dominant, config), "kernel": wl.dominant,
                 "kernel_ms_mean": k_ms, "kernel_ms_median": kern["median"], "kernel_ms_p10": kern["p10"],
                 "kernel_ms_p90": kern["p90"], "kernel_runs": kern["n"], "kernel_timing": kern["how"],
                 "algorithmic_per_launch": per_launch})

    hbm_frac = (total_kv / world) / (ms_per_step / 1e3) / 1e9 / peaks["hbm"][0]
    # (the timed regions last half a second or more: the sustained bf16 rate)
    tensor_frac = (total_flops / world) / (ms_per_step / 1e3) / 1e12 / peaks["bf16_sustained"][0]

    e2e = None
    if with_e2e and not args.no_e2e:
        e = time_e2e(wl, world, est_ms)
        e2e = {"value": value_of(config, {"kv_bytes": total_kv, "flops": total_flops}, e["ms_per_step"] / 1e3),
               "unit": unit, **e}
    assert pa.device_error(stream) == 0

    rec = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": steps, "warmup": W_req,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{config}: {DESCRIPTIONS.get(config, '')}",
            "seed": args.seed, "global_batch": wl.batch.num_seqs * world, "tokens_per_step": int(total_tokens),
            "kv_bytes_per_step": int(total_kv), "causal_flops_per_step": int(total_flops),
            "l2": (f"inputs rotate over {R} KV pool copies ({R} x {work['kv_bytes'] / 2**20:.0f} MiB "
                   f"> 3 x L2 {wl.l2 / 2**20:.0f} MiB)") if R > 1 else "KV bytes per step > 3 x L2",
            "graph": f"CUDA graphs of {M} steps", "timed_region": region_how,
            "settle_ms": round(settle_reps * M * est_ms, 1),
            "kv_chunk": wl.plan["kv_chunk"], "splits": wl.plan["splits"],
            "decode_variant": f"{wl.plan['decode_warps']} warps x {wl.plan['decode_stages']} stages, "
                              f"cluster {wl.plan['decode_cluster']}",
            "early_metadata": bool(wl.early),
            "parallelism": f"dp{world}" if world > 1 else "single GPU",
        },
        "tok_s": total_tokens * steps / (region_ms_max / 1e3),
        # one attention layer per step; a 32-layer model's attention alone could
        # run at most this many tokens/s
        "tok_s_32_layer_attention_ceiling": total_tokens * steps / (region_ms_max / 1e3) / 32,
        # whole step against each roofline: KV bytes / HBM, causal FLOPs / bf16
        # tensor peak, and the binding one, max(B / BW, F / peak) / t
        "hbm_frac_step": hbm_frac,
        "tensor_frac_step": tensor_frac,
        "roofline_frac_step": max(hbm_frac, tensor_frac),
        "roofline": roof,
        "peaks": {"hbm_gbs": peaks["hbm"][0], "bf16_tflops": peaks["bf16"][0],
                  "bf16_tflops_sustained": peaks["bf16_sustained"][0], "source": peaks["hbm"][1]},
        "e2e": e2e,
        "gpu_launches": wl.plan["launches"] * steps,
        "clocks": sampler.summary(t_load0, t_load1, "the settle, timed and kernel-timing phases"),
    }
    batch = wl.batch
    del wl
    torch.cuda.empty_cache()
    return rec, batch


def measure_layers(config, L, args, dev, rank, world, local, steps=50):
    """A decoder step of L attention layers, every layer with its own paged KV
    cache, queries and output, one pa_forward per layer: one CUDA graph of the
    whole step against L one-layer graphs replayed back to back and L eager
    calls.  Also checks that the one-graph step gives the eager outputs."""
    import torch
    import paged_kv_cache_forward_gb300 as pa
    from paged_kv_cache_forward_gb300 import workloads as W
    batch = W.CONFIGS[config](seed=rank_seed(args.seed, rank))
    work = work_of(batch)
    pool_bytes = 2 * batch.k_cache.numel() * batch.k_cache.element_size()
    if L * pool_bytes > (96 << 30):
        raise SystemExit(f"{L} layers x {pool_bytes / 2**30:.1f} GiB of KV pool exceed 96 GiB")
    d = batch.to(dev)
    gen = torch.Generator(device=dev).manual_seed(rank_seed(args.seed, rank) + 1)
    ks = [d.k_cache] + [torch.randn(d.k_cache.shape, generator=gen, device=dev).to(torch.bfloat16)
                        for _ in range(L - 1)]
    vs = [d.v_cache] + [torch.randn(d.v_cache.shape, generator=gen, device=dev).to(torch.bfloat16)
                        for _ in range(L - 1)]
    qs = [d.q] + [torch.randn(d.q.shape, generator=gen, device=dev).to(torch.bfloat16) for _ in range(L - 1)]
    outs = [torch.empty_like(d.q) for _ in range(L)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)  # inputs and caches were made on the default stream
    plan = pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens, kv_chunk=args.kv_chunk)
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, kv_chunk=args.kv_chunk, stream=stream)

    def layer(i):
        pa.forward(qs[i], ks[i], vs[i], d.block_table, d.seq_lens, d.query_start_loc, outs[i],
                   scale=batch.scale, kv_chunk=args.kv_chunk, stream=stream,
                   early_metadata=0 if args.no_early_metadata else 1)

    def model_step():
        for i in range(L):
            layer(i)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            model_step()
    stream.synchronize()
    assert pa.device_error(stream) == 0
    g_full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full, stream=stream):
        model_step()
    g_layers = []
    for i in range(L):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer(i)
        g_layers.append(g)
    modes = {
        "graph_full": lambda: g_full.replay(),
        "graph_per_layer": lambda: [g.replay() for g in g_layers],
        "eager": model_step,
    }
    sampler = ClockSampler(local).start()
    times = {}
    t0 = time.time()
    for name, fn in modes.items():
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                fn()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            a.record()
            for _ in range(steps):
                fn()
            b.record()
        stream.synchronize()
        torch.cuda.synchronize(dev)
        barrier(world)
        times[name] = reduce_max(a.elapsed_time(b), world, dev) / steps
    t1 = time.time()
    sampler.stop()
    assert pa.device_error(stream) == 0
    ref = [o.clone() for o in outs]
    with torch.cuda.stream(stream):
        g_full.replay()
    stream.synchronize()
    identical = all(torch.equal(a, b) for a, b in zip(ref, outs))
    total_kv = reduce_sum(work["kv_bytes"], world, dev) * L
    total_flops = reduce_sum(work["flops"], world, dev) * L
    ms = times["graph_full"]
    metric, unit, _ = metric_of(config)
    peaks = measured_peaks()
    rec = {
        "metric": metric, "value": value_of(config, {"kv_bytes": total_kv, "flops": total_flops}, ms / 1e3),
        "unit": unit, "n_gpus": world, "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{L} layers x {config}: {DESCRIPTIONS.get(config, '')}",
            "layers": L, "kv_bytes_per_step": int(total_kv), "kv_chunk": plan["kv_chunk"],
            "splits": plan["splits"], "early_metadata": not args.no_early_metadata,
            "l2": f"KV bytes per step {total_kv / 2**20:.0f} MiB (> 3 x L2)" if total_kv > 3 * (128 << 20)
            else f"KV bytes per step {total_kv / 2**20:.0f} MiB (<= 3 x L2)",
            "parallelism": f"dp{world}" if world > 1 else "single GPU",
        },
        "graph_modes_ms_per_step": times,
        "launch_overhead_us_per_layer": {
            k: (v - times["graph_full"]) * 1e3 / L for k, v in times.items() if k != "graph_full"},
        "us_per_layer": ms * 1e3 / L,
        "hbm_frac_step": (total_kv / world) / (ms / 1e3) / 1e9 / peaks["hbm"][0],
        "graph_matches_eager": identical,
        "gpu_launches": plan["launches"] * L * steps,
        "clocks": sampler.summary(t0, t1, "the timed modes"),
    }
    del g_full, g_layers, ks, vs, qs, outs
    torch.cuda.empty_cache()
    return rec, identical


def measure_cache_write(args, dev, rank, world, local, steps=None):
    """The paged KV-cache write (pa_cache_write) of the varlen prefill's new
    tokens (Llama shape: 8 KV heads, head_dim 128): each token's K and V rows
    scattered to its page slot, 16 consecutive tokens to a page, pages drawn at
    random from a pool.  Algorithmic bytes per launch = read and write of K and V
    (4 x tokens x 2 KiB) + the 8-byte slot of every token; rotating over R sets of
    buffers larger than 3 x L2 together."""
    import torch
    import paged_kv_cache_forward_gb300 as pa
    from paged_kv_cache_forward_gb300 import workloads as W
    b = W.varlen_prefill(seed=rank_seed(args.seed, rank))
    T, Hkv, D, P = b.num_tokens, b.num_kv_heads, b.head_dim, b.page_size
    row = Hkv * D * 2
    nbytes = 4 * T * row + 8 * T
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    R = 1 if nbytes > 3 * l2 else int(math.ceil(3 * l2 / nbytes)) + 1
    gen = torch.Generator(device=dev).manual_seed(rank_seed(args.seed, rank) + 7)
    pages = (T + P - 1) // P + 1
    sets = []
    for _ in range(R):
        perm = torch.randperm(pages, device=dev, generator=gen)
        t = torch.arange(T, device=dev)
        slots = (perm[t // P] * P + t % P).to(torch.int64)
        sets.append((torch.randn(T, Hkv, D, device=dev, generator=gen).to(torch.bfloat16),
                     torch.randn(T, Hkv, D, device=dev, generator=gen).to(torch.bfloat16), slots,
                     torch.zeros(pages, P, Hkv, D, device=dev, dtype=torch.bfloat16),
                     torch.zeros(pages, P, Hkv, D, device=dev, dtype=torch.bfloat16)))
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)

    def call(i):
        kn, vn, sl, kc, vc = sets[i % R]
        pa.cache_write(kn, vn, sl, kc, vc, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(1, args.warmup)):
            call(i)
    stream.synchronize()
    assert pa.device_error(stream) == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for i in range(10):
            call(i)
        e1.record()
    stream.synchronize()
    est_ms = e0.elapsed_time(e1) / 10
    steps = steps or max(R, int(min(256, max(16, 0.05e3 / max(est_ms, 1e-3)))) // R * R)
    start, stop = timing_events(external=True)
    external = start is not None
    if not external:
        start, stop = timing_events(external=False)
    start.record(stream)
    stop.record(stream)
    stream.synchronize()

    def steps_fn(i):
        if external and i == 0:
            start.record(stream)
        call(i)
        if external and i == steps - 1:
            stop.record(stream)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            steps_fn(i)
    sampler = ClockSampler(local).start()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for _ in range(int(math.ceil(args.settle_ms / max(est_ms * steps, 1e-3)))):
            g.replay()
    stream.synchronize()
    times = []
    for _ in range(20):
        barrier(world)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(30e-6 * SM_HZ_NOMINAL))
            if not external:
                start.record()
            g.replay()
            if not external:
                stop.record()
        stream.synchronize()
        times.append(reduce_max(start.elapsed_time(stop), world, dev) / steps)
    t1 = time.time()
    sampler.stop()
    assert pa.device_error(stream) == 0
    st = stats_ms(times)
    peak, src = measured_peaks()["hbm"]
    total = reduce_sum(nbytes, world, dev)
    achieved = nbytes / (st["mean"] / 1e3) / 1e9
    rec = {
        "metric": "paged KV-cache write GB/s", "value": total / (st["median"] / 1e3) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": st["median"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"cache write of the varlen prefill's {T} new tokens, Hkv {Hkv}, D {D}, page {P}",
                   "bytes_per_step": nbytes,
                   "l2": f"rotating over {R} buffer sets ({R} x {nbytes / 2**20:.0f} MiB > 3 x L2)" if R > 1
                   else "bytes per step > 3 x L2",
                   "timed_region": f"median of 20 replays of one {steps}-step graph, events as its first and last "
                                   "nodes" if external else f"median of 20 replays of one {steps}-step graph"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{src} (copy bandwidth)", "kernel": "cache_write", "kernel_ms_mean": st["mean"],
                     "kernel_ms_median": st["median"], "kernel_ms_p10": st["p10"], "kernel_ms_p90": st["p90"],
                     "algorithmic_per_launch": nbytes, "traffic": None},
        "gpu_launches": steps * 20,
        "clocks": sampler.summary(t0, t1, "the timed replays"),
    }
    del sets, g
    torch.cuda.empty_cache()
    return rec


def _brief(rec):
    """The figures of a sub-record that a reader compares across workloads."""
    keep = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "hbm_frac_step", "tensor_frac_step",
            "roofline_frac_step", "tok_s", "roofline", "e2e", "gpu_launches", "clocks", "config", "graph_modes_ms_per_step",
            "launch_overhead_us_per_layer", "us_per_layer", "graph_matches_eager")
    out = {k: rec[k] for k in keep if k in rec}
    if out.get("e2e"):
        out["e2e"] = {k: v for k, v in out["e2e"].items() if k != "mode"}
    return out


def run_ours(args):
    import torch
    import paged_kv_cache_forward_gb300 as pa
    from paged_kv_cache_forward_gb300 import build as build_mod

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_mod.build()
    pa.load()

    line, batch = measure(args.config, args, dev, rank, world, local, steps=args.steps)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(batch, args.config, args.cpu_seconds)
    del batch
    line["cpu_baseline"] = cpu

    ok = True
    if world == 1 and not args.no_sub_records:
        subs = {}
        for cfg in SUB_CONFIGS:
            if cfg == args.config:
                continue
            rec, _ = measure(cfg, args, dev, rank, world, local, warmup=args.warmup, region_s=0.5)
            subs[cfg] = _brief(rec)
        subs["cache_write"] = _brief(measure_cache_write(args, dev, rank, world, local))
        cfg, L = LAYERS_SUB
        rec, identical = measure_layers(cfg, L, args, dev, rank, world, local)
        ok = ok and identical
        subs[f"layers{L}_{cfg}"] = _brief(rec)
        line["sub_records"] = subs
        line["gpu_launches_sub_records"] = sum(r["gpu_launches"] for r in subs.values())
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0 if ok else 1


def run_layers(args):
    """--layers L: the L-layer decoder step of --config as the JSON line."""
    import torch
    import paged_kv_cache_forward_gb300 as pa
    from paged_kv_cache_forward_gb300 import build as build_mod

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_mod.build()
    pa.load()
    rec, identical = measure_layers(args.config, args.layers, args, dev, rank, world, local, steps=args.steps or 50)
    if rank == 0:
        print(json.dumps(rec))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0 if identical else 1


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.layers:
        return run_layers(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
