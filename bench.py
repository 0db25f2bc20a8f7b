#!/usr/bin/env python3
"""Benchmark of the paged-attention forward pass (libpagedattn) on GB300.

One "step" is one pa_forward call over one batch (the split-KV decode kernel
with its log-sum-exp merge, the persistent prefill kernel: whatever the batch
needs), replayed from CUDA graphs captured with a static launch grid.  The default workload is the
Llama-3.1-8B-shaped single-stream decode at context 32768 (32 query heads,
8 KV heads, head_dim 128, page 16, bf16 N(0,1), pages scattered in a pool 1.5x
the need).  Other workloads: --config (see paged_kv_cache_forward_gb300.workloads).

L2: each step reads one of R identical copies of the KV pool in rotation, with
R * (KV bytes per step) > 3 * L2, so no step finds its pages in L2.

Prints one JSON line.  value = algorithmic KV bytes (or causal FLOPs for
prefill) of all steps on all ranks / the max over ranks of the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
"""

from __future__ import annotations

import argparse
import datetime as dt
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "llama_decode_32768"
FALLBACK_HBM_GBS = 6800.0      # profiling recipe's fallback, one earlier GB300 measurement
FALLBACK_BF16_TFLOPS = 1900.0
CSRC = os.path.join(ROOT, "paged_kv_cache_forward_gb300", "csrc")
KERNEL_SOURCES = {
    "decode_splitkv": ["decode.cu", "pa_device.cuh"],
    "prefill": ["prefill_tc.cu", "tc_device.cuh", "pa_device.cuh"],
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


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 2 s of work)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kv-chunk", type=int, default=0, help="override the tuned split size (sweeps)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle leg")
    ap.add_argument("--layers", type=int, default=0,
                    help="model-step mode: L layers, each with its own KV cache, one pa_forward per layer; "
                         "times one CUDA graph of all L layers against L one-layer graphs and eager calls")
    ap.add_argument("--min-warm-ms", type=float, default=500.0,
                    help="graph warm-up time before the timed region (clocks settle); 0 for profiling runs")
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
    dec_kv = sum(L for n, L in zip(q_lens, batch.seq_lens.tolist()) if 1 <= n <= qmax) * 2 * batch.num_kv_heads * D * 2
    dec_tokens = sum(n for n in q_lens if 1 <= n <= qmax)
    return dict(kv_bytes=kv, flops=flops, tokens=batch.num_tokens,
                decode_bytes=dec_kv + dec_tokens * Hq * D * 2 + pages * 4,
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
        bf16_sustained=(float(bf16s), "measured") if bf16s else (1700.0, "fallback"),
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


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling (200 ms) running across the warm-up and timed region."""

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

    def summary(self, t0: float, t1: float):
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
        note = "samples inside the timed region"
        if not inside:
            inside = rows[-3:]
            note = "timed region shorter than the sampling period; last samples of the loaded run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "no samples"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3][i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "note": note}


# ------------------------------------------------------------- CPU baseline

def cpu_baseline(batch, config, target_s: float):
    """The fp64 oracle, as it stands, on this host's cores, on a bounded sample."""
    import oracle
    Hq = batch.num_q_heads
    work = work_of(batch)
    total_rows = batch.num_tokens * Hq
    # keys per row decide the cost; pick rows evenly over the batch
    rows = [(t, h) for t in range(batch.num_tokens) for h in range(Hq)]
    n = len(rows)
    probe = rows[:: max(1, n // 64)][:64]
    t = time.perf_counter()
    oracle.batch_attention(batch, rows=probe)
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
        oracle.batch_attention(batch, rows=sample)
    elapsed = time.perf_counter() - t
    frac = len(sample) * reps / total_rows
    step_s = elapsed / frac
    metric, unit, _ = metric_of(config)
    return {"value": value_of(config, work, step_s), "unit": unit, "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{len(sample)} of {total_rows} (token, head) rows x {reps} repetition(s), "
                      f"{elapsed:.1f} s; step time scaled by the row fraction"}


def run_reference(args):
    """--impl reference: the fp64 CPU oracle timed as the reference arm."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from paged_kv_cache_forward_gb300 import workloads as W
    torch.manual_seed(0)
    batch = W.CONFIGS[args.config](seed=args.seed)
    metric, unit, _ = metric_of(args.config)
    steps = args.steps or 3
    warm = max(0, min(args.warmup, 1))
    budget = min(120.0 / max(1, steps + warm), args.cpu_seconds)
    for _ in range(warm):
        cpu_baseline(batch, args.config, min(budget, 5.0))
    vals = [cpu_baseline(batch, args.config, budget) for _ in range(steps)]
    v = statistics.median(x["value"] for x in vals)
    step_s = (work_of(batch)["flops"] / v / 1e12) if args.config == "varlen_prefill" else \
        (work_of(batch)["kv_bytes"] / v / 1e9)
    line = {
        "impl": "reference", "metric": metric, "value": v, "unit": unit, "n_gpus": args.gpus, "steps": steps,
        "warmup": warm, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.config}: {DESCRIPTIONS.get(args.config, '')}", "seed": args.seed},
        "cpu_baseline": {"value": v, "unit": unit, "cores": vals[0]["cores"], "kind": "oracle",
                         "sample": vals[0]["sample"]},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------- ours

def run_ours(args):
    import torch
    import paged_kv_cache_forward_gb300 as pa
    from paged_kv_cache_forward_gb300 import build as build_mod
    from paged_kv_cache_forward_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_mod.build()
    pa.load()

    batch = W.CONFIGS[args.config](seed=rank_seed(args.seed, rank))
    work = work_of(batch)
    metric, unit, bound = metric_of(args.config)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    per_step = max(work["kv_bytes"], 1)
    R = 1 if per_step > 3 * l2 else int(math.ceil(3 * l2 / per_step)) + 1

    d = batch.to(dev)
    ks = [d.k_cache] + [d.k_cache.clone() for _ in range(R - 1)]
    vs = [d.v_cache] + [d.v_cache.clone() for _ in range(R - 1)]
    out = torch.empty_like(d.q)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)  # inputs and pool copies were made on the default stream
    plan = pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens, kv_chunk=args.kv_chunk)
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, kv_chunk=args.kv_chunk, stream=stream)
    G = batch.num_q_heads // batch.num_kv_heads
    qmax = 16 // G if G <= 16 else 1
    has_decode = any(1 <= n <= qmax for n in batch.q_lens())
    dominant = "prefill" if (args.config == "varlen_prefill" or not has_decode) else "decode_splitkv"

    def call(i, events=None):
        pa.forward(d.q, ks[i % R], vs[i % R], d.block_table, d.seq_lens, d.query_start_loc, out,
                   scale=batch.scale, kv_chunk=args.kv_chunk, events=events, stream=stream)

    # eager warm-up (loads the kernels, sets attributes)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            call(i)
    stream.synchronize()
    assert pa.device_error(stream) == 0

    # time one eager step to size the default step count (about 2 s of timed work)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for i in range(10):
            call(i)
        e1.record()
    stream.synchronize()
    est_ms = e0.elapsed_time(e1) / 10
    steps = args.steps if args.steps else int(min(200000, max(200, 2000.0 / max(est_ms, 1e-3))))

    # graphs of M consecutive steps each, rotating over the R pool copies.  The
    # dominant kernel's launches are timed by pairs of external events: when a
    # step is that one kernel, each pair brackets a run of RUN consecutive
    # launches (one run in every EVERY steps; the mean launch duration is the
    # run's time / RUN); when a step launches more kernels, each pair brackets
    # the dominant kernel of one step in EVERY.  (An event node between two
    # kernels costs the graph a few microseconds, which a lone bracket charges
    # to the kernel it surrounds.)  Their durations give roofline.achieved.
    EVERY = 8
    M = min(steps, max(R, 256))
    M = max(R, (M // R) * R) if M >= R else M
    key = "prefill" if dominant == "prefill" else "decode"
    RUN = 16 if plan["launches"] == 1 and M >= 16 else 1
    if RUN > 1:
        EVERY = 64

    def make_graph(n):
        starts = [i for i in range(0, n, EVERY) if i + RUN <= n]
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in starts]
        # torch creates the CUDA event on its first record(); do that outside the
        # capture so that the library receives real handles to re-record.
        for e_a, e_b in evs:
            e_a.record(stream)
            e_b.record(stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                ev = {}
                k, r = divmod(i, EVERY)
                if k < len(evs):
                    if r == 0:
                        ev[f"{key}_start_event"] = evs[k][0]
                    if r == RUN - 1:
                        ev[f"{key}_stop_event"] = evs[k][1]
                call(i, events=ev or None)
        return g, evs

    full, rem = divmod(steps, M)
    g_main, ev_main = make_graph(M)
    g_rem, ev_rem = make_graph(rem) if rem else (None, [])

    sampler = ClockSampler(local).start()
    # graph warm-up: at least W steps, and at least ~0.5 s so that clocks settle
    warm_reps = max(1, int(math.ceil(args.warmup / M)), int(args.min_warm_ms / max(est_ms * M, 1e-3)))
    for _ in range(warm_reps):
        g_main.replay()
    stream.synchronize()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    with torch.cuda.stream(stream):
        start.record()
        for _ in range(full):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        stop.record()
    stream.synchronize()
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier(world)
    sampler.stop()
    region_ms = start.elapsed_time(stop)
    # the last replay of each graph left its events' times
    kernel_ms = [a.elapsed_time(b) / RUN for a, b in ev_main + ev_rem]
    assert pa.device_error(stream) == 0

    region_ms_max = reduce_max(region_ms, world, dev)
    ms_per_step = region_ms_max / steps
    total_kv = reduce_sum(work["kv_bytes"], world, dev)
    total_flops = reduce_sum(work["flops"], world, dev)
    total_tokens = reduce_sum(work["tokens"], world, dev)
    if args.config == "varlen_prefill":
        value = total_flops * steps / (region_ms_max / 1e3) / 1e12
    else:
        value = total_kv * steps / (region_ms_max / 1e3) / 1e9

    # roofline of the dominant kernel
    peaks = measured_peaks()
    k_ms = statistics.mean(kernel_ms)
    if dominant == "prefill":
        peak, src = peaks["bf16"]
        achieved = work["flops"] / (k_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": src}
    else:
        peak, src = peaks["hbm"]
        achieved = work["decode_bytes"] / (k_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": src}
    traffic = committed_traffic(dominant, args.config)
    qs = statistics.quantiles(kernel_ms, n=10) if len(kernel_ms) >= 2 else [k_ms] * 9
    roof.update({"traffic": traffic, "kernel": dominant, "kernel_ms_mean": k_ms,
                 "kernel_ms_median": statistics.median(kernel_ms),
                 "kernel_ms_p10": qs[0], "kernel_ms_p90": qs[-1],
                 "algorithmic_per_launch": work["flops"] if dominant == "prefill" else work["decode_bytes"]})

    hbm_frac = (total_kv / world) / (ms_per_step / 1e3) / 1e9 / peaks["hbm"][0]
    tensor_frac = (total_flops / world) / (ms_per_step / 1e3) / 1e12 / peaks["bf16"][0]

    # end to end through the public API: pinned host inputs -> device, forward, result -> host
    e2e = None
    if not args.no_e2e:
        # A step's inputs (q, block table, lengths, query offsets) packed in one
        # pinned host buffer and one device arena (16-byte aligned parts), so a
        # step is one host-to-device copy, pa_forward on views of the arena, and
        # one device-to-host copy of out.
        parts = [batch.q, batch.block_table, batch.seq_lens, batch.query_start_loc]
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
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        n_e2e = min(steps, 2048)

        def e2e_step(i):
            dbuf.copy_(hbuf, non_blocking=True)
            pa.forward(eq, ks[i % R], vs[i % R], ebt, esl, eqsl, out, scale=batch.scale, kv_chunk=args.kv_chunk,
                       stream=stream)
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
        # (b) the same steps captured in a CUDA graph (copies from pinned memory
        # and the forward), replayed: what a serving loop that captures its
        # decode step sees
        Me = min(64, n_e2e)
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=stream):
            for i in range(Me):
                e2e_step(i)
        reps = max(1, n_e2e // Me)
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
                pa.forward(qv, ks[i % R], vs[i % R], btv, slv, qslv, outs2[k], scale=batch.scale,
                           kv_chunk=args.kv_chunk, stream=stream)
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
        gp.replay()
        pipe_ms = reduce_max(timed(lambda r: gp.replay(), reps), world, dev) / (reps * Me)
        del gp
        h2d = sum(t.numel() * t.element_size() for t in parts)
        work_all = {"kv_bytes": total_kv, "flops": total_flops}
        what = ("per step: q and metadata copied (one packed copy) from pinned host memory, pa_forward, out "
                "copied to pinned host memory, serial on one stream; KV cache resident")
        modes = {
            "graph_pipelined": (pipe_ms, "per step: q and metadata copied (one packed copy) from pinned host memory "
                                         "on a side stream, pa_forward, out copied to pinned host memory on a second "
                                         "side stream, two alternating input/output buffers so that neighbouring "
                                         "steps' copies overlap the forward; captured in CUDA graphs of 64 steps; "
                                         "KV cache resident"),
            "graph": (graph_ms, what + "; steps captured in CUDA graphs of 64 and replayed"),
            "eager": (eager_ms, what + "; launched eagerly from the host"),
        }
        best = min(modes, key=lambda m: modes[m][0])
        e_ms = modes[best][0]
        e2e = {"value": value_of(args.config, work_all, e_ms / 1e3),
               "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hout.numel() * hout.element_size(),
               "ms_per_step": e_ms, "steps": n_e2e, "mode": best + ": " + modes[best][1],
               "modes_ms_per_step": {m: v[0] for m, v in modes.items()}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(batch, args.config, args.cpu_seconds)

    clocks = sampler.summary(t0, t1)
    if rank == 0:
        line = {
            "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": steps,
            "warmup": warm_reps * M, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": f"{args.config}: {DESCRIPTIONS.get(args.config, '')}",
                "seed": args.seed, "global_batch": batch.num_seqs * world, "tokens_per_step": int(total_tokens),
                "kv_bytes_per_step": int(total_kv), "causal_flops_per_step": int(total_flops),
                "l2": f"inputs rotate over {R} KV pool copies ({R} x {work['kv_bytes'] / 2**20:.0f} MiB "
                      f"> 3 x L2 {l2 / 2**20:.0f} MiB)" if R > 1 else "KV bytes per step > 3 x L2",
                "graph": f"CUDA graphs of {M} steps", "kv_chunk": plan["kv_chunk"], "splits": plan["splits"],
                "decode_stages": plan["decode_stages"],
                "kernel_timing": (f"CUDA events around runs of {RUN} consecutive launches of the dominant "
                                  f"kernel (the whole step), one run in {EVERY} steps of the timed graphs "
                                  f"({len(kernel_ms)} runs of the last replays)" if RUN > 1 else
                                  f"CUDA events around the dominant kernel of one step in {EVERY} of the "
                                  f"timed graphs ({len(kernel_ms)} launches of the last replays)"),
                "parallelism": f"dp{world}" if world > 1 else "single GPU",
            },
            "tok_s": total_tokens * steps / (region_ms_max / 1e3),
            # one attention layer per step; a 32-layer model's attention alone
            # could run at most this many tokens/s
            "tok_s_32_layer_attention_ceiling": total_tokens * steps / (region_ms_max / 1e3) / 32,
            # whole step against each roofline: KV bytes / HBM, causal FLOPs /
            # bf16 tensor peak, and the binding one, max(B / BW, F / peak) / t
            "hbm_frac_step": hbm_frac,
            "tensor_frac_step": tensor_frac,
            "roofline_frac_step": max(hbm_frac, tensor_frac),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": plan["launches"] * steps,
            "clocks": clocks,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_layers(args):
    """A decoder step of L attention layers: every layer has its own paged KV
    cache (same shape, same block table), its own queries and output, and one
    pa_forward call.  Times three ways of launching the same L calls: one CUDA
    graph of the whole step, L one-layer graphs replayed back to back, and L
    eager calls.  value = KV bytes of all layers per second in the one-graph mode."""
    import torch
    import paged_kv_cache_forward_gb300 as pa
    from paged_kv_cache_forward_gb300 import build as build_mod
    from paged_kv_cache_forward_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_mod.build()
    pa.load()

    L = args.layers
    batch = W.CONFIGS[args.config](seed=rank_seed(args.seed, rank))
    work = work_of(batch)
    metric, unit, _ = metric_of(args.config)
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
                   scale=batch.scale, kv_chunk=args.kv_chunk, stream=stream)

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
    steps = args.steps or 50
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

    # the one-graph step must give the eager step's outputs
    ref = [o.clone() for o in outs]
    g_full.replay()
    stream.synchronize()
    identical = all(torch.equal(a, b) for a, b in zip(ref, outs))

    total_kv = reduce_sum(work["kv_bytes"], world, dev) * L
    total_flops = reduce_sum(work["flops"], world, dev) * L
    ms = times["graph_full"]
    value = value_of(args.config, {"kv_bytes": total_kv, "flops": total_flops}, ms / 1e3)
    peaks = measured_peaks()
    if rank == 0:
        line = {
            "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": f"{L} layers x {args.config}: {DESCRIPTIONS.get(args.config, '')}",
                "layers": L, "kv_bytes_per_step": int(total_kv), "kv_chunk": plan["kv_chunk"],
                "splits": plan["splits"], "l2": f"KV bytes per step {total_kv / 2**20:.0f} MiB "
                                                 f"({'>' if total_kv > 3 * (128 << 20) else '<='} 3 x L2)",
                "parallelism": f"dp{world}" if world > 1 else "single GPU",
            },
            "graph_modes_ms_per_step": times,
            "launch_overhead_us_per_layer": {
                k: (v - times["graph_full"]) * 1e3 / L for k, v in times.items() if k != "graph_full"},
            "us_per_layer": ms * 1e3 / L,
            "hbm_frac_step": (total_kv / world) / (ms / 1e3) / 1e9 / peaks["hbm"][0],
            "graph_matches_eager": identical,
            "gpu_launches": plan["launches"] * L * steps,
            "clocks": sampler.summary(t0, t1),
        }
        print(json.dumps(line))
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
