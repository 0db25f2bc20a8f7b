"""Offline sweep that produces the split table (csrc/lut_gb300.inc).

The Triton unified-attention page (section "What three things the IBM paper got
right", third item) replaces run-time autotuning by offline micro-benchmarks
distilled into a small decision tree keyed on GPU, sequence length and batch.
This is that step for GB300: for every (context bound, batch size) cell of a
grid it times pa_forward on Llama-3.1-8B-shaped decode batches (32 query heads,
8 KV heads, head_dim 128; one sequence at the context bound, or a batch with
lengths uniform in [bound/16, bound]) for a set of
(split size, decode kernel variant) pairs -- a variant is the warps per CTA
and the pipeline depth per warp -- and keeps the fastest.  The result is written as a table that the
library compiles in; nothing is tuned at run time.

    python -m paged_kv_cache_forward_gb300.sweep [--out csrc/lut_gb300.inc] [--log profiles/...md]

Needs a GPU.  Inputs are random bf16 drawn on the device (values do not change
the timing of this HBM-bound kernel); steps rotate over enough KV pool copies
that no step finds its pages in L2.
"""

from __future__ import annotations

import argparse
import datetime
import math
import re
import os
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import paged_kv_cache_forward_gb300 as pa  # noqa: E402

BOUNDS = [1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072]
BATCHES = [1, 2, 4, 8, 16, 32, 64, 128, 256]
HQ, HKV, D, PAGE = 32, 8, 128, 16
MAX_KV_BYTES = 6 << 30


SMEM_PER_SM = 228 << 10
REGS_PER_SM = 65536
REGS_PER_THREAD = 168
VARIANTS = "4x2,4x3,4x4,8x2,8x3,12x2"  # warps x stages


def resident_ctas(warps: int, stages: int) -> int:
    """Decode CTAs an SM holds: shared memory (K and V of one page per stage per
    warp, 1 KiB reserved per CTA) and registers (at most 168 per thread)."""
    per_cta = warps * stages * 2 * PAGE * D * 2 + 1024
    return max(1, min(SMEM_PER_SM // per_cta, REGS_PER_SM // (warps * 32 * REGS_PER_THREAD)))


def candidates(bound: int, batch: int, sms: int, warps: int, stages: int):
    base = {64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384}
    # split sizes that give whole waves of CTAs at this variant's residency
    per_sm = resident_ctas(warps, stages)
    for k in (1, 2, 3):
        pages = math.ceil(bound * batch * HKV / (k * per_sm * sms) / PAGE)
        base.add(max(1, pages) * PAGE)
    return sorted(c for c in base if 16 <= c <= bound)


def time_shape(bound, batch, chunk, pools, stream, warps=0, stages=0, cluster=0, steps_per_graph=16, reps=30):
    q, ks, vs, bt, sl, qsl, out = pools
    R = len(ks)
    pa.prepare(q, ks[0], bt, sl, kv_chunk=chunk, stream=stream, decode_stages=stages,
               decode_warps=warps, decode_cluster=cluster)
    with torch.cuda.stream(stream):
        for i in range(2):
            pa.forward(q, ks[i % R], vs[i % R], bt, sl, qsl, out, kv_chunk=chunk, stream=stream,
                       decode_stages=stages, decode_warps=warps, decode_cluster=cluster)
    stream.synchronize()
    M = max(R, (steps_per_graph // R) * R)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(M):
            pa.forward(q, ks[i % R], vs[i % R], bt, sl, qsl, out, kv_chunk=chunk, stream=stream,
                       decode_stages=stages, decode_warps=warps, decode_cluster=cluster)
    for _ in range(3):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    stream.synchronize()
    code = pa.device_error(stream)
    if code:
        raise RuntimeError(f"device error {code} ({pa.DEVICE_ERRORS.get(code)}) at bound {bound}, batch {batch}, "
                           f"split {chunk}, variant {warps}x{stages}, cluster {cluster}")
    return e0.elapsed_time(e1) * 1e3 / (reps * M)  # us per step


def seq_lengths(bound, batch):
    """One sequence at the bound; a batch has lengths uniform in [bound/16, bound]
    (as a serving batch mixes lengths; with every sequence at the bound the
    table would favour unsplit CTAs, whose longest sequences then set the time)."""
    if batch == 1:
        return [bound]
    g = torch.Generator().manual_seed(bound * 1000 + batch)
    lo = max(1, bound // 16)
    return torch.randint(lo, bound + 1, (batch,), generator=g).tolist()


def make_pools(bound, batch, l2_bytes, gen):
    pages = bound // PAGE
    lens = seq_lengths(bound, batch)
    kv = sum(lens) * HKV * D * 2 * 2
    R = 1 if kv > 3 * l2_bytes else int(math.ceil(3 * l2_bytes / kv)) + 1
    nb = batch * pages + 1
    dev = "cuda"
    q = torch.randn(batch, HQ, D, device=dev, generator=gen).to(torch.bfloat16)
    ks, vs = [], []
    for _ in range(R):
        ks.append(torch.randn(nb, PAGE, HKV, D, device=dev, generator=gen).to(torch.bfloat16))
        vs.append(torch.randn(nb, PAGE, HKV, D, device=dev, generator=gen).to(torch.bfloat16))
    perm = torch.randperm(nb, device=dev, generator=gen).to(torch.int32)
    bt = perm[: batch * pages].reshape(batch, pages).contiguous()
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    qsl = torch.arange(batch + 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    return (q, ks, vs, bt, sl, qsl, out), kv


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(HERE, "csrc", "lut_gb300.inc"))
    ap.add_argument("--no-write", action="store_true", help="print the results only")
    ap.add_argument("--log", default=os.path.join(os.path.dirname(HERE), "profiles", "split_table_sweep__gb300.md"))
    ap.add_argument("--bounds", default=",".join(map(str, BOUNDS)))
    ap.add_argument("--batches", default=",".join(map(str, BATCHES)))
    ap.add_argument("--variants", default=VARIANTS, help="decode variants to try: warps x stages")
    ap.add_argument("--clusters", default="2,4,8,16", help="cluster sizes to try (pages dealt round-robin, merge in DSMEM)")
    ap.add_argument("--merge", action="store_true",
                    help="replace only the swept (bound, batch) cells of the existing table and log")
    args = ap.parse_args(argv)
    bounds = [int(x) for x in args.bounds.split(",")]
    batches = [int(x) for x in args.batches.split(",")]
    variants = [tuple(int(y) for y in v.split("x")) for v in args.variants.split(",")]
    clusters = [int(c) for c in args.clusters.split(",") if c]

    from paged_kv_cache_forward_gb300 import build
    build.build()
    pa.load()
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    stream = torch.cuda.Stream()
    gen = torch.Generator(device="cuda").manual_seed(0)
    best = {}
    lines = []
    for batch in batches:
        for bound in bounds:
            if batch * bound * HKV * D * 4 > MAX_KV_BYTES:
                continue
            pools, kv = make_pools(bound, batch, l2, gen)
            # the pools were filled on the default stream; the timing runs on
            # `stream`, which does not order itself after it
            torch.cuda.synchronize()
            res = []
            for w, st in variants:
                # (split size, 1): splits merged through the workspace;
                # (0, C): the pages dealt round-robin to a cluster of C CTAs
                cands = [(c, 1) for c in candidates(bound, batch, sms, w, st)] + [(0, c) for c in clusters]
                for chunk, cl in cands:
                    try:
                        us = time_shape(bound, batch, chunk, pools, stream, warps=w, stages=st, cluster=cl)
                    except RuntimeError as e:  # reported, and the candidate is not used
                        print(f"skipped: {e}", flush=True)
                        continue
                    res.append((us, chunk, st, w, cl))
            res.sort()
            us, chunk, st, w, cl = res[0]
            best[(bound, batch)] = (chunk, st, w, cl)
            name = lambda c, cl: f"c{cl}" if cl > 1 else f"{c}"
            row = " ".join(f"{name(c, k)}/{ww}x{t}:{kv / u / 1e3:.0f}"
                           for u, c, t, ww, k in sorted(res, key=lambda x: (x[3], x[2], x[4], x[1])))
            lines.append(f"| {batch} | {bound} | {name(chunk, cl)} | {w}x{st} | {us:.1f} | {kv / us / 1e3:.0f} | {row} |")
            print(lines[-1], flush=True)
            del pools
            torch.cuda.empty_cache()

    # table: (max_bound, max_units) cells, batch-major, so the first match is the
    # smallest swept batch >= B and, within it, the smallest swept bound >= bound;
    # units = sequences x KV heads (x row groups), so other head counts map onto
    # the Llama-shaped sweep by their parallelism
    if args.merge:
        cells, old_lines = read_table(args.out), read_log(args.log)
        cells.update(best)
        for line in lines:
            old_lines[tuple(int(x) for x in line.split("|")[1:3])] = line
        best = cells
        batches = sorted({k[1] for k in best})
        bounds = sorted({k[0] for k in best})
        lines = [old_lines[(bt, bd)] for bt in batches for bd in bounds if (bt, bd) in old_lines]
    entries = []
    for batch in batches:
        for bound in bounds:
            if (bound, batch) in best:
                entries.append((bound, batch) + best[(bound, batch)])
    last_batch = max(e[1] for e in entries)
    fallback = max(entries, key=lambda e: (e[1], e[0]))[2:]
    stamp = datetime.date.today().isoformat()
    if not args.no_write:
        write_table(args.out, entries, last_batch, fallback, props.name, stamp)
    with open(args.log, "w") as f:
        f.write(f"# Split-size sweep on {props.name} ({stamp})\n\n"
                f"Command: `python -m paged_kv_cache_forward_gb300.sweep {' '.join(argv or sys.argv[1:])}`\n\n"
                "Llama-3.1-8B-shaped decode (Hq 32, Hkv 8, D 128); batch 1 at the bound, larger batches\n"
                "with lengths uniform in [bound/16, bound] (seeded per cell),\n"
                "graph-replayed pa_forward steps rotating over KV pool copies larger than 3 x L2.\n"
                "GB/s = KV bytes per step / step time.\n\n"
                "Split `cN`: the pages dealt round-robin to a thread-block cluster of N CTAs.\n\n"
                "| batch | bound | best split | warps x stages | us/step | GB/s | split/variant:GB/s for every candidate |\n"
                "|---|---|---|---|---|---|---|\n")
        f.write("\n".join(lines) + "\n")
    print(f"wrote {args.log}" + ("" if args.no_write else f" and {args.out}"))


def read_table(path):
    """The cells of an existing table: {(bound, batch): (chunk, stages, warps, cluster)}
    (the last batch's cells carry max_units 1 << 30; the fallback row is dropped)."""
    cells = {}
    rows = re.findall(r"\{(\d+), (\d+|1 << 30), (\d+), (\d+), (\d+), (\d+)\}", open(path).read())
    for bound, units, chunk, st, w, cl in rows:
        batch = max(BATCHES) if units == "1 << 30" or int(units) >= 1 << 30 else int(units) // HKV
        cells[(int(bound), batch)] = (int(chunk), int(st), int(w), int(cl))
    return cells


def read_log(path):
    """The rows of an existing sweep log: {(batch, bound): line}."""
    out = {}
    if os.path.exists(path):
        for line in open(path):
            m = re.match(r"\| (\d+) \| (\d+) \|", line)
            if m:
                out[(int(m.group(1)), int(m.group(2)))] = line.rstrip("\n")
    return out


def write_table(path, entries, last_batch, fallback, gpu_name, stamp):
    with open(path, "w") as f:
        f.write("// Keys per split and decode kernel variant, keyed on the context bound\n"
                "// (max_pages * page_size) and the number of decode units:\n"
                "// {max_bound, max_units, kv_chunk, decode_stages, decode_warps, decode_cluster}\n"
                "// (units = sequences x KV heads x row groups)\n"
                "// (cluster > 1: the pages dealt round-robin to a cluster of that many CTAs).  The first\n"
                "// entry that matches wins; the last entry is the fallback.  Written by\n"
                f"// paged_kv_cache_forward_gb300/sweep.py on {gpu_name} ({stamp}).\n"
                "static const LutEntry kSplitTable[] = {\n")
        for bound, batch, chunk, st, w, cl in entries:
            mb = (1 << 30) if batch == last_batch else batch * HKV
            f.write(f"    {{{bound}, {mb}, {chunk or 16}, {st}, {w}, {cl}}},\n")
        f.write(f"    {{1 << 30, 1 << 30, {fallback[0] or 16}, {fallback[1]}, {fallback[2]}, {fallback[3]}}},\n}};\n")


if __name__ == "__main__":
    main()
