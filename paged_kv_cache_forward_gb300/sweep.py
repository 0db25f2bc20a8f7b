"""Offline sweep that produces the split table (csrc/lut_gb300.inc).

The Triton unified-attention page (section "What three things the IBM paper got
right", third item) replaces run-time autotuning by offline micro-benchmarks
distilled into a small decision tree keyed on GPU, sequence length and batch.
This is that step for GB300: for every (head dim, batch size, context bound)
cell of a grid it times pa_forward on decode batches (32 query heads, 8 KV
heads; one sequence at the context bound, or a batch with lengths uniform in
[bound/16, bound]) for a set of (split, decode kernel variant) candidates -- a
split is a number of keys per CTA merged through the workspace, or a
thread-block cluster of C CTAs that the sequence's pages are dealt to; a
variant is the warps per CTA and the pipeline depth per warp -- and keeps the
fastest.  Every candidate is timed once; the five fastest are timed twice more
and the cell takes the best median of three.  The result is written as a table
that the library compiles in; nothing is tuned at run time.

The table is keyed on decode units (sequences x KV heads x row groups of 16
query heads), not on the batch, so other head counts map onto the sweep by their
parallelism; --validate-groups times, for a few cells with 1, 8 and 32 query
heads per KV head, the table's pick against the best candidate and records the
ratio in the log.

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
import statistics
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import paged_kv_cache_forward_gb300 as pa  # noqa: E402

DIMS = [128, 64, 256]
BOUNDS = [1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072]
BATCHES = {128: [1, 2, 4, 8, 16, 32, 64, 128, 256], 64: [1, 4, 16, 64, 256], 256: [1, 4, 16, 64, 256]}
HQ, HKV, PAGE = 32, 8, 16
SUB_UNIT_KV_HEADS = [1, 2, 4]  # batch-1 cells with fewer KV heads: 1, 2 and 4 decode units
MAX_KV_BYTES = 6 << 30
TOP = 5          # candidates re-timed after the first pass
REPEATS = 3      # timings per re-timed candidate (the cell takes the best median)
MIN_MS = 10.0    # graph replays per timing: at least this long, and at least 3

SMEM_PER_SM = 228 << 10
REGS_PER_SM = 65536
REGS_PER_THREAD = 168
VARIANTS = {64: "4x2,4x3,4x4,8x2,8x3,12x2", 128: "4x2,4x3,4x4,8x2,8x3,12x2", 256: "4x2,4x3"}
CLUSTERS = "2,4,8,12,16"
EARLY = 1        # pa_options.early_metadata in the timed calls (--no-early-metadata: 0)
# Wide groups (more than 16 query heads per KV head: CTAs of 16 heads, each page
# read by every row group of its KV head) have their own cells: Hq 32 / Hkv 1.
WIDE = {128: (32, 1, [1, 2, 4, 8, 16, 64])}  # head_dim: (Hq, Hkv, batches)
WIDE_NAME = "kSplitTableWide"
GROUP_CELLS = [(1, 2048), (1, 8192), (1, 32768), (8, 8192), (64, 4096)]  # (batch, bound) for --validate-groups
GROUP_SHAPES = [(8, 8), (64, 8), (32, 1)]  # (Hq, Hkv): 1, 8 and 32 query heads per KV head


def resident_ctas(warps: int, stages: int, d: int) -> int:
    """Decode CTAs an SM holds: shared memory (K and V of one page per stage per
    warp, 1 KiB reserved per CTA) and registers (at most 168 per thread)."""
    per_cta = warps * stages * 2 * PAGE * d * 2 + 1024
    return max(1, min(SMEM_PER_SM // per_cta, REGS_PER_SM // (warps * 32 * REGS_PER_THREAD)))


def max_keys_per_cta(d: int) -> int:
    """The most keys of one sequence a CTA may stream.  A cell's lengths cannot
    stand for every batch with the same key: the plan only knows the bound, so a
    sequence at the bound must not leave its few CTAs streaming long after the
    rest of the batch is done.  8192 keys at D = 128 (4 MiB of K and V) is what
    the GPU as a whole streams in the time one sequence at the largest bound
    takes on its own (batch-1 cells pick 6912 keys at 131072), so a longer
    per-CTA stream would set the step time whenever the other sequences are short."""
    return 8192 * 128 // d


def candidates(bound: int, units: int, sms: int, warps: int, stages: int, d: int):
    """Split sizes: powers of two, and those that give whole waves of CTAs at this
    variant's residency, up to max_keys_per_cta."""
    base = {64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384}
    per_sm = resident_ctas(warps, stages, d)
    for k in (1, 2, 3):
        pages = math.ceil(bound * units / (k * per_sm * sms) / PAGE)
        base.add(max(1, pages) * PAGE)
    return sorted(c for c in base if 16 <= c <= bound and c <= max_keys_per_cta(d))


def time_shape(pools, stream, chunk=0, warps=0, stages=0, cluster=0, steps_per_graph=16):
    """Microseconds per pa_forward step, from graph replays on `stream`."""
    q, ks, vs, bt, sl, qsl, out = pools
    R = len(ks)
    pa.prepare(q, ks[0], bt, sl, kv_chunk=chunk, stream=stream, decode_stages=stages,
               decode_warps=warps, decode_cluster=cluster)
    with torch.cuda.stream(stream):
        for i in range(2):
            pa.forward(q, ks[i % R], vs[i % R], bt, sl, qsl, out, kv_chunk=chunk, stream=stream,
                       decode_stages=stages, decode_warps=warps, decode_cluster=cluster, early_metadata=EARLY)
    stream.synchronize()
    M = max(R, (steps_per_graph // R) * R)
    # (captured directly: the torch.cuda.graph context manager also runs a
    # garbage collection per capture, which dominated the sweep's time)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        g.capture_begin()
        try:
            for i in range(M):
                pa.forward(q, ks[i % R], vs[i % R], bt, sl, qsl, out, kv_chunk=chunk, stream=stream,
                           decode_stages=stages, decode_warps=warps, decode_cluster=cluster, early_metadata=EARLY)
        finally:
            g.capture_end()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        g.replay()
        e0.record()
        g.replay()
        e1.record()
    stream.synchronize()
    reps = max(3, int(math.ceil(MIN_MS / max(e0.elapsed_time(e1), 1e-3))))
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    stream.synchronize()
    code = pa.device_error(stream)
    if code:
        raise RuntimeError(f"device error {code} ({pa.DEVICE_ERRORS.get(code)}) at split {chunk}, "
                           f"variant {warps}x{stages}, cluster {cluster}")
    return e0.elapsed_time(e1) * 1e3 / (reps * M)


def seq_lengths(bound, batch, d=128, hkv=HKV):
    """One sequence at the bound; a batch has lengths uniform in [bound/16, bound]
    (as a serving batch mixes lengths; with every sequence at the bound the
    table would favour unsplit CTAs, whose longest sequences then set the time).
    Where such a batch would hold more than MAX_KV_BYTES of KV, the bound is set
    by one long sequence and the others are a serving mix of 1024..16384 keys
    (the shape of a mixed prefill/decode batch with one long conversation)."""
    if batch == 1:
        return [bound]
    g = torch.Generator().manual_seed(bound * 1000 + batch)
    lo = max(1, bound // 16)
    if batch * bound * hkv * d * 4 <= MAX_KV_BYTES:
        return torch.randint(lo, bound + 1, (batch,), generator=g).tolist()
    return [bound] + torch.randint(min(1024, bound), min(16384, bound) + 1, (batch - 1,), generator=g).tolist()


def make_pools(bound, batch, d, hq, hkv, l2_bytes, gen):
    """The inputs of one cell: a pool holding just the pages the lengths use (in
    random order), R copies of it when one step's KV bytes fit 3 x L2."""
    pages = bound // PAGE
    lens = seq_lengths(bound, batch, d, hkv)
    kv = sum(lens) * hkv * d * 2 * 2
    R = 1 if kv > 3 * l2_bytes else int(math.ceil(3 * l2_bytes / kv)) + 1
    used = [(n + PAGE - 1) // PAGE for n in lens]
    nb = sum(used) + 1
    dev = "cuda"
    q = torch.randn(batch, hq, d, device=dev, generator=gen).to(torch.bfloat16)
    ks, vs = [], []
    for _ in range(R):
        ks.append(torch.randn(nb, PAGE, hkv, d, device=dev, generator=gen).to(torch.bfloat16))
        vs.append(torch.randn(nb, PAGE, hkv, d, device=dev, generator=gen).to(torch.bfloat16))
    perm = torch.randperm(nb, device=dev, generator=gen).to(torch.int32)
    bt = torch.zeros(batch, pages, dtype=torch.int32, device=dev)  # entries past a sequence are never used
    off = 0
    for i, u in enumerate(used):
        bt[i, :u] = perm[off:off + u]
        off += u
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    qsl = torch.arange(batch + 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    torch.cuda.synchronize()  # filled on the default stream; timing runs on another
    return (q, ks, vs, bt, sl, qsl, out), kv


def all_candidates(bound, units, sms, d, variants, clusters):
    """(split keys, stages, warps, cluster) for every variant: static splits of the
    given keys (cluster 1), and clusters of C CTAs (split 0)."""
    out = []
    for w, st in variants:
        out += [(c, st, w, 1) for c in candidates(bound, units, sms, w, st, d)]
        out += [(0, st, w, c) for c in clusters if math.ceil(bound / c) <= max_keys_per_cta(d)]
    return out


def sweep_cell(pools, stream, cands):
    """Every candidate once, the TOP fastest REPEATS times in all; returns
    [(median us, cand, [timings])] sorted, with the unrepeated ones after."""
    first = []
    for cand in cands:
        chunk, st, w, cl = cand
        try:
            us = time_shape(pools, stream, chunk=chunk, warps=w, stages=st, cluster=cl)
        except RuntimeError as e:  # reported, and the candidate is not used
            print(f"skipped: {e}", flush=True)
            continue
        first.append((us, cand))
    first.sort()
    res = []
    for us, cand in first[:TOP]:
        chunk, st, w, cl = cand
        ts = [us] + [time_shape(pools, stream, chunk=chunk, warps=w, stages=st, cluster=cl)
                     for _ in range(REPEATS - 1)]
        res.append((statistics.median(ts), cand, ts))
    res.sort()
    return res + [(us, cand, [us]) for us, cand in first[TOP:]]


def name_of(chunk, cl):
    return f"c{cl}" if cl > 1 else f"{chunk}"


def validate_groups(args, sms, l2, stream, gen, lines):
    """The table's pick against the best candidate for other group sizes."""
    lines.append("")
    lines.append("## Other group sizes (head_dim 128): the table's pick (keyed on decode units) against the best "
                 "candidate")
    lines.append("")
    lines.append("| Hq / Hkv | batch | bound | table pick | us | best | us | pick / best |")
    lines.append("|---|---|---|---|---|---|---|---|")
    variants = [tuple(int(y) for y in v.split("x")) for v in VARIANTS[128].split(",")]
    clusters = [int(c) for c in args.clusters.split(",") if c]
    for hq, hkv in GROUP_SHAPES:
        for batch, bound in GROUP_CELLS:
            pools, kv = make_pools(bound, batch, 128, hq, hkv, l2, gen)
            p = pa.plan_for(pools[0], pools[1][0], pools[3], pools[4])
            cl = p["decode_cluster"]
            pick = (0 if cl > 1 else p["kv_chunk"], p["decode_stages"], p["decode_warps"], cl)
            t_pick = statistics.median(
                time_shape(pools, stream, chunk=pick[0], warps=pick[2], stages=pick[1], cluster=pick[3])
                for _ in range(REPEATS))
            units = batch * hkv * ((hq // hkv + 15) // 16)
            res = sweep_cell(pools, stream, all_candidates(bound, units, sms, 128, variants, clusters))
            us, (chunk, st, w, c2), _ = res[0]
            lines.append(f"| {hq} / {hkv} | {batch} | {bound} | {name_of(pick[0], pick[3])} {pick[2]}x{pick[1]} | "
                         f"{t_pick:.1f} | {name_of(chunk, c2)} {w}x{st} | {us:.1f} | {t_pick / us:.3f} |")
            print(lines[-1], flush=True)
            del pools
            torch.cuda.empty_cache()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(HERE, "csrc", "lut_gb300.inc"))
    ap.add_argument("--no-write", action="store_true", help="print the results only")
    ap.add_argument("--log", default=os.path.join(os.path.dirname(HERE), "profiles", "split_table_sweep__gb300.md"))
    ap.add_argument("--dims", default=",".join(map(str, DIMS)))
    ap.add_argument("--bounds", default=",".join(map(str, BOUNDS)))
    ap.add_argument("--batches", default="", help="batch sizes (default: per head dim)")
    ap.add_argument("--variants", default="", help="decode variants to try: warps x stages (default: per head dim)")
    ap.add_argument("--clusters", default=CLUSTERS, help="cluster sizes to try (pages dealt round-robin, merge in DSMEM)")
    ap.add_argument("--validate-groups", action="store_true",
                    help="instead of sweeping: time the built table's pick against the best candidate for 1, 8 and "
                         "32 query heads per KV head, and write that to --log")
    ap.add_argument("--only-sub-units", action="store_true",
                    help="sweep only the batch-1 cells with 1, 2 and 4 KV heads (fewer than 8 decode units)")
    ap.add_argument("--merge", action="store_true",
                    help="replace only the swept cells of the existing table and log")
    ap.add_argument("--wide-only", action="store_true",
                    help="sweep only the wide-group cells (more than 16 query heads per KV head)")
    ap.add_argument("--no-early-metadata", action="store_true",
                    help="time calls without pa_options.early_metadata (the table is swept with it by default)")
    args = ap.parse_args(argv)
    global EARLY
    EARLY = 0 if args.no_early_metadata else 1
    dims = [int(x) for x in args.dims.split(",") if x]
    bounds = [int(x) for x in args.bounds.split(",")]
    clusters = [int(c) for c in args.clusters.split(",") if c]

    from paged_kv_cache_forward_gb300 import build
    build.build()
    pa.load()
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    stream = torch.cuda.Stream()
    gen = torch.Generator(device="cuda").manual_seed(0)
    if args.validate_groups:
        extra = [f"# Split table check for other group sizes on {props.name} ({datetime.date.today().isoformat()})",
                 "", f"Command: `python -m paged_kv_cache_forward_gb300.sweep {' '.join(argv or sys.argv[1:])}`"]
        validate_groups(args, sms, l2, stream, gen, extra)
        with open(args.log, "w") as f:
            f.write("\n".join(extra) + "\n")
        print(f"wrote {args.log}")
        return
    best, best_wide = {}, {}
    lines = {}
    for d in dims:
        batches = [int(x) for x in args.batches.split(",")] if args.batches else BATCHES[d]
        variants = [tuple(int(y) for y in v.split("x")) for v in (args.variants or VARIANTS[d]).split(",")]
        variants = [v for v in variants if d != 256 or v[0] == 4]
        # (batch, KV heads): one sequence with fewer KV heads gives the cells
        # below 8 units; then batches of the 8-KV-head shape
        shapes = [(1, h) for h in SUB_UNIT_KV_HEADS] if not args.batches else []
        if not args.only_sub_units:
            shapes += [(b, HKV) for b in batches]
        # (batch, Hq, KV heads, wide)
        cases = [(b, 4 * h, h, False) for b, h in shapes] if not args.wide_only else []
        if d in WIDE and not args.only_sub_units:
            hq_w, hkv_w, batches_w = WIDE[d]
            cases += [(b, hq_w, hkv_w, True) for b in batches_w]
        for batch, hq, hkv, wide in cases:
            units = batch * hkv * ((hq // hkv + 15) // 16)
            for bound in bounds:
                if sum(seq_lengths(bound, batch, d, hkv)) * hkv * d * 4 > MAX_KV_BYTES:
                    continue
                pools, kv = make_pools(bound, batch, d, hq, hkv, l2, gen)
                res = sweep_cell(pools, stream, all_candidates(bound, units, sms, d, variants, clusters))
                us, (chunk, st, w, cl), ts = res[0]
                (best_wide if wide else best)[(d, bound, units)] = (chunk, st, w, cl)
                row = " ".join(f"{name_of(c, k)}/{ww}x{t}:{kv / u / 1e3:.0f}" + ("*" if len(tsx) > 1 else "")
                               for u, (c, t, ww, k), tsx in sorted(res, key=lambda x: (x[1][2], x[1][1], x[1][3],
                                                                                      x[1][0])))
                spread = f"{min(ts):.1f}-{max(ts):.1f}"
                shape = f"{batch} x {hkv}" + (f" (Hq {hq})" if wide else "")
                key = (d, units, bound, shape)
                lines[key] = (f"| {d} | {shape} | {units} | {bound} | {name_of(chunk, cl)} | "
                              f"{w}x{st} | {us:.1f} ({spread}) | {kv / us / 1e3:.0f} | {row} |")
                print(lines[key], flush=True)
                del pools
                torch.cuda.empty_cache()

    if args.merge:
        cells, cells_w, old_lines = read_table(args.out), read_table(args.out, WIDE_NAME), read_log(args.log)
        cells.update(best)
        cells_w.update(best_wide)
        old_lines.update(lines)
        best, best_wide, lines = cells, cells_w, old_lines
    stamp = datetime.date.today().isoformat()
    if not args.no_write:
        write_table(args.out, best, props.name, stamp, best_wide)
    with open(args.log, "w") as f:
        f.write(f"# Split-size sweep on {props.name} ({stamp})\n\n"
                f"Command: `python -m paged_kv_cache_forward_gb300.sweep {' '.join(argv or sys.argv[1:])}`\n\n"
                "Decode batches with 4 query heads per KV head: one sequence with 1, 2, 4 or 8 KV heads at\n"
                "the bound, larger batches (8 KV heads) with lengths uniform in [bound/16, bound] (seeded\n"
                "per cell), or, where those would exceed 6 GiB of KV, one sequence at the bound and the\n"
                "others uniform in [1024, 16384]; units = sequences x KV heads, the table's key,\n"
                "candidates that leave at most 8192 x 128 / head_dim keys of a sequence to one CTA,\n"
                "and wide-group cells (Hq 32 / Hkv 1: two row groups of 16 query heads read each page)\n"
                "for the table's second array,\n"
                "graph-replayed pa_forward steps rotating over KV pool copies larger than 3 x L2,\n"
                f"early_metadata {EARLY} (the metadata is the same for every call).\n"
                "GB/s = KV bytes per step / step time.  Every candidate is timed once; the five fastest\n"
                f"(marked *) {REPEATS} times, and the cell keeps the best median (its spread in brackets).\n\n"
                "Split `cN`: the pages dealt round-robin to a thread-block cluster of N CTAs.\n\n"
                "| head_dim | batch x KV heads | units | bound | best split | warps x stages | us/step | GB/s | "
                "split/variant:GB/s for every candidate |\n"
                "|---|---|---|---|---|---|---|---|---|\n")
        f.write("\n".join(lines[k] for k in sorted(lines)) + "\n")
    print(f"wrote {args.log}" + ("" if args.no_write else f" and {args.out}"))


def read_table(path, array="kSplitTable"):
    """The cells of one array of an existing table: {(head_dim, bound, units):
    (chunk, stages, warps, cluster)} (the catch-all rows and the head-dim-0 end
    row are dropped)."""
    m = re.search(re.escape(array) + r"\[\] = \{(.*?)\n\};", open(path).read(), re.S)
    cells = {}
    if m is None:
        return cells
    rows = re.findall(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\}", m.group(1))
    for d, bound, units, chunk, st, w, cl in rows:
        if int(d):
            cells[(int(d), int(bound), int(units))] = (int(chunk), int(st), int(w), int(cl))
    return cells


def read_log(path):
    """The rows of an existing sweep log: {(head_dim, units, bound, shape): line}."""
    out = {}
    if os.path.exists(path):
        for line in open(path):
            m = re.match(r"\| (\d+) \| ([^|]+?) \| (\d+) \| (\d+) \|", line)
            if m:
                out[(int(m.group(1)), int(m.group(3)), int(m.group(4)), m.group(2))] = line.rstrip("\n")
    return out


def _table_rows(best):
    """Rows {head_dim, max_bound, max_units, ...}: per head dim, units-major, so the
    first match is the smallest swept number of units >= the call's and, within
    it, the smallest swept bound >= the call's.  Each head dim ends with
    catch-all rows: its largest units' cells for any number of units, and that
    group's largest bound for any bound."""
    out = []
    for d in sorted({k[0] for k in best}):
        cells = {k[1:]: v for k, v in best.items() if k[0] == d}
        units = sorted({u for _, u in cells})
        bounds = sorted({bd for bd, _ in cells})
        row = lambda bound, mu, c: f"    {{{d}, {bound}, {mu}, {c[0] or 16}, {c[1]}, {c[2]}, {c[3]}}},\n"
        for u in units:
            for bound in bounds:
                if (bound, u) in cells:
                    out.append(row(bound, u, cells[(bound, u)]))
        top = units[-1]
        for bound in bounds:
            if (bound, top) in cells:
                out.append(row(bound, "1 << 30", cells[(bound, top)]))
        out.append(row("1 << 30", "1 << 30", cells[max(b for b, u in cells if u == top), top]))
    return out


def write_table(path, best, gpu_name, stamp, best_wide=None):
    """kSplitTable from `best`, then kSplitTableWide (calls with more than one row
    group of 16 query heads per KV head) from `best_wide`; a head dim without wide
    rows takes the first table (a row of head dim 0 keeps the array non-empty)."""
    with open(path, "w") as f:
        f.write("// Keys per split and decode kernel variant, keyed on the head dim, the\n"
                "// context bound (max_pages * page_size) and the number of decode units:\n"
                "// {head_dim, max_bound, max_units, kv_chunk, decode_stages, decode_warps, decode_cluster}\n"
                "// (units = sequences x KV heads x row groups of 16 query heads)\n"
                "// (cluster > 1: the pages dealt round-robin to a cluster of that many CTAs).  The first\n"
                "// entry that matches wins.  Written by paged_kv_cache_forward_gb300/sweep.py on\n"
                f"// {gpu_name} ({stamp}).\n"
                "static const LutEntry kSplitTable[] = {\n")
        f.writelines(_table_rows(best))
        f.write("};\n\n"
                "// Calls with more than 16 query heads per KV head (several row groups per KV\n"
                "// head, each reading the same pages); a head dim without rows here takes the\n"
                "// table above.\n"
                f"static const LutEntry {WIDE_NAME}[] = {{\n")
        f.writelines(_table_rows(best_wide or {}))
        f.write("    {0, 0, 0, 0, 0, 0, 0},\n};\n")

if __name__ == "__main__":
    main()
