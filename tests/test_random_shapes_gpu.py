"""Randomised parity sweep: seeded random batches (sequence count, new-token and
context lengths, head counts, head dim, split size, decode variant, cluster
mode) through the C ABI against the fp64 oracle.  Each case is small enough for
the full oracle; together they cover combinations the hand-written cases do not
(empty sequences next to prefill and multi-token decode rows, lengths at and
around page and tile boundaries, G from 1 to 32)."""

import random

import pytest
import torch

import oracle
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import assert_close, run

pytestmark = pytest.mark.gpu

HEADS = [(8, 8), (16, 4), (32, 8), (12, 4), (32, 1), (16, 2), (4, 1)]
DIMS = [64, 128, 256]
VARIANTS = {64: [(4, 2), (4, 3), (4, 4), (8, 2), (8, 3), (12, 2)], 128: [(4, 2), (4, 3), (4, 4), (8, 2), (8, 3),
                                                                         (12, 2)], 256: [(4, 2), (4, 3)]}


def draw_case(seed):
    r = random.Random(seed)
    Hq, Hkv = r.choice(HEADS)
    D = r.choice(DIMS)
    G = Hq // Hkv
    qmax = 16 // G if G <= 16 else 1
    B = r.randint(1, 6)
    q_lens, seq_lens = [], []
    for _ in range(B):
        kind = r.choice(["empty", "decode", "multi", "prefill", "prefill"])
        L = r.choice([1, 15, 16, 17, 127, 128, 129, r.randint(1, 700), r.randint(1, 2500)])
        if kind == "empty":
            n = 0
        elif kind == "decode":
            n = 1
        elif kind == "multi":
            n = min(L, r.randint(1, qmax))
        else:
            n = min(L, r.choice([qmax + 1, 31, 32, 33, 64, 65, r.randint(2, 300)]))
        q_lens.append(n)
        seq_lens.append(L)
    if sum(q_lens) == 0:
        q_lens[0] = 1
    opts = {}
    mode = r.choice(["table", "chunk", "variant", "cluster"])
    if mode == "chunk":
        opts["kv_chunk"] = 16 * r.choice([1, 3, 8, 32, 100])
    elif mode == "variant":
        opts["decode_warps"], opts["decode_stages"] = r.choice(VARIANTS[D])
    elif mode == "cluster":
        opts["decode_cluster"] = r.choice([2, 3, 5, 8, 16])
    return q_lens, seq_lens, Hq, Hkv, D, opts


@pytest.mark.parametrize("seed", range(1024))
def test_random_case(seed):
    q_lens, seq_lens, Hq, Hkv, D, opts = draw_case(1000 + seed)
    b = W.make_batch(q_lens, seq_lens, Hq, Hkv, D, seed=2000 + seed, max_pages=(max(seq_lens) + 15) // 16 + 3)
    got = run(b, **opts)
    what = f"q_lens {q_lens} seq_lens {seq_lens} heads {Hq}/{Hkv} D {D} {opts}"
    assert_close(got, oracle.batch_attention(b), what)
    torch.cuda.synchronize()


@pytest.mark.parametrize("seed", range(64))
def test_random_batch_early_metadata(seed):
    """pa_options.early_metadata on random batches: the output equals the default
    call's bit for bit, and two calls captured back to back in a CUDA graph (the
    second reading the first's output as its queries, so it may be scheduled
    while the first still runs) equal the same two calls with a device
    synchronisation between them."""
    import paged_kv_cache_forward_gb300 as pa
    q_lens, seq_lens, Hq, Hkv, D, opts = draw_case(seed + 50000)
    b = W.make_batch(q_lens, seq_lens, Hq, Hkv, D, seed=seed + 50000)
    d = b.to("cuda")
    outs = []
    for early in (0, 1):
        out = torch.full_like(d.q, float("nan"))
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale,
                   early_metadata=early, **opts)
        torch.cuda.synchronize()
        assert pa.device_error() == 0
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref = torch.empty_like(d.q)
    pa.forward(outs[0], d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, ref, scale=b.scale, **opts)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s, **opts)
    torch.cuda.synchronize()
    mid, fin = torch.empty_like(d.q), torch.empty_like(d.q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, mid, scale=b.scale,
                   stream=s, early_metadata=1, **opts)
        pa.forward(mid, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, fin, scale=b.scale,
                   stream=s, early_metadata=1, **opts)
    mid.fill_(float("nan"))
    fin.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    assert pa.device_error(s) == 0
    assert torch.equal(fin.view(torch.int16), ref.view(torch.int16))
