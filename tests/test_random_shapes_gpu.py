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
