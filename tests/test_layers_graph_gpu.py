"""A decoder step of L attention layers in one CUDA graph.

The Triton unified-attention page (section "A counter-intuitive finding: AMD
cards depend more on full graphs") measures that capturing the whole model step
in one graph, rather than piece by piece, removes per-launch overhead.  Here L
pa_forward calls, each with its own queries, paged KV cache, block table and
output, are captured in one graph; the graph is replayed, then replayed again
after new contents (new queries, caches, block tables, lengths and query split,
same shapes) were copied into the same buffers.  Sampled rows of every layer are
compared with the oracle after each replay.
"""

import pytest
import torch

import oracle
import paged_kv_cache_forward_gb300 as pa
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, sample_rows

pytestmark = pytest.mark.gpu

POOL, MAX_PAGES = 420, 200


def _layer_batch(layer: int, contents: int, Hq: int, Hkv: int, D: int) -> W.Batch:
    # same shapes for every layer and both contents (T, pool, max_pages); the
    # lengths and the split of the T = 43 query rows between sequences differ
    if contents == 0:
        ql, sl = [1, 1, 1, 40], [3000, 517, 1, 300]
    else:
        ql, sl = [40, 1, 1, 1], [40, 2999, 700, 5]
    return W.make_batch(ql, sl, Hq, Hkv, D, seed=1000 * contents + layer, pool_pages=POOL, max_pages=MAX_PAGES)


def _copy_into(dst, src: W.Batch):
    for name in ("q", "k_cache", "v_cache", "block_table", "seq_lens", "query_start_loc"):
        getattr(dst, name).copy_(getattr(src, name))


def _check(batches, outs, what):
    for i, b in enumerate(batches):
        rows = sample_rows(b, 24, seed=i)
        ref = oracle.batch_attention(b, rows=rows)
        got = outs[i].cpu()
        sel = torch.stack([got[t, h] for t, h in rows])
        assert_close(sel, ref, f"{what}, layer {i}")


@pytest.mark.parametrize("L,Hq,Hkv,D", [(4, 32, 8, 128), (32, 32, 8, 128), (8, 16, 2, 64)])
def test_layers_in_one_graph_replayed_with_new_contents(L, Hq, Hkv, D):
    ensure_built()
    first = [_layer_batch(i, 0, Hq, Hkv, D) for i in range(L)]
    dev = [b.to("cuda") for b in first]
    outs = [torch.full_like(d.q, float("nan")) for d in dev]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    # the largest shapes of the step: every layer has the same dims
    pa.prepare(dev[0].q, dev[0].k_cache, dev[0].block_table, dev[0].seq_lens, stream=s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for d, o in zip(dev, outs):
            pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, o,
                       scale=first[0].scale)
    g.replay()
    torch.cuda.synchronize()
    assert pa.device_error(s) == 0
    _check(first, outs, "first contents")

    second = [_layer_batch(i, 1, Hq, Hkv, D) for i in range(L)]
    for d, b in zip(dev, second):
        _copy_into(d, b)
    for o in outs:
        o.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert pa.device_error(s) == 0
    _check(second, outs, "new contents")
