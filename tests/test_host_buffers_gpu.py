"""Decode calls whose q, metadata and output live in pinned host memory.

The decode kernel reads q and the metadata and writes out with plain loads and
stores, so for shapes that allow no prefill rows these may be pinned host
buffers that the device addresses directly (over NVLink-C2C on Grace-Blackwell):
the output must equal, bit for bit, the same call on device buffers (same
kernels, same plan), and match the oracle.  Shapes that allow prefill rows must
refuse a host q before launching anything (the prefill kernel reads q with
tensor copies)."""

from __future__ import annotations

import pytest
import torch

import oracle
import paged_kv_cache_forward_gb300 as pa
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import assert_close, ensure_built

pytestmark = pytest.mark.gpu

# Shapes whose dims allow no prefill rows: one sequence with one new token.
_CASES = {
    "decode_1024": lambda: W.llama_decode(1024, seed=121),
    "decode_8192": lambda: W.llama_decode(8192, seed=122),
    "decode_32768": lambda: W.llama_decode(32768, seed=123),
    "short": lambda: W.make_batch([1], [7], 32, 8, 128, seed=124),
    "mha": lambda: W.make_batch([1], [5000], 32, 32, 128, seed=125),
    "g32": lambda: W.make_batch([1], [4000], 64, 2, 128, seed=126),
    "d64": lambda: W.make_batch([1], [3000], 16, 4, 64, seed=127),
    "d256": lambda: W.make_batch([1], [2500], 16, 2, 256, seed=128),
}


def _pinned(t: torch.Tensor) -> torch.Tensor:
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


@pytest.mark.parametrize("case", sorted(_CASES))
@pytest.mark.parametrize("cluster", [0, 4])
@pytest.mark.parametrize("early", [0, 1])
def test_host_buffers_decode_is_bit_identical(case, cluster, early):
    ensure_built()
    b = _CASES[case]()
    d = b.to("cuda")
    assert pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens)["prefill_ctas"] == 0
    out_d = torch.full_like(d.q, float("nan"))
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out_d, scale=b.scale,
               decode_cluster=cluster, early_metadata=early)
    hq, hbt, hsl, hqsl = (_pinned(t) for t in (b.q, b.block_table, b.seq_lens, b.query_start_loc))
    out_h = _pinned(torch.full_like(b.q, float("nan")))
    pa.forward(hq, d.k_cache, d.v_cache, hbt, hsl, hqsl, out_h, scale=b.scale, decode_cluster=cluster,
               early_metadata=early)
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    assert torch.equal(out_d.cpu().view(torch.int16), out_h.view(torch.int16)), case
    assert_close(out_h, oracle.batch_attention(b), f"{case} cluster {cluster} early {early}")


def test_host_buffers_in_a_graph_see_new_host_contents():
    """Captured once with host buffers, replayed after the host rewrote q and the
    lengths in place: each replay gives the eager device result for the new
    contents (the kernel reads the host memory at replay time)."""
    ensure_built()
    b = W.llama_decode(8192, seed=127)
    d = b.to("cuda")
    hq, hbt, hsl, hqsl = (_pinned(t) for t in (b.q, b.block_table, b.seq_lens, b.query_start_loc))
    out_h = _pinned(torch.zeros_like(b.q))
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.forward(hq, d.k_cache, d.v_cache, hbt, hsl, hqsl, out_h, scale=b.scale, stream=s, early_metadata=1)
    gen = torch.Generator().manual_seed(128)
    for length in (8192, 5000, 77):
        q_new = torch.randn(b.q.shape, generator=gen).to(torch.bfloat16)
        hq.copy_(q_new)
        hsl.fill_(length)
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert pa.device_error(s) == 0
        d_q = q_new.cuda()
        d_sl = torch.full_like(d.seq_lens, length)
        ref = torch.empty_like(d_q)
        pa.forward(d_q, d.k_cache, d.v_cache, d.block_table, d_sl, d.query_start_loc, ref, scale=b.scale)
        torch.cuda.synchronize()
        assert torch.equal(ref.cpu().view(torch.int16), out_h.view(torch.int16)), length


@pytest.mark.parametrize("noalloc", [False, True])
@pytest.mark.parametrize("shape", ["mixed", "batched_decode"])
def test_host_q_refused_when_shapes_allow_prefill(noalloc, shape):
    """q in host memory with dims that allow prefill rows (a mixed batch, or
    single-token sequences whose token count could sit in one sequence): the
    call fails with PA_ERR_INVALID_ARG before any launch (out keeps its
    contents)."""
    ensure_built()
    if shape == "mixed":
        b = W.make_batch([300, 1], [800, 2000], 32, 8, 128, seed=129)
    else:
        b = W.make_batch([1] * 24, [513 + 300 * i for i in range(24)], 32, 8, 128, seed=130)
    d = b.to("cuda")
    assert pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens)["prefill_ctas"] > 0
    hq = _pinned(b.q)
    out = torch.full_like(d.q, 7.0)
    fn = pa.forward_noalloc if noalloc else pa.forward
    with pytest.raises(RuntimeError, match="device memory"):
        fn(hq, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
