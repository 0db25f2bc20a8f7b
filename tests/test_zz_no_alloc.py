"""pa_forward_noalloc: the forward pass for callers that cannot let a library
allocate device memory -- hosts whose device memory is owned or budgeted up
front by their own allocator (an inference server that gives all free memory
to its KV-cache pool, a plugin inside another framework), and latency-critical
loops where an allocation's cost or failure at an arbitrary call is not
acceptable.  It runs the same kernels with the same launch plan as pa_forward,
keeping its split scratch in the library's fixed device array, so it must give
pa_forward's output bit for bit, call after call, and allocate nothing.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It passes both alone in a
fresh process and after the rest of the suite.
"""

import pytest
import torch

import oracle
import paged_kv_cache_forward_gb300 as pa
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import assert_close, ensure_built

pytestmark = pytest.mark.gpu


def _batch():
    # decode sequences long enough to be split (the scratch path), a chunked
    # prefill, and an empty sequence, in one batch
    return W.make_batch([1, 1, 37, 0, 1], [5000, 700, 300, 9, 1], 32, 8, 128, seed=61, max_pages=400)


def _reference(d, b):
    ref = torch.full_like(d.q, float("nan"))
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, ref, scale=b.scale)
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    return ref


def _noalloc(d, b, out, err):
    out.fill_(float("nan"))
    pa.forward_noalloc(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out,
                       scale=b.scale, device_error=err)
    torch.cuda.synchronize()


def test_noalloc_matches_pa_forward_and_the_oracle_two_calls_in_a_row():
    ensure_built()
    b = _batch()
    d = b.to("cuda")
    assert pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens)["splits"] > 1
    ref = _reference(d, b)
    want = oracle.batch_attention(b)
    assert_close(ref.cpu(), want, "pa_forward vs oracle")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(d.q)
    for call in range(2):
        _noalloc(d, b, out, err)
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item())}"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}: differs from pa_forward"
        assert_close(out.cpu(), want, f"call {call} vs oracle")


def test_noalloc_without_an_error_word_and_without_allocating():
    """device_error = NULL keeps the error word in the scratch itself; calls made
    after the first allocate no device memory (the free bytes the driver reports
    do not move)."""
    ensure_built()
    b = _batch()
    d = b.to("cuda")
    ref = _reference(d, b)
    out = torch.empty_like(d.q)
    _noalloc(d, b, out, None)  # loads the library's code (and its array) on this GPU if not yet done
    pa.release_workspaces()
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for call in range(2):
        _noalloc(d, b, out, None)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}: differs from pa_forward"
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, f"free device memory moved by {free_before - free_after} bytes"


def test_noalloc_reports_a_bad_block_id_in_the_callers_word():
    ensure_built()
    b = W.make_batch([1, 1], [900, 40], 32, 8, 128, seed=62)
    good = oracle.batch_attention(b, rows=[(1, h) for h in range(32)])
    bad = W.Batch(**{**b.__dict__, "block_table": b.block_table.clone()})
    bad.block_table[0, 3] = b.num_blocks + 5  # outside the pool: checked, skipped, reported
    d = bad.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(d.q)
    _noalloc(d, bad, out, err)
    assert int(err.item()) == 1
    # the context is still usable, and the sequence with valid pages is right
    assert_close(out[1].cpu(), good, "the sequence with valid pages")


def test_noalloc_rejects_shapes_beyond_the_scratch():
    ensure_built()
    # 256 sequences x 8192-token bound: the split partials need far more than 32 MiB
    dims = pa.Dims(num_tokens=256, num_blocks=4, num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
                   page_size=16, max_pages=8192)
    need = pa.plan(dims)["workspace_bytes"]
    assert need > 32 << 20
    q = torch.zeros(256, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(256, 8192, dtype=torch.int32, device="cuda")
    sl = torch.ones(256, dtype=torch.int32, device="cuda")
    qsl = torch.arange(257, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.forward_noalloc(q, kc, kc, bt, sl, qsl, scale=0.1)
    assert e.value.status == 2
    assert "scratch" in str(e.value)
