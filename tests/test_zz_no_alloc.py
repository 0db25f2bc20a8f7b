"""pa_forward_noalloc: the forward pass for callers that cannot let a library
allocate device memory (code inside CUDA-graph capture, hosts that own or
budget all device memory, latency-critical loops).  It must give the same
result as pa_forward, call after call, using only the library's fixed scratch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It passes both alone in a
fresh process and after the rest of the suite.
"""

import pytest
import torch

import paged_kv_cache_forward_gb300 as pa
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import TOL_MAX, TOL_MEAN, ensure_built

pytestmark = pytest.mark.gpu


def _batch():
    # decode sequences long enough to be split (the scratch path), a chunked
    # prefill, and an empty sequence, in one batch
    return W.make_batch([1, 1, 37, 0, 1], [5000, 700, 300, 9, 1], 32, 8, 128, seed=61, max_pages=400)


def test_noalloc_matches_pa_forward_two_calls_in_a_row():
    ensure_built()
    b = _batch()
    d = b.to("cuda")
    assert pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens)["splits"] > 1
    ref = torch.full_like(d.q, float("nan"))
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, ref, scale=b.scale)
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(d.q, float("nan"))
        pa.forward_noalloc(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out,
                           scale=b.scale, device_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = (out.double() - ref.double()).abs()
        assert torch.isfinite(out.float()).all(), f"call {call}: non-finite output"
        assert diff.max().item() <= TOL_MAX and diff.mean().item() <= TOL_MEAN, f"call {call}"


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
