"""The synthetic input recipe (paged_kv_cache_forward_gb300/workloads.py) on the
CPU: each configuration has the shapes, ranges and structure the design states
(pool sizes, distinct physical pages, NaN poison where nothing may read, K
scaled for the batched decode), and a seed fixes every bit."""

import math

import pytest
import torch

from paged_kv_cache_forward_gb300 import workloads as W


def _isnan(t):
    return torch.isnan(t.float())


def _structure(b, pool_factor=1.5):
    """Distinct physical pages per used slot, padded entries on the poison page,
    NaN exactly on unused pages and tail slots; returns the pages in use."""
    P = b.page_size
    pages = []
    for s, L in enumerate(b.seq_lens.tolist()):
        npg = (L + P - 1) // P
        row = b.block_table[s].tolist()
        pages += row[:npg]
        assert all(p == b.poison_page for p in row[npg:])
        if L % P:
            last = row[npg - 1]
            assert _isnan(b.k_cache[last, L % P:]).all() and _isnan(b.v_cache[last, L % P:]).all()
            assert not _isnan(b.k_cache[last, :L % P]).any() and not _isnan(b.v_cache[last, :L % P]).any()
    assert len(set(pages)) == len(pages) and b.poison_page not in pages
    used = torch.zeros(b.num_blocks, dtype=torch.bool)
    used[pages] = True
    assert _isnan(b.k_cache[~used]).all() and _isnan(b.v_cache[~used]).all()
    assert b.query_start_loc[0] == 0 and b.query_start_loc[-1] == b.num_tokens
    assert not _isnan(b.q).any()
    return pages


def test_tiny_decode():
    b = W.tiny_decode(0)
    assert (b.num_seqs, b.num_tokens, b.num_q_heads, b.num_kv_heads, b.head_dim) == (1, 1, 4, 1, 64)
    assert b.seq_lens.tolist() == [256] and b.num_blocks == 64 and b.max_pages == 16
    assert b.scale == 1.0 / 8.0
    _structure(b)


@pytest.mark.parametrize("ctx", [1024, 8192])
def test_llama_decode(ctx):
    b = W.llama_decode(ctx, seed=0)
    assert (b.num_seqs, b.num_tokens, b.num_q_heads, b.num_kv_heads, b.head_dim) == (1, 1, 32, 8, 128)
    assert b.seq_lens.tolist() == [ctx] and b.max_pages == ctx // 16
    assert b.num_blocks == math.ceil(1.5 * ctx / 16)  # pool 1.5x the need
    assert abs(b.scale - 1.0 / math.sqrt(128)) < 1e-7
    _structure(b)


def test_batched_decode_ranges_and_k_scale():
    b = W.batched_decode(seed=0)
    L = b.seq_lens.tolist()
    assert b.num_seqs == 64 and b.q_lens() == [1] * 64 and all(512 <= x <= 8192 for x in L)
    pages = _structure(b)
    k = b.k_cache[pages].float()
    v = b.v_cache[pages].float()
    k, v = k[~torch.isnan(k)], v[~torch.isnan(v)]  # (the last pages' tail slots are poison)
    assert 0.45 < k.std().item() < 0.55 and 0.95 < v.std().item() < 1.05  # K x 0.5, V ~ N(0, 1)


def test_varlen_prefill_ranges():
    b = W.varlen_prefill(seed=0, poison=True)
    n, L = b.q_lens(), b.seq_lens.tolist()
    assert b.num_seqs == 8
    assert all(128 <= a <= 2048 for a in n) and all(0 <= c - a <= 4096 for a, c in zip(n, L))
    _structure(b)


def test_mixed_layout():
    b = W.mixed_batch(seed=0)
    n, L = b.q_lens(), b.seq_lens.tolist()
    assert n == [512] * 4 + [1] * 61
    assert L[:4] == [512] * 4 and all(1024 <= x <= 16384 for x in L[4:64]) and L[64] == 131072


def test_seed_fixes_every_bit():
    a, b, c = W.tiny_decode(3), W.tiny_decode(3), W.tiny_decode(4)
    for name in ("q", "k_cache", "v_cache", "block_table"):
        x, y, z = getattr(a, name), getattr(b, name), getattr(c, name)
        if x.dtype == torch.bfloat16:
            x, y, z = (t.view(torch.int16) for t in (x, y, z))
        assert torch.equal(x, y)
        assert not torch.equal(x, z)
