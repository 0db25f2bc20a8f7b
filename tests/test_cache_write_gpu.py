"""pa_cache_write against the oracle's scatter (bit-exact), and write-then-attend:
K/V written by the kernel into the cache give the attention the oracle computes
from the oracle-written cache."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_forward_gb300 as pa
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, run

pytestmark = pytest.mark.gpu


def _new_rows(b: W.Batch, seed: int):
    """K/V rows for every new token of the batch and their slots (bottom-right:
    token i of sequence s sits at position L - n + i)."""
    g = torch.Generator().manual_seed(seed)
    T, Hkv, D = b.num_tokens, b.num_kv_heads, b.head_dim
    k_new = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    slots = []
    for s, (n, L) in enumerate(zip(b.q_lens(), b.seq_lens.tolist())):
        for j in range(L - n, L):
            slots.append(int(b.block_table[s, j // 16]) * 16 + j % 16)
    return k_new, v_new, torch.tensor(slots, dtype=torch.int64)


def _bits(x):
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("Hkv,D", [(8, 128), (1, 64), (2, 64)])
def test_cache_write_bit_exact(Hkv, D):
    ensure_built()
    b = W.make_batch([5, 1, 40, 1], [70, 33, 40, 2], 4 * Hkv, Hkv, D, seed=90 + D)
    k_new, v_new, slots = _new_rows(b, 3)
    slots[2] = -1  # padding
    want_k, want_v = oracle.cache_write(k_new, v_new, slots, b.k_cache, b.v_cache)
    kc, vc = b.k_cache.cuda(), b.v_cache.cuda()
    pa.cache_write(k_new.cuda(), v_new.cuda(), slots.cuda(), kc, vc)
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    assert np.array_equal(_bits(kc), want_k) and np.array_equal(_bits(vc), want_v)


def test_write_then_attend():
    ensure_built()
    b = W.make_batch([37, 1, 3, 1], [300, 900, 64, 17], 32, 8, 128, seed=95)
    k_new, v_new, slots = _new_rows(b, 4)
    # the oracle's cache after the write, and the attention over it
    k_ref, v_ref = oracle.cache_write(k_new, v_new, slots, b.k_cache, b.v_cache)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    ref = oracle.attention(b.q, as_bf16(k_ref), as_bf16(v_ref), b.block_table, b.seq_lens, b.query_start_loc,
                           b.scale)
    d = b.to("cuda")
    pa.cache_write(k_new.cuda(), v_new.cuda(), slots.cuda(), d.k_cache, d.v_cache)
    out = torch.full_like(d.q, float("nan"))
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale)
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    assert_close(out.cpu(), ref, "write then attend")


def test_cache_write_bad_slot_flags_and_skips():
    ensure_built()
    b = W.make_batch([2], [20], 8, 2, 64, seed=96)
    k_new, v_new, slots = _new_rows(b, 5)
    slots[1] = b.num_blocks * 16  # one past the pool
    kc, vc = b.k_cache.cuda(), b.v_cache.cuda()
    pa.cache_write(k_new.cuda(), v_new.cuda(), slots.cuda(), kc, vc)
    torch.cuda.synchronize()
    assert pa.device_error() == 1
    # the valid row was still written
    s0 = int(slots[0])
    assert torch.equal(kc[s0 // 16, s0 % 16].cpu(), k_new[0])
