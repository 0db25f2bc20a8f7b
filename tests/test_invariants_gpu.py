"""GPU invariants that the definition of attention fixes, independent of the oracle.

out = softmax(scale * q K^T) V (the GPU programming guide page, section
"Decomposing multi-head attention (MHA)") is a convex combination of the visible
V rows: its weights are non-negative and sum to 1.  So

  * V rows all equal to c (per KV head) give out = c, whatever the scores;
  * V = 1 everywhere gives out = 1;
  * a causal chunked prefill of n new tokens over a cached prefix of P keys
    gives, for its token i, what a decode call with context P + i + 1 gives
    ("Flash Attention in Triton" on the same page: future tokens get -inf).

The kernels round P to bf16 for the P V product and sum the same rounded P into
the normaliser l, so the first two hold to fp32 rounding of a ratio whose two
sums hold the same terms; written back as bf16 the output must then equal c (or
1) bit for bit.  That holds through every path: one split, splits merged through
the workspace, a thread-block cluster merge, the prefill kernel (several KV
tiles, diagonal tiles, ragged tails), and a mixed batch.
"""

import pytest
import torch

import oracle
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import assert_close, run

pytestmark = pytest.mark.gpu


def _fill_visible_v(b: W.Batch, rows_per_head: torch.Tensor) -> W.Batch:
    """V of every visible position of every sequence set to rows_per_head[kv_head]
    (bf16); everything else (unused pages, the poison page, tail slots) keeps its
    NaN poison."""
    v = b.v_cache.clone()
    P = b.page_size
    for s, L in enumerate(b.seq_lens.tolist()):
        npg = (L + P - 1) // P
        pages = b.block_table[s, :npg].long()
        if npg > 1:
            v[pages[:-1]] = rows_per_head.to(torch.bfloat16)[None, None]
        if npg:
            last = L - (npg - 1) * P
            v[pages[-1], :last] = rows_per_head.to(torch.bfloat16)[None]
    return W.Batch(**{**b.__dict__, "v_cache": v})


def _expected(b: W.Batch, rows_per_head: torch.Tensor) -> torch.Tensor:
    G = b.num_q_heads // b.num_kv_heads
    per_q_head = rows_per_head.to(torch.bfloat16).repeat_interleave(G, dim=0)  # [Hq, D]
    return per_q_head[None].expand(b.num_tokens, -1, -1)


def _assert_bits_equal(got: torch.Tensor, want: torch.Tensor, what: str):
    assert torch.isfinite(got.float()).all(), f"{what}: non-finite output"
    bad = (got.view(torch.int16) != want.contiguous().view(torch.int16))
    if bad.any():
        diff = (got.double() - want.double()).abs()
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.numel()} elements differ from the constant "
                             f"(max |diff| {diff.max().item():.3e})")


# (name, q_lens, seq_lens, Hq, Hkv, D, options)
CONSTANT_V_CASES = [
    ("decode_one_split", [1, 1, 1], [100, 1000, 37], 32, 8, 128, dict(kv_chunk=1024)),
    ("decode_workspace_merge", [1, 1, 1, 1], [2000, 1000, 37, 1], 32, 8, 128, dict(kv_chunk=64)),
    ("decode_cluster", [1, 1, 1], [3000, 17, 700], 32, 8, 128, dict(decode_cluster=4)),
    ("decode_table", [1, 1, 1], [5000, 1, 300], 32, 8, 128, {}),
    ("multi_token_decode", [3, 4, 2], [500, 77, 2], 32, 8, 128, dict(kv_chunk=128)),
    ("prefill", [300, 129, 77], [300, 529, 110], 32, 8, 128, {}),
    ("prefill_d64_g8", [200, 45], [260, 45], 16, 2, 64, {}),
    ("prefill_d256", [150, 33], [350, 33], 16, 4, 256, {}),
    ("mixed", [40, 1, 1, 17, 1, 2, 1], [40, 700, 1, 100, 3000, 2, 16], 32, 8, 128, {}),
    ("mixed_mqa", [70, 1, 1], [90, 2000, 5], 8, 1, 128, {}),
]


@pytest.mark.parametrize("case", CONSTANT_V_CASES, ids=[c[0] for c in CONSTANT_V_CASES])
def test_constant_v_rows_give_the_constant(case):
    name, ql, sl, Hq, Hkv, D, opts = case
    b = W.make_batch(ql, sl, Hq, Hkv, D, seed=len(name) + D)
    c = torch.randn(Hkv, D, generator=torch.Generator().manual_seed(7))
    bc = _fill_visible_v(b, c)
    got = run(bc, **opts)
    _assert_bits_equal(got, _expected(bc, c), f"constant V, {name}")


def test_constant_v_mixed_full_size():
    """The mixed workload (4 x 512 prefill, 60 decode up to 16384 keys, one decode
    at 131072 keys) with constant V rows: every output row is the constant."""
    b = W.mixed_batch(seed=0)
    c = torch.randn(b.num_kv_heads, b.head_dim, generator=torch.Generator().manual_seed(8))
    v = torch.empty_like(b.v_cache)
    v[:] = c.to(torch.bfloat16)[None, None]  # K keeps its NaN poison on unused pages and tail slots
    bc = W.Batch(**{**b.__dict__, "v_cache": v})
    got = run(bc)
    _assert_bits_equal(got, _expected(bc, c), "constant V, mixed full size")


# (name, q_lens, seq_lens, Hq, Hkv, D, options)
ONES_CASES = [
    ("llama_decode_splits", [1, 1], [8192, 333], 32, 8, 128, dict(kv_chunk=256)),
    ("llama_cluster", [1], [4096], 32, 8, 128, dict(decode_cluster=8)),
    ("mqa_g1", [1, 9, 1, 33], [333, 9, 17, 50], 8, 8, 128, {}),
    ("g8_d64", [1, 2, 130], [1500, 40, 130], 16, 2, 64, {}),
    ("g32_d128", [1, 1, 64], [2000, 3, 100], 32, 1, 128, {}),
    ("d256", [1, 3, 200], [900, 50, 260], 32, 8, 256, {}),
    ("prefill_long", [1000, 257], [3000, 257], 32, 8, 128, {}),
]


@pytest.mark.parametrize("case", ONES_CASES, ids=[c[0] for c in ONES_CASES])
def test_v_ones_give_one(case):
    """V = 1: the weights of every row sum to 1, so every output element is 1."""
    name, ql, sl, Hq, Hkv, D, opts = case
    b = W.make_batch(ql, sl, Hq, Hkv, D, seed=3 * D + Hq)
    ones = torch.ones(Hkv, D)
    bo = _fill_visible_v(b, ones)
    got = run(bo, **opts)
    _assert_bits_equal(got, torch.ones_like(got), f"V = 1, {name}")


# (prefix P, new tokens n, Hq, Hkv, D)
CHUNK_CASES = [
    (0, 300, 32, 8, 128),     # prefill from scratch, ~10 query tiles of 32 tokens
    (37, 129, 32, 8, 128),    # prefix not on a page or tile boundary
    (500, 70, 32, 8, 128),
    (1000, 5, 32, 8, 128),    # short chunk: still the prefill kernel (n > 4 at G = 4)
    (200, 3, 32, 8, 128),     # multi-token decode path against single-token decode
    (64, 90, 16, 2, 64),
    (130, 40, 16, 4, 256),
]


@pytest.mark.parametrize("case", CHUNK_CASES, ids=[f"P{c[0]}_n{c[1]}_G{c[2] // c[3]}_D{c[4]}" for c in CHUNK_CASES])
def test_chunked_prefill_equals_decode_calls(case):
    """A chunk of n new tokens over a cached prefix of P keys, computed in one
    call, against n single-token decode calls over the same pages with contexts
    P + 1, ..., P + n (each decode sequence shares the chunk's block-table row).
    Both are held to the oracle's tolerance and to each other."""
    P, n, Hq, Hkv, D = case
    a = W.make_batch([n], [P + n], Hq, Hkv, D, seed=P + n + D)
    chunk = run(a)
    # n decode sequences: token i of the chunk, context P + i + 1, same pages
    bt = a.block_table.expand(n, -1).contiguous()
    dec = W.Batch(**{**a.__dict__, "block_table": bt,
                     "seq_lens": torch.arange(P + 1, P + n + 1, dtype=torch.int32),
                     "query_start_loc": torch.arange(n + 1, dtype=torch.int32)})
    calls = run(dec)
    ref = oracle.batch_attention(a)
    assert_close(chunk, ref, f"chunk P={P} n={n} vs oracle")
    assert_close(calls, ref, f"decode calls P={P} n={n} vs oracle")
    assert_close(chunk, calls.double().numpy(), f"chunk vs decode calls P={P} n={n}")
