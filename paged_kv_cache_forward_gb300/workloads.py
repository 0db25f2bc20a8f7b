"""Seeded synthetic inputs for paged attention.

This module only *draws* inputs.  It holds none of the attention arithmetic and
imports neither the CUDA binding nor the CPU oracle, so both sides can be fed the
same bits from it.

Layout of one batch (all tensors on the CPU; the caller moves them):

  q               [T, Hq, D]           bf16   T = sum of new-query lengths n_b
  k_cache/v_cache [NB, P, Hkv, D]      bf16   P = page size (16); one token of one
                                              KV head is D contiguous values
  block_table     [B, max_pages]       int32  logical page -> physical page
  seq_lens        [B]                  int32  L_b = cached prefix + new tokens
  query_start_loc [B + 1]              int32  exclusive prefix sum of n_b

The n_b new queries of sequence b are its last n_b positions (bottom-right causal
alignment): query i of b sits at absolute position L_b - n_b + i.

Draw order for ``make_batch`` with ``torch.Generator('cpu').manual_seed(seed)``
(lengths are drawn first by the config helpers, from the same generator):
  1. ``randperm(NB)`` -- physical pages; the first sum(ceil(L_b/P)) go to the
     sequences in order, the next one is the poison page (padded block-table
     entries point at it), the rest stay unused.
  2. q: ``randn(T, Hq, D)`` in fp32, rounded to bf16 (round-to-nearest-even).
  3. k_cache then v_cache: ``randn`` in fp32 in chunks of ``_CHUNK_PAGES`` pages,
     times ``k_scale`` for K, rounded to bf16.
  4. Poison (``poison=True``): unused pages, the poison page and the slots past
     L_b in each sequence's last page are set to NaN.  A kernel that reads any of
     them without masking turns the output NaN instead of faulting.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

PAGE_SIZE = 16
_CHUNK_PAGES = 4096
BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass
class Batch:
    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    scale: float
    poison_page: int
    seed: int

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_cache.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def page_size(self) -> int:
        return int(self.k_cache.shape[1])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def q_lens(self) -> List[int]:
        qsl = self.query_start_loc.tolist()
        return [qsl[i + 1] - qsl[i] for i in range(len(qsl) - 1)]

    def kv_bytes(self) -> int:
        """Bytes of K and V the batch's context covers (each token once per KV head)."""
        per_token = 2 * self.num_kv_heads * self.head_dim * 2
        return int(self.seq_lens.to(torch.int64).sum().item()) * per_token

    def causal_pairs(self) -> int:
        """Number of visible (query token, key) pairs, summed over sequences."""
        total = 0
        for n, L in zip(self.q_lens(), self.seq_lens.tolist()):
            prefix = L - n
            total += n * prefix + n * (n + 1) // 2
        return total

    def to(self, device) -> "Batch":
        return dataclasses.replace(
            self,
            q=self.q.to(device),
            k_cache=self.k_cache.to(device),
            v_cache=self.v_cache.to(device),
            block_table=self.block_table.to(device),
            seq_lens=self.seq_lens.to(device),
            query_start_loc=self.query_start_loc.to(device),
        )


def _randn_bf16(g: torch.Generator, shape, mult: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x.to(torch.bfloat16)


def _pool_randn(g: torch.Generator, nb: int, page: int, hkv: int, d: int, mult: float) -> torch.Tensor:
    out = torch.empty((nb, page, hkv, d), dtype=torch.bfloat16)
    for s in range(0, nb, _CHUNK_PAGES):
        e = min(nb, s + _CHUNK_PAGES)
        out[s:e] = _randn_bf16(g, (e - s, page, hkv, d), mult)
    return out


def make_batch(
    q_lens: Sequence[int],
    seq_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    *,
    seed: int,
    g: Optional[torch.Generator] = None,
    page_size: int = PAGE_SIZE,
    k_scale: float = 1.0,
    pool_factor: float = 1.5,
    pool_pages: Optional[int] = None,
    max_pages: Optional[int] = None,
    scale: Optional[float] = None,
    poison: bool = True,
    name: str = "custom",
) -> Batch:
    """Draw one batch.  ``q_lens[b] <= seq_lens[b]`` (the new tokens are the last ones)."""
    assert len(q_lens) == len(seq_lens)
    for n, L in zip(q_lens, seq_lens):
        if not (0 <= n <= L):
            raise ValueError(f"need 0 <= q_len <= seq_len, got {n}, {L}")
    if g is None:
        g = torch.Generator().manual_seed(seed)
    B = len(seq_lens)
    pages_per_seq = [(L + page_size - 1) // page_size for L in seq_lens]
    need = sum(pages_per_seq)
    if max_pages is None:
        max_pages = max([1] + pages_per_seq)
    if max(pages_per_seq + [0]) > max_pages:
        raise ValueError("max_pages smaller than a sequence's page count")
    if pool_pages is None:
        pool_pages = max(int(math.ceil(pool_factor * need)), need + 1)
    nb = pool_pages
    if nb < need + 1:
        raise ValueError("pool needs at least one spare page for the poison page")

    perm = torch.randperm(nb, generator=g)
    poison_page = int(perm[need].item())
    bt = torch.full((B, max_pages), poison_page, dtype=torch.int32)
    cur = 0
    for b, npg in enumerate(pages_per_seq):
        bt[b, :npg] = perm[cur:cur + npg].to(torch.int32)
        cur += npg

    T = sum(q_lens)
    q = _randn_bf16(g, (T, num_q_heads, head_dim))
    k_cache = _pool_randn(g, nb, page_size, num_kv_heads, head_dim, k_scale)
    v_cache = _pool_randn(g, nb, page_size, num_kv_heads, head_dim, 1.0)

    if poison:
        used = torch.zeros(nb, dtype=torch.bool)
        used[perm[:need]] = True
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
        k_cache[~used] = nan
        v_cache[~used] = nan
        for b, L in enumerate(seq_lens):
            if L % page_size:
                last = int(bt[b, pages_per_seq[b] - 1])
                k_cache[last, L % page_size:] = nan
                v_cache[last, L % page_size:] = nan

    qsl = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        qsl[1:] = torch.cumsum(torch.tensor(list(q_lens), dtype=torch.int64), 0).to(torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return Batch(
        name=name,
        q=q,
        k_cache=k_cache,
        v_cache=v_cache,
        block_table=bt,
        seq_lens=torch.tensor(list(seq_lens), dtype=torch.int32),
        query_start_loc=qsl,
        scale=float(scale),
        poison_page=poison_page,
        seed=seed,
    )


def _uniform_ints(g: torch.Generator, lo: int, hi: int, n: int) -> List[int]:
    """n integers uniform on [lo, hi], both ends included."""
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# --------------------------------------------------------------------------
# The five workloads.  Llama-3.1-8B contributes only its attention shape
# (32 query heads, 8 KV heads, head_dim 128); no weights are involved.
# --------------------------------------------------------------------------

LLAMA = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


def tiny_decode(seed: int = 0, poison: bool = True) -> Batch:
    """1 sequence, 1 new token, GQA 4 (4 query heads / 1 KV head), head_dim 64,
    context 256 in 16 pages drawn from a 64-page pool, scale 1/sqrt(64)."""
    return make_batch([1], [256], 4, 1, 64, seed=seed, pool_pages=64, max_pages=16,
                      scale=1.0 / 8.0, poison=poison, name="tiny_decode")


def llama_decode(ctx: int, seed: int = 0, poison: bool = True) -> Batch:
    """Single-stream decode at one context length (1024, 8192 or 32768)."""
    return make_batch([1], [ctx], **LLAMA, seed=seed, max_pages=ctx // PAGE_SIZE,
                      poison=poison, name=f"llama_decode_{ctx}")


def batched_decode(seed: int = 0, batch: int = 64, lo: int = 512, hi: int = 8192,
                   poison: bool = True) -> Batch:
    """64 decode sequences, context uniform on [512, 8192], K scaled by 0.5."""
    g = torch.Generator().manual_seed(seed)
    lens = _uniform_ints(g, lo, hi, batch)
    return make_batch([1] * batch, lens, **LLAMA, seed=seed, g=g, k_scale=0.5,
                      max_pages=(hi + PAGE_SIZE - 1) // PAGE_SIZE, poison=poison,
                      name="batched_decode")


def varlen_prefill(seed: int = 0, batch: int = 8, n_lo: int = 128, n_hi: int = 2048,
                   p_lo: int = 0, p_hi: int = 4096, poison: bool = True) -> Batch:
    """Causal chunked prefill: new lengths U[128, 2048], cached prefixes U[0, 4096]."""
    g = torch.Generator().manual_seed(seed)
    n = _uniform_ints(g, n_lo, n_hi, batch)
    p = _uniform_ints(g, p_lo, p_hi, batch)
    lens = [a + b for a, b in zip(n, p)]
    return make_batch(n, lens, **LLAMA, seed=seed, g=g,
                      max_pages=(n_hi + p_hi + PAGE_SIZE - 1) // PAGE_SIZE, poison=poison,
                      name="varlen_prefill")


def mixed_batch(seed: int = 0, n_prefill: int = 4, prefill_len: int = 512, n_decode: int = 60,
                d_lo: int = 1024, d_hi: int = 16384, long_ctx: int = 131072,
                poison: bool = True) -> Batch:
    """4 prefill sequences of 512 new tokens (no cached prefix), 60 decode sequences
    with context U[1024, 16384], and one decode sequence at 131072, in that order."""
    g = torch.Generator().manual_seed(seed)
    dl = _uniform_ints(g, d_lo, d_hi, n_decode)
    q_lens = [prefill_len] * n_prefill + [1] * n_decode + ([1] if long_ctx else [])
    lens = [prefill_len] * n_prefill + dl + ([long_ctx] if long_ctx else [])
    bound = max(lens)
    return make_batch(q_lens, lens, **LLAMA, seed=seed, g=g,
                      max_pages=(bound + PAGE_SIZE - 1) // PAGE_SIZE, poison=poison,
                      name="mixed")


def spec_decode(seed: int = 0, batch: int = 16, n: int = 4, lo: int = 2048, hi: int = 8192,
                poison: bool = True) -> Batch:
    """Speculative decoding: 16 sequences each verifying 4 draft tokens, context
    uniform on [2048, 8192] (the 4 new tokens included)."""
    g = torch.Generator().manual_seed(seed)
    lens = _uniform_ints(g, lo, hi, batch)
    return make_batch([n] * batch, lens, **LLAMA, seed=seed, g=g,
                      max_pages=(hi + PAGE_SIZE - 1) // PAGE_SIZE, poison=poison, name="spec_decode")


CONFIGS = {
    "tiny_decode": tiny_decode,
    "llama_decode_1024": lambda seed=0, poison=True: llama_decode(1024, seed, poison),
    "llama_decode_8192": lambda seed=0, poison=True: llama_decode(8192, seed, poison),
    "llama_decode_32768": lambda seed=0, poison=True: llama_decode(32768, seed, poison),
    "batched_decode": batched_decode,
    "varlen_prefill": varlen_prefill,
    "mixed": mixed_batch,
    "spec_decode": spec_decode,
}


# --------------------------------------------------------------------------
# Structured inputs for the exact indexing / masking checks.
# --------------------------------------------------------------------------

def position_code(t: int, head_dim: int) -> torch.Tensor:
    """Mixed-radix one-hot code of logical position t: the D channels form 4 groups
    of D/4; group k holds a one-hot of base-(D/4) digit k of t.  Values are 0/1, so
    the code is exact in bf16.  D=64 covers 16**4 positions, D=128 covers 32**4."""
    r = head_dim // 4
    if t < 0 or t >= r ** 4:
        raise ValueError("position out of range for the code")
    v = torch.zeros(head_dim, dtype=torch.float32)
    x = t
    for k in range(4):
        v[k * r + (x % r)] = 1.0
        x //= r
    return v


def decode_position_code(v: torch.Tensor) -> int:
    """Inverse of position_code for an exact code (raises if v is not one)."""
    head_dim = v.shape[-1]
    r = head_dim // 4
    t = 0
    for k in reversed(range(4)):
        grp = v[k * r:(k + 1) * r]
        nz = torch.nonzero(grp).flatten().tolist()
        if len(nz) != 1 or float(grp[nz[0]]) != 1.0:
            raise ValueError("not a position code")
        t = t * r + nz[0]
    return t


def logical_to_physical(block_table_row: torch.Tensor, j: int, page_size: int = PAGE_SIZE):
    """(physical page, slot) that holds logical position j of one sequence."""
    return int(block_table_row[j // page_size]), j % page_size


def position_codes(pos: torch.Tensor, head_dim: int) -> torch.Tensor:
    """Vectorised position_code: [N] int64 positions -> [N, D] float32 codes."""
    r = head_dim // 4
    pos = pos.to(torch.int64)
    if pos.numel() and (int(pos.min()) < 0 or int(pos.max()) >= r ** 4):
        raise ValueError("position out of range for the code")
    out = torch.zeros((pos.numel(), head_dim), dtype=torch.float32)
    x = pos.clone()
    rows = torch.arange(pos.numel())
    for k in range(4):
        out[rows, k * r + (x % r)] = 1.0
        x = x // r
    return out


def spike_batch(q_lens, seq_lens, num_q_heads, num_kv_heads, head_dim, *, seed: int,
                spikes: int = 4, max_pages=None, pool_factor: float = 1.5):
    """Inputs whose exact output is known by construction (scale 1).

    V at logical position j is position_code(j).  K is zero except "spikes": for
    every (sequence, KV head, head-in-group g) there are up to ``spikes`` positions
    f_1 < f_2 < ... with K[f_k][g] = 100 * k, f_1 <= the sequence's first query
    position.  Query head h = hk * G + g is the one-hot e_g.  Its scores are 100*k
    at the spikes it can see and 0 elsewhere; the largest visible one beats every
    other by >= 100 (2^-144 after exp2, which flushes to 0 in fp32), so the exact
    output is position_code(largest f_k <= p).  A key read from the wrong page or
    slot, a wrong head, or a future key leaking through the causal mask changes
    the output bits.

    Returns (batch, expected) with expected [T, Hq] int64 positions.
    """
    b = make_batch(q_lens, seq_lens, num_q_heads, num_kv_heads, head_dim, seed=seed,
                   max_pages=max_pages, pool_factor=pool_factor, scale=1.0, poison=True)
    G = num_q_heads // num_kv_heads
    if G > head_dim:
        raise ValueError("one channel per head in a group is needed")
    g = torch.Generator().manual_seed(seed + 7919)
    P = b.page_size
    used = torch.zeros(b.num_blocks, dtype=torch.bool)
    nan = float("nan")
    # clean data everywhere a sequence has a page; tails and unused pages stay NaN
    for s, L in enumerate(seq_lens):
        npg = (L + P - 1) // P
        pages = b.block_table[s, :npg].to(torch.int64)
        used[pages] = True
        j = torch.arange(L)
        codes = position_codes(j, head_dim).to(torch.bfloat16)
        pg = pages[j // P]
        sl = j % P
        b.k_cache[pg, sl] = torch.zeros((L, num_kv_heads, head_dim), dtype=torch.bfloat16)
        b.v_cache[pg, sl] = codes[:, None, :].expand(L, num_kv_heads, head_dim)
    b.q.zero_()
    for h in range(num_q_heads):
        b.q[:, h, h % G] = 1.0
    T = sum(q_lens)
    expected = torch.full((T, num_q_heads), -1, dtype=torch.int64)
    qsl = b.query_start_loc.tolist()
    for s, (n, L) in enumerate(zip(q_lens, seq_lens)):
        if n == 0:
            continue
        first = L - n
        for hk in range(num_kv_heads):
            for gi in range(G):
                f1 = int(torch.randint(0, first + 1, (1,), generator=g))
                rest = torch.randperm(L - f1 - 1, generator=g)[: spikes - 1] + f1 + 1 if L - f1 - 1 > 0 else \
                    torch.zeros(0, dtype=torch.int64)
                fs = [f1] + sorted(rest.tolist())
                for k, f in enumerate(fs):
                    page = int(b.block_table[s, f // P])
                    b.k_cache[page, f % P, hk, gi] = 100.0 * (k + 1)
                ft = torch.tensor(fs)
                for i in range(n):
                    p = first + i
                    expected[qsl[s] + i, hk * G + gi] = int(ft[ft <= p].max())
    del nan, used
    return b, expected
