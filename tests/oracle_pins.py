"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each ``pin_*`` takes a loaded oracle library (the real one, or a mutated copy in
test_oracle_mutants.py) and raises AssertionError if the oracle disagrees with
the fact.  None of them re-types the oracle's formula: they use closed forms,
invariances of the definition, or a library routine on a special case
(torch's scaled_dot_product_attention with an identity block table).

Definition pinned: out = softmax(Q K^T * scale) V, from the GPU programming guide
page ("From megabytes to megawatts ...", section "Decomposing multi-head
attention (MHA)"), masked causally ("Flash Attention in Triton", future tokens
get -inf) with bottom-right alignment, read through a block table (the paged KV
cache of the Triton unified-attention page, section "Why is switching the card so
hard").
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from paged_kv_cache_forward_gb300 import workloads as W

NAN = float("nan")


def _run(lib, b: W.Batch):
    return oracle.batch_attention(b, lib=lib)


def _bf(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _set_logical(b: W.Batch, seq: int, j: int, kv_head: int, k=None, v=None):
    page, slot = W.logical_to_physical(b.block_table[seq], j, b.page_size)
    if k is not None:
        b.k_cache[page, slot, kv_head] = _bf(k)
    if v is not None:
        b.v_cache[page, slot, kv_head] = _bf(v)


def _q_lens(b):
    return b.q_lens()


# ---------------------------------------------------------------- closed forms

def pin_single_key(lib):
    """L = 1: the only key has weight exactly 1, so out is V[0] exactly."""
    for D, Hq, Hkv in ((64, 4, 1), (128, 8, 2)):
        b = W.make_batch([1], [1], Hq, Hkv, D, seed=11, pool_pages=5, max_pages=3)
        out = _run(lib, b)
        page = int(b.block_table[0, 0])
        for h in range(Hq):
            want = b.v_cache[page, 0, h // (Hq // Hkv)].to(torch.float64).numpy()
            assert np.array_equal(out[0, h], want), "single key must return its V row"


def pin_constant_v(lib):
    """Every visible V row equal to c: out = c for any weights (they sum to 1)."""
    b = W.make_batch([3, 1, 5], [40, 17, 5], 8, 2, 64, seed=12, pool_factor=2.0, max_pages=4)
    c = torch.randn(2, 64, generator=torch.Generator().manual_seed(5))
    for s, L in enumerate(b.seq_lens.tolist()):
        for j in range(L):
            for hk in range(2):
                _set_logical(b, s, j, hk, v=c[hk])
    out = _run(lib, b)
    cb = _bf(c).to(torch.float64).numpy()
    for t in range(b.num_tokens):
        for h in range(8):
            assert np.max(np.abs(out[t, h] - cb[h // 4])) < 1e-12


def pin_zero_keys_mean(lib):
    """K = 0: all visible scores are 0, so out is the plain mean of the visible V
    rows; the count of visible rows (p + 1 with p = L - n + i) pins the causal
    alignment of every query of a chunked prefill."""
    q_lens, seq_lens = [4, 1, 3], [9, 6, 3]
    b = W.make_batch(q_lens, seq_lens, 4, 2, 64, seed=13, pool_factor=2.0, max_pages=2)
    for s, L in enumerate(seq_lens):
        for j in range(L):
            for hk in range(2):
                _set_logical(b, s, j, hk, k=torch.zeros(64))
    out = _run(lib, b)
    t = 0
    for s, (n, L) in enumerate(zip(q_lens, seq_lens)):
        for i in range(n):
            p = L - n + i
            for h in range(4):
                hk = h // 2
                rows = []
                for j in range(p + 1):
                    page, slot = W.logical_to_physical(b.block_table[s], j)
                    rows.append(b.v_cache[page, slot, hk].to(torch.float64))
                want = torch.stack(rows).mean(0).numpy()
                assert np.max(np.abs(out[t, h] - want)) < 1e-12, (s, i, h)
            t += 1


def pin_two_key_logistic(lib):
    """Two keys with scores 0 and scale*a: w_1 = 1 / (1 + exp(-scale*a)); the
    scale enters once, multiplied into the dot product."""
    D = 64
    scale = 0.37
    a = 5.0
    b = W.make_batch([1], [2], 1, 1, D, seed=14, pool_pages=3, max_pages=1, scale=scale)
    e0 = torch.zeros(D)
    e0[3] = 1.0
    b.q[0, 0] = _bf(e0)
    k1 = torch.zeros(D)
    k1[3] = a
    _set_logical(b, 0, 0, 0, k=torch.zeros(D), v=torch.zeros(D))
    v1 = torch.zeros(D)
    v1[7] = 1.0
    _set_logical(b, 0, 1, 0, k=k1, v=v1)
    out = _run(lib, b)
    s = float(np.float32(scale)) * a
    w1 = 1.0 / (1.0 + math.exp(-s))
    assert abs(out[0, 0, 7] - w1) < 1e-14
    assert np.max(np.abs(np.delete(out[0, 0], 7))) == 0.0


def pin_large_logits(lib):
    """Scores near 1e3 (exp overflows without the max subtraction): the result
    is the same as with the scores shifted down, since softmax is shift-invariant."""
    D = 64
    b = W.make_batch([1], [3], 1, 1, D, seed=15, pool_pages=2, max_pages=1, scale=1.0)
    q = torch.zeros(D)
    q[0] = 32.0
    b.q[0, 0] = _bf(q)
    vals = [1000.0, 992.0, 976.0]  # q.k = 32 * k0; k0 = 31.25, 31, 30.5 are exact in bf16
    vs = torch.eye(D)[:3]
    for j, v in enumerate(vals):
        k = torch.zeros(D)
        k[0] = v / 32.0
        _set_logical(b, 0, j, 0, k=k, v=vs[j])
    out = _run(lib, b)
    e = np.exp(np.array(vals) - vals[0])
    w = e / e.sum()
    assert np.all(np.isfinite(out)), "softmax must not overflow"
    assert np.max(np.abs(out[0, 0, :3] - w)) < 1e-14


def pin_lse(lib):
    """The log-sum-exp of a row's scores, lse = log(sum_j exp(s_j)) over the
    visible keys, in closed form: K = 0 gives log(p + 1) (every visible score is
    0; the count pins the causal alignment); two keys with scores 0 and s give
    log(1 + e^s); scores near 1e3 give 1000 + log(1 + e^-8 + e^-24) (no overflow,
    and the row max is added back)."""
    q_lens, seq_lens = [4, 1], [9, 6]
    b = W.make_batch(q_lens, seq_lens, 4, 2, 64, seed=23, pool_factor=2.0, max_pages=1)
    for s_, L in enumerate(seq_lens):
        for j in range(L):
            for hk in range(2):
                _set_logical(b, s_, j, hk, k=torch.zeros(64))
    _, lse = oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, b.query_start_loc, b.scale,
                              return_lse=True, lib=lib)
    t = 0
    for n, L in zip(q_lens, seq_lens):
        for i in range(n):
            assert np.max(np.abs(lse[t] - math.log(L - n + i + 1))) < 1e-13, (t, lse[t])
            t += 1
    D, scale, a = 64, 0.37, 5.0
    b = W.make_batch([1], [2], 1, 1, D, seed=24, pool_pages=3, max_pages=1, scale=scale)
    e0 = torch.zeros(D)
    e0[3] = 1.0
    b.q[0, 0] = _bf(e0)
    k1 = torch.zeros(D)
    k1[3] = a
    _set_logical(b, 0, 0, 0, k=torch.zeros(D))
    _set_logical(b, 0, 1, 0, k=k1)
    _, lse = oracle.attention_rows(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, b.query_start_loc,
                                   b.scale, rows=[(0, 0)], return_lse=True, lib=lib)
    s1 = float(np.float32(scale)) * a
    assert abs(lse[0] - math.log1p(math.exp(s1))) < 1e-14, lse[0]
    b = W.make_batch([1], [3], 1, 1, D, seed=25, pool_pages=2, max_pages=1, scale=1.0)
    q = torch.zeros(D)
    q[0] = 32.0
    b.q[0, 0] = _bf(q)
    for j, v in enumerate([1000.0, 992.0, 976.0]):
        k = torch.zeros(D)
        k[0] = v / 32.0
        _set_logical(b, 0, j, 0, k=k)
    _, lse = oracle.attention_rows(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, b.query_start_loc,
                                   b.scale, rows=[(0, 0)], return_lse=True, lib=lib)
    want = 1000.0 + math.log1p(math.exp(-8.0) + math.exp(-24.0))
    assert abs(lse[0] - want) < 1e-12, (lse[0], want)


# ------------------------------------------------------------------ invariants

def pin_row_sums(lib):
    """Weights of every row are >= 0, sum to 1, and are 0 past position p."""
    q_lens, seq_lens = [5, 1], [21, 33]
    b = W.make_batch(q_lens, seq_lens, 8, 2, 64, seed=16, pool_factor=1.5, max_pages=3)
    t = 0
    for s, (n, L) in enumerate(zip(q_lens, seq_lens)):
        for i in range(n):
            p = L - n + i
            for h in range(8):
                w, _ = oracle.attention_weights(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens,
                                                b.query_start_loc, b.scale, t, h, lib=lib)
                assert abs(w.sum() - 1.0) < 1e-12
                assert np.all(w[: p + 1] > 0) and np.all(w[p + 1:] == 0)
            t += 1


def _rescatter(b: W.Batch, seed: int, pool_pages: int) -> W.Batch:
    """Same logical K/V, moved to a different random set of physical pages in a
    pool of another size (the unused pages poisoned with NaN)."""
    g = torch.Generator().manual_seed(seed)
    nb = pool_pages
    perm = torch.randperm(nb, generator=g)
    k = torch.full((nb,) + tuple(b.k_cache.shape[1:]), NAN, dtype=torch.bfloat16)
    v = k.clone()
    bt = torch.full_like(b.block_table, int(perm[-1]))
    cur = 0
    for s, L in enumerate(b.seq_lens.tolist()):
        for pg in range((L + b.page_size - 1) // b.page_size):
            src = int(b.block_table[s, pg])
            dst = int(perm[cur])
            cur += 1
            k[dst] = b.k_cache[src]
            v[dst] = b.v_cache[src]
            bt[s, pg] = dst
    assert cur < nb
    return W.Batch(name=b.name, q=b.q, k_cache=k, v_cache=v, block_table=bt, seq_lens=b.seq_lens,
                   query_start_loc=b.query_start_loc, scale=b.scale, poison_page=int(perm[-1]), seed=seed)


def pin_block_permutation(lib):
    """Output depends on the logical cache only: re-scattering the pages to other
    physical ids (and another pool size) changes nothing, bit for bit."""
    b = W.make_batch([3, 1, 2], [50, 37, 16], 8, 2, 64, seed=17, pool_factor=1.5, max_pages=4)
    out = _run(lib, b)
    b2 = _rescatter(b, seed=99, pool_pages=b.num_blocks + 7)
    out2 = _run(lib, b2)
    assert np.array_equal(out, out2)


def pin_causal_hiding(lib):
    """Changing K and V at positions after p leaves query p's row unchanged."""
    q_lens, seq_lens = [6], [20]
    b = W.make_batch(q_lens, seq_lens, 4, 1, 64, seed=18, pool_pages=4, max_pages=2)
    out = _run(lib, b)
    g = torch.Generator().manual_seed(3)
    for i in range(6):
        p = 20 - 6 + i
        b2 = W.Batch(**{**b.__dict__, "k_cache": b.k_cache.clone(), "v_cache": b.v_cache.clone()})
        for j in range(p + 1, 20):
            _set_logical(b2, 0, j, 0, k=torch.randn(64, generator=g) * 50, v=torch.randn(64, generator=g) * 50)
        out2 = _run(lib, b2)
        assert np.array_equal(out[i], out2[i]), i
        if i < 5:
            assert not np.array_equal(out[5], out2[5]) or p + 1 >= 20


def pin_position_code_spike(lib):
    """V holds mixed-radix one-hot codes of the logical position; K is zero except
    a large spike at one target position t*.  The softmax then puts all but
    ~exp(-40) of the weight on t*, so the output is the code of t*: this checks
    the page / slot / head addressing through a random block table."""
    D, Hq, Hkv = 64, 8, 2
    q_lens, seq_lens = [1, 4], [70, 45]
    b = W.make_batch(q_lens, seq_lens, Hq, Hkv, D, seed=19, pool_factor=2.0, max_pages=5, scale=1.0)
    beta = 8.0
    for s, L in enumerate(seq_lens):
        for j in range(L):
            for hk in range(Hkv):
                _set_logical(b, s, j, hk, k=torch.zeros(D), v=W.position_code(j, D))
    # query head h selects channel h; KV head hk holds a spike for channel h at t*(s, h)
    targets = {}
    t = 0
    for s, (n, L) in enumerate(zip(q_lens, seq_lens)):
        for i in range(n):
            for h in range(Hq):
                qv = torch.zeros(D)
                qv[h] = beta
                b.q[t, h] = _bf(qv)
            t += 1
    for s, (n, L) in enumerate(zip(q_lens, seq_lens)):
        first_visible = L - n  # the position the first new query sits at
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            tstar = (7 * h + 3 * s) % (first_visible + 1)
            targets[(s, h)] = tstar
            page, slot = W.logical_to_physical(b.block_table[s], tstar)
            kk = b.k_cache[page, slot, hk].to(torch.float32)
            kk[h] = beta
            b.k_cache[page, slot, hk] = _bf(kk)
    out = _run(lib, b)
    t = 0
    for s, (n, L) in enumerate(zip(q_lens, seq_lens)):
        for i in range(n):
            for h in range(Hq):
                want = W.position_code(targets[(s, h)], D).double().numpy()
                assert np.max(np.abs(out[t, h] - want)) < 1e-12, (s, i, h)
            t += 1


# ------------------------------------------------------ library special case

def _sdpa_reference(b: W.Batch, seq_start_pages):
    """torch SDPA in fp64 on the dense K/V of each sequence (identity block table:
    sequence s occupies pages seq_start_pages[s], +1, ...), with GQA by repeating
    each KV head over its group and an explicit bottom-right causal mask."""
    Hq, Hkv, D, P = b.num_q_heads, b.num_kv_heads, b.head_dim, b.page_size
    G = Hq // Hkv
    outs = []
    qsl = b.query_start_loc.tolist()
    for s, L in enumerate(b.seq_lens.tolist()):
        n = qsl[s + 1] - qsl[s]
        if n == 0:
            continue
        npg = (L + P - 1) // P
        p0 = seq_start_pages[s]
        K = b.k_cache[p0:p0 + npg].reshape(npg * P, Hkv, D)[:L].double()
        V = b.v_cache[p0:p0 + npg].reshape(npg * P, Hkv, D)[:L].double()
        K = K.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
        V = V.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
        Q = b.q[qsl[s]:qsl[s + 1]].double().permute(1, 0, 2)[None]
        i = torch.arange(n)[:, None]
        j = torch.arange(L)[None, :]
        mask = j <= (L - n + i)
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, attn_mask=mask, scale=float(np.float32(b.scale)))
        outs.append(o[0].permute(1, 0, 2))
    return torch.cat(outs).numpy()


def _identity_batch(q_lens, seq_lens, Hq, Hkv, D, seed, scale=None, k_mult=1.0):
    b = W.make_batch(q_lens, seq_lens, Hq, Hkv, D, seed=seed, pool_factor=1.0, scale=scale,
                     poison=True)
    starts, cur = [], 0
    bt = torch.full_like(b.block_table, b.num_blocks - 1)
    for s, L in enumerate(seq_lens):
        npg = (L + 15) // 16
        starts.append(cur)
        bt[s, :npg] = torch.arange(cur, cur + npg, dtype=torch.int32)
        cur += npg
    # fresh finite data on the used pages, NaN tails kept out of the dense slices
    g = torch.Generator().manual_seed(seed + 1000)
    k = torch.full_like(b.k_cache, NAN)
    v = torch.full_like(b.v_cache, NAN)
    k[:cur] = (torch.randn(k[:cur].shape, generator=g) * k_mult).to(torch.bfloat16)
    v[:cur] = torch.randn(v[:cur].shape, generator=g).to(torch.bfloat16)
    b2 = W.Batch(name="identity", q=b.q, k_cache=k, v_cache=v, block_table=bt, seq_lens=b.seq_lens,
                 query_start_loc=b.query_start_loc, scale=b.scale, poison_page=b.num_blocks - 1, seed=seed)
    return b2, starts


def pin_sdpa_identity_table(lib):
    """Identity block table: oracle equals torch SDPA (fp64, explicit mask)."""
    cases = [
        ([1], [1], 4, 1, 64),
        ([1], [37], 32, 8, 128),
        ([7, 1, 16, 2], [7, 30, 40, 2], 8, 2, 64),   # prefill without / with prefix, decode
        ([5, 3], [21, 64], 8, 8, 128),                 # G = 1
        ([2, 9], [33, 9], 16, 2, 64),                  # G = 8
    ]
    for k, (ql, sl, Hq, Hkv, D) in enumerate(cases):
        b, starts = _identity_batch(ql, sl, Hq, Hkv, D, seed=20 + k, k_mult=2.0)
        out = _run(lib, b)
        ref = _sdpa_reference(b, starts)
        assert out.shape == ref.shape
        assert np.max(np.abs(out - ref)) < 1e-12, (k, np.max(np.abs(out - ref)))


def pin_validation(lib):
    """Contract violations are rejected, not read out of bounds."""
    import ctypes
    b = W.make_batch([2], [10], 4, 1, 64, seed=21, pool_pages=3, max_pages=1)
    dims = dict(num_tokens=2, num_seqs=1, num_q_heads=4, num_kv_heads=1, head_dim=64, page_size=16,
                num_blocks=3, max_pages=1)
    ok = oracle.validate(b.block_table, b.seq_lens, b.query_start_loc, dims)
    assert ok == 0
    assert oracle.validate(b.block_table, torch.tensor([1], dtype=torch.int32), b.query_start_loc, dims) == 3
    assert oracle.validate(b.block_table, torch.tensor([17], dtype=torch.int32), b.query_start_loc, dims) == 3
    assert oracle.validate(torch.tensor([[3]], dtype=torch.int32), b.seq_lens, b.query_start_loc, dims) == 4
    assert oracle.validate(b.block_table, b.seq_lens, torch.tensor([0, 3], dtype=torch.int32), dims) == 2
    del ctypes


# --------------------------------------------------------- paged cache write

def _slots_for(b: W.Batch, seq: int, positions):
    return [int(b.block_table[seq, j // b.page_size]) * b.page_size + j % b.page_size for j in positions]


def pin_cache_write_round_trip(lib):
    """Writing new tokens through the slot mapping puts them where the block table
    says logical position j lives (torch indexing of [NB, P, Hkv, D]); negative
    slots leave the cache untouched; slots past the pool are refused."""
    b = W.make_batch([3, 1, 5], [40, 17, 5], 8, 2, 64, seed=41, pool_factor=2.0, max_pages=4)
    g = torch.Generator().manual_seed(9)
    qsl = b.query_start_loc.tolist()
    T = b.num_tokens
    k_new = torch.randn(T, 2, 64, generator=g).to(torch.bfloat16)
    v_new = torch.randn(T, 2, 64, generator=g).to(torch.bfloat16)
    slots = []
    for s_, (n, L) in enumerate(zip(b.q_lens(), b.seq_lens.tolist())):
        slots += _slots_for(b, s_, range(L - n, L))
    slots[1] = -1  # padding: no write
    kc, vc = oracle.cache_write(k_new, v_new, torch.tensor(slots), b.k_cache, b.v_cache, lib=lib)
    want_k = b.k_cache.clone()
    want_v = b.v_cache.clone()
    for t, sl in enumerate(slots):
        if sl >= 0:
            want_k[sl // 16, sl % 16] = k_new[t]
            want_v[sl // 16, sl % 16] = v_new[t]
    bits = lambda x: x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(kc, bits(want_k)) and np.array_equal(vc, bits(want_v))
    bad = torch.tensor([0] * (T - 1) + [b.num_blocks * 16])
    try:
        oracle.cache_write(k_new, v_new, bad, b.k_cache, b.v_cache, lib=lib)
    except oracle.OracleError:
        pass
    else:
        raise AssertionError("a slot past the pool was accepted")


ALL_PINS = [
    pin_single_key,
    pin_constant_v,
    pin_zero_keys_mean,
    pin_two_key_logistic,
    pin_large_logits,
    pin_lse,
    pin_row_sums,
    pin_block_permutation,
    pin_causal_hiding,
    pin_position_code_spike,
    pin_sdpa_identity_table,
    pin_cache_write_round_trip,
]
