"""GPU parity: the CUDA path against the fp64 oracle on the same seeded inputs.

Bar (the problem's stated tolerance): max-abs error <= 1.5e-2 and mean-abs
error <= 2e-3 over all compared elements; block-table indexing and causal
masking bit-exact (position-code spikes); block permutation, causal hiding and
graph replay bit-exact against the same kernel.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_forward_gb300 as pa
from paged_kv_cache_forward_gb300 import workloads as W

from gpu_util import assert_close, errors, run, sample_rows

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------ the five configs

def test_tiny_decode_all_seeds():
    for seed in range(5):
        b = W.tiny_decode(seed)
        assert_close(run(b), oracle.batch_attention(b), f"tiny seed {seed}")


# Seeds 0-4 of every configuration (the full-size prefill and mixed batches on
# sampled rows).
SEEDS = range(5)


@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("ctx", [1024, 8192, 32768])
def test_llama_decode(ctx, seed):
    b = W.llama_decode(ctx, seed=seed)
    assert_close(run(b), oracle.batch_attention(b), f"llama decode {ctx} seed {seed}")


@pytest.mark.parametrize("seed", SEEDS)
def test_batched_decode(seed):
    b = W.batched_decode(seed=seed)
    assert_close(run(b), oracle.batch_attention(b), f"batched decode seed {seed}")


@pytest.mark.parametrize("seed", SEEDS)
def test_varlen_prefill_full_size_sampled(seed):
    b = W.varlen_prefill(seed=seed)
    got = run(b)
    rows = sample_rows(b, 600, seed=1 + seed)
    ref = oracle.batch_attention(b, rows=rows)
    sel = torch.stack([got[t, h] for t, h in rows])
    assert_close(sel, ref, f"varlen prefill seed {seed} (sampled rows)")


@pytest.mark.parametrize("seed", SEEDS)
def test_mixed_full_size_sampled_in_graph(seed):
    b = W.mixed_batch(seed=seed)
    d = b.to("cuda")
    out = torch.full_like(d.q, float("nan"))
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale)
    g.replay()
    torch.cuda.synchronize()
    assert pa.device_error(s) == 0
    got = out.cpu()
    assert torch.isfinite(got.float()).all()
    rows = sample_rows(b, 400, seed=2 + seed)
    T = b.num_tokens
    rows += [(T - 1, h) for h in range(b.num_q_heads)]  # the 131072-context decode row
    rows = sorted(set(rows))
    ref = oracle.batch_attention(b, rows=rows)
    sel = torch.stack([got[t, h] for t, h in rows])
    assert_close(sel, ref, f"mixed seed {seed} (sampled rows)")


# --------------------------------------------------- smaller full comparisons

def test_prefill_small_full():
    for seed in range(3):
        g = torch.Generator().manual_seed(100 + seed)
        B = 4
        n = torch.randint(2, 200, (B,), generator=g).tolist()
        p = torch.randint(0, 300, (B,), generator=g).tolist()
        b = W.make_batch(n, [a + c for a, c in zip(n, p)], 32, 8, 128, seed=seed)
        assert_close(run(b), oracle.batch_attention(b), f"prefill small seed {seed}")


def test_mixed_small_full():
    q_lens = [40, 1, 1, 17, 1, 2, 1]
    seq_lens = [40, 700, 1, 100, 3000, 2, 16]
    b = W.make_batch(q_lens, seq_lens, 32, 8, 128, seed=5)
    assert_close(run(b), oracle.batch_attention(b), "mixed small")


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 1, 64), (8, 8, 128), (16, 2, 64), (32, 1, 128), (12, 4, 128),
                                      (64, 2, 64), (32, 8, 256), (16, 2, 256), (8, 8, 256)])
def test_head_shapes(Hq, Hkv, D):
    q_lens = [1, 9, 1, 33]
    seq_lens = [333, 9, 17, 50]
    b = W.make_batch(q_lens, seq_lens, Hq, Hkv, D, seed=Hq + Hkv + D)
    assert_close(run(b), oracle.batch_attention(b), f"heads {Hq}/{Hkv} D {D}")


@pytest.mark.parametrize("chunk", [16, 48, 256, 4096])
def test_split_invariance(chunk):
    b = W.make_batch([1, 1, 1, 5], [2000, 1, 777, 300], 32, 8, 128, seed=9, max_pages=128)
    ref = oracle.batch_attention(b)
    got = run(b, kv_chunk=chunk)
    assert_close(got, ref, f"kv_chunk {chunk}")
    whole = run(b, kv_chunk=128 * 16)
    mx, _ = errors(got, whole.double().numpy())
    assert mx <= 2 * 2 ** -8 * 4, mx  # a few bf16 ulps of |out| <= ~4


@pytest.mark.parametrize("warps,stages", [(4, 2), (4, 3), (4, 4), (8, 2), (8, 3), (12, 2)])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_variants(warps, stages, D):
    """Every decode variant (warps per CTA, pipeline depth) against the oracle;
    the depth does not change which warp reads which page, so variants with the
    same warp count are bit-identical.  Multi-token rows and a split merge included."""
    b = W.make_batch([1, 1, 3, 1, 2], [4000, 1, 777, 65, 2500], 32, 8, D, seed=31 + D, max_pages=256)
    ref = oracle.batch_attention(b)
    for chunk in (0, 256):
        got = run(b, kv_chunk=chunk, decode_stages=stages, decode_warps=warps)
        assert_close(got, ref, f"{warps}x{stages} D {D} chunk {chunk}")
        base = run(b, kv_chunk=chunk, decode_stages=2, decode_warps=warps)
        assert torch.equal(got.view(torch.int16), base.view(torch.int16)), (warps, stages, chunk)


@pytest.mark.parametrize("cluster", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("warps,stages", [(4, 2), (8, 3), (12, 2)])
def test_decode_cluster_mode(cluster, warps, stages):
    """Splits merged in distributed shared memory: the pages of each (sequence,
    KV head) dealt round-robin to a cluster of CTAs.  Sequences with fewer pages
    than the cluster has CTAs leave some CTAs without keys; multi-token rows
    included."""
    b = W.make_batch([1, 1, 3, 1, 2, 1], [4000, 1, 777, 65, 2500, 16], 32, 8, 128, seed=41 + cluster,
                     max_pages=256)
    ref = oracle.batch_attention(b)
    got = run(b, decode_cluster=cluster, decode_warps=warps, decode_stages=stages)
    assert_close(got, ref, f"cluster {cluster} {warps}x{stages}")


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 1, 128), (16, 2, 64), (8, 8, 128)])
def test_decode_cluster_mode_head_shapes(Hq, Hkv, D):
    b = W.make_batch([1, 1, 1], [3000, 129, 40], Hq, Hkv, D, seed=Hq * Hkv + D, max_pages=200)
    ref = oracle.batch_attention(b)
    for cluster in (4, 16):
        assert_close(run(b, decode_cluster=cluster), ref, f"heads {Hq}/{Hkv} D {D} cluster {cluster}")


def test_decode_cluster_spikes_bit_exact():
    b, exp = W.spike_batch([1, 2, 1, 4], [40, 1000, 5000, 17], 32, 8, 128, seed=27, max_pages=320)
    want = _codes(exp, 128)
    for cluster in (2, 7, 16):
        got = run(b, decode_cluster=cluster)
        bad = (got.view(torch.int16) != want.view(torch.int16)).any(-1)
        assert not bad.any(), (cluster, torch.nonzero(bad)[:5].tolist())


def test_head_dim_256():
    """D = 256: one query tile per prefill CTA (its O takes 256 TMEM columns),
    single-stage K/V rings, P V with N = 256; the 4-warp decode variants.  Several
    KV tiles, a ragged tail, a sequence end mid-page, multi-token decode rows."""
    b = W.make_batch([200, 1, 130, 2, 1], [700, 1500, 130, 333, 17], 32, 8, 256, seed=256, max_pages=100)
    ref = oracle.batch_attention(b)
    assert_close(run(b), ref, "D 256")
    for st in (2, 3):
        assert_close(run(b, decode_stages=st, decode_warps=4), ref, f"D 256 4x{st}")
    assert_close(run(b, decode_cluster=4), ref, "D 256 cluster 4")
    assert_close(run(b, kv_chunk=64), ref, "D 256 64-key splits")


def test_head_dim_256_spikes_bit_exact():
    b, exp = W.spike_batch([1, 37, 2, 130], [5000, 300, 90, 130], 16, 4, 256, seed=28, max_pages=320)
    want = _codes(exp, 256)
    got = run(b)
    bad = (got.view(torch.int16) != want.view(torch.int16)).any(-1)
    assert not bad.any(), torch.nonzero(bad)[:5].tolist()


# ------------------------------------------------------------------- edge cases

def test_edge_lengths():
    # single key, exact page multiples, one-token prefill, n == L prefill, empty sequences
    q_lens = [1, 1, 0, 2, 16, 1, 0, 3]
    seq_lens = [1, 16, 0, 2, 16, 32, 5, 3]
    b = W.make_batch(q_lens, seq_lens, 8, 2, 128, seed=11, max_pages=4)
    got = run(b)
    assert_close(got, oracle.batch_attention(b), "edge lengths")
    # the single-key row is V[0] exactly
    page = int(b.block_table[0, 0])
    for h in range(8):
        assert torch.equal(got[0, h], b.v_cache[page, 0, h // 4])


def test_empty_and_zero_token_batches():
    b = W.make_batch([0, 0], [5, 0], 8, 2, 128, seed=12)
    d = b.to("cuda")
    out = torch.zeros_like(d.q)
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale)
    torch.cuda.synchronize()
    assert out.numel() == 0


def test_max_pages_exact_fit_and_poison_neighbours():
    # every page of the table used, NaN everywhere else in the pool
    b = W.make_batch([1, 4], [64 * 16, 64 * 16], 32, 8, 128, seed=13, max_pages=64, pool_factor=1.05)
    assert_close(run(b), oracle.batch_attention(b), "exact fit")


# ------------------------------------------------------------- bit-exact checks

def _codes(expected, D):
    T, Hq = expected.shape
    return W.position_codes(expected.flatten(), D).reshape(T, Hq, D).to(torch.bfloat16)


@pytest.mark.parametrize("case", ["decode", "prefill", "mixed", "tiny"])
def test_position_code_spikes_bit_exact(case):
    if case == "decode":
        b, exp = W.spike_batch([1] * 6, [1, 15, 16, 17, 1000, 5000], 32, 8, 128, seed=21)
    elif case == "prefill":
        b, exp = W.spike_batch([37, 128, 5], [37, 300, 70], 32, 8, 128, seed=22)
    elif case == "mixed":
        b, exp = W.spike_batch([64, 1, 1, 9], [64, 20000, 33, 40], 32, 8, 128, seed=23)
    else:
        b, exp = W.spike_batch([1], [256], 4, 1, 64, seed=24, max_pages=16)
    got = run(b)
    want = _codes(exp, b.head_dim)
    bad = (got.view(torch.int16) != want.view(torch.int16)).any(-1)
    assert not bad.any(), f"{int(bad.sum())} rows differ, first {torch.nonzero(bad)[:5].tolist()}"


def test_spikes_bit_exact_across_splits():
    b, exp = W.spike_batch([1, 1, 3], [4000, 257, 900], 32, 8, 128, seed=25, max_pages=256)
    want = _codes(exp, 128)
    for chunk in (16, 64, 1024, 4096):
        got = run(b, kv_chunk=chunk)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), chunk


def _rescatter(b: W.Batch, seed: int, extra: int) -> W.Batch:
    g = torch.Generator().manual_seed(seed)
    nb = b.num_blocks + extra
    perm = torch.randperm(nb, generator=g)
    k = torch.full((nb,) + tuple(b.k_cache.shape[1:]), float("nan"), dtype=torch.bfloat16)
    v = k.clone()
    bt = torch.full_like(b.block_table, int(perm[-1]))
    cur = 0
    for s, L in enumerate(b.seq_lens.tolist()):
        for pg in range((L + 15) // 16):
            src, dst = int(b.block_table[s, pg]), int(perm[cur])
            cur += 1
            k[dst] = b.k_cache[src]
            v[dst] = b.v_cache[src]
            bt[s, pg] = dst
    return W.Batch(name=b.name, q=b.q, k_cache=k, v_cache=v, block_table=bt, seq_lens=b.seq_lens,
                   query_start_loc=b.query_start_loc, scale=b.scale, poison_page=int(perm[-1]), seed=seed)


def test_block_permutation_bit_exact():
    b = W.make_batch([1, 23, 1, 2], [900, 100, 33, 2], 32, 8, 128, seed=31)
    got = run(b)
    got2 = run(_rescatter(b, 77, 13))
    assert torch.equal(got.view(torch.int16), got2.view(torch.int16))


def test_causal_hiding_bit_exact():
    n, L = 70, 200
    b = W.make_batch([n], [L], 32, 8, 128, seed=32)
    got = run(b)
    k2, v2 = b.k_cache.clone(), b.v_cache.clone()
    g = torch.Generator().manual_seed(4)
    cut = L - n + 30  # query 30 sits at this position
    for j in range(cut + 1, L):
        page, slot = W.logical_to_physical(b.block_table[0], j)
        k2[page, slot] = (torch.randn(8, 128, generator=g) * 30).to(torch.bfloat16)
        v2[page, slot] = (torch.randn(8, 128, generator=g) * 30).to(torch.bfloat16)
    b2 = W.Batch(**{**b.__dict__, "k_cache": k2, "v_cache": v2})
    got2 = run(b2)
    assert torch.equal(got[:31].view(torch.int16), got2[:31].view(torch.int16))
    assert not torch.equal(got[31:], got2[31:])


# ------------------------------------------------------------------ CUDA graphs

def test_graph_replay_new_contents_bit_exact():
    """Capture once; replay with other lengths, tables and query split of the
    same shapes: the static grid must give the eager results bit for bit."""
    Hq, Hkv, D, mp = 32, 8, 128, 64
    b1 = W.make_batch([1, 6, 1, 1], [700, 40, 1000, 5], Hq, Hkv, D, seed=41, max_pages=mp, pool_pages=200)
    b2 = W.make_batch([3, 1, 4, 1], [3, 1024, 4, 600], Hq, Hkv, D, seed=42, max_pages=mp, pool_pages=200)
    e1, e2 = run(b1), run(b2)
    d = b1.to("cuda")
    out = torch.full_like(d.q, float("nan"))
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b1.scale)
    for b, e in ((b1, e1), (b2, e2), (b1, e1)):
        for name in ("q", "k_cache", "v_cache", "block_table", "seq_lens", "query_start_loc"):
            getattr(d, name).copy_(getattr(b, name))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.cpu().view(torch.int16), e.view(torch.int16))


def test_mixed_batch_is_ordered_on_the_callers_stream():
    """The prefill kernel of a mixed batch runs on the library's side stream:
    work enqueued on the caller's stream before the call (new q) must be seen by
    it, and work enqueued after (a copy of out) must see its rows."""
    b = W.make_batch([300, 1, 1, 150, 1], [800, 2000, 40, 150, 9000], 32, 8, 128, seed=79)
    g = torch.Generator().manual_seed(80)
    q2 = torch.randn(b.q.shape, generator=g).to(torch.bfloat16)
    d = b.to("cuda")
    q2d = q2.to("cuda")
    out = torch.full_like(d.q, float("nan"))
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)  # keep the stream busy so that ordering matters
        d.q.copy_(q2d)
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale,
                   stream=s)
        res = out.clone()
    s.synchronize()
    assert pa.device_error(s) == 0
    b.q = q2
    assert_close(res.cpu(), oracle.batch_attention(b), "mixed batch on a user stream")


def test_capture_without_prepare_is_refused():
    b = W.make_batch([1], [50000], 32, 8, 128, seed=43, max_pages=4096, pool_pages=3200)
    d = b.to("cuda")
    out = torch.empty_like(d.q)
    s = torch.cuda.Stream()  # a fresh stream has no workspace
    g = torch.cuda.CUDAGraph()
    with pytest.raises(pa.PagedAttnError) as e:
        with torch.cuda.graph(g, stream=s):
            pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out,
                       scale=b.scale, kv_chunk=512)
    assert e.value.status == 3
    torch.cuda.synchronize()


# --------------------------------------------------------- device-side checks

def test_bad_block_id_sets_error_word_without_fault():
    b = W.make_batch([1, 2], [40, 30], 8, 2, 128, seed=51)
    b.block_table[0, 1] = b.num_blocks + 5  # out of range: the kernels skip it
    run(b, check_errors=False)
    assert pa.device_error() == 1
    assert pa.device_error() == 0  # cleared
    # the context is still usable
    b2 = W.tiny_decode(0)
    assert_close(run(b2), oracle.batch_attention(b2), "after error")


def test_prefill_wait_that_runs_out_aborts_cleanly():
    """A wait of the prefill kernel that runs out (the test option withholds one
    K tile; no memory is touched that a normal call would not touch): the
    kernel gives up after its bounded wait, records error 4 and returns; the
    context stays usable and the next call is exact (its item counters are back
    at zero)."""
    b = W.make_batch([300, 200, 1], [300, 400, 900], 32, 8, 128, seed=81)
    run(b, check_errors=False, test_stall_prefill=1)
    assert pa.device_error() == 4
    assert pa.device_error() == 0  # cleared
    b2 = W.make_batch([100, 64, 1], [500, 64, 300], 32, 8, 128, seed=82)
    assert_close(run(b2), oracle.batch_attention(b2), "after a prefill abort")


def test_query_longer_than_context_flagged():
    b = W.make_batch([3], [3], 8, 2, 128, seed=52)
    b.seq_lens[0] = 2  # 3 new tokens but 2 keys: contract violation
    got = run(b, check_errors=False)
    assert pa.device_error() == 3
    assert torch.isfinite(got.float()).all()


@pytest.mark.parametrize("D", [64, 128, 256])
def test_prefill_items_beyond_the_grid(D):
    """Several times more (tile pair, KV head) items than SMs: each persistent
    prefill CTA takes items one after another from the item counter.  Sampled
    rows against the oracle; two eager calls and a graph of three forwards,
    replayed twice, bit-exact (the counter returns to zero after every launch)."""
    n = [700, 1500, 300, 1200, 900, 2000]
    p = [0, 333, 1000, 17, 2500, 64]
    b = W.make_batch(n, [a + c for a, c in zip(n, p)], 32, 8, D, seed=77)
    e1 = run(b)
    e2 = run(b)
    assert torch.equal(e1.view(torch.int16), e2.view(torch.int16))
    rows = sample_rows(b, 300, seed=7)
    ref = oracle.batch_attention(b, rows=rows)
    assert_close(torch.stack([e1[t, h] for t, h in rows]), ref, f"prefill items beyond the grid, D {D}")
    d = b.to("cuda")
    outs = [torch.full_like(d.q, float("nan")) for _ in range(3)]
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for o in outs:
            pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, o, scale=b.scale)
    for _ in range(2):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pa.device_error(s) == 0
        for o in outs:
            assert torch.equal(o.cpu().view(torch.int16), e1.view(torch.int16))


def test_prefill_query_longer_than_context_between_good_sequences():
    """A prefill-sized query longer than its sequence (a contract violation) is
    flagged and its rows written as zeros, without disturbing the items of the
    sequences around it."""
    b = W.make_batch([200, 150, 300], [400, 150, 300], 32, 8, 128, seed=78)
    qsl = b.query_start_loc.tolist()
    rows = [(t, h) for t in list(range(qsl[0], qsl[1], 7)) + list(range(qsl[2], qsl[3], 7)) for h in (0, 13, 31)]
    ref = oracle.batch_attention(b, rows=rows)  # (the oracle refuses the broken batch below)
    b.seq_lens[1] = 100  # 150 new tokens but 100 keys
    got = run(b, check_errors=False)
    assert pa.device_error() == 3
    assert torch.equal(got[qsl[1]:qsl[2]].float(), torch.zeros_like(got[qsl[1]:qsl[2]].float()))
    assert_close(torch.stack([got[t, h] for t, h in rows]), ref, "good sequences around a bad one")


def test_many_splits_long_context():
    # 1024 splits of 64 keys for each of two 65536-key sequences: the split merge
    # reads a long run of partials and the ticket counters see many arrivals
    b = W.make_batch([1, 1], [65536, 65536], 32, 8, 128, seed=71, max_pages=4096)
    got = run(b, kv_chunk=64)
    rows = [(0, h) for h in range(32)] + [(1, h) for h in range(0, 32, 3)]
    ref = oracle.batch_attention(b, rows=rows)
    assert_close(torch.stack([got[t, h] for t, h in rows]), ref, "65536 x 2, 64-key splits")


# ------------------------------------------------- multi-token (speculative) decode

@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 8, 128), (16, 2, 64), (12, 4, 128)])
def test_multi_token_decode(Hq, Hkv, D):
    """Sequences with 1 .. 16/G new tokens take the decode path (rows = tokens x
    G heads, each row masked at its own position); one more token goes to the
    prefill kernel."""
    G = Hq // Hkv
    nmax = 16 // G
    q_lens = list(range(1, nmax + 1)) + [nmax, nmax + 1]
    seq_lens = [300 + 37 * i for i in range(nmax)] + [5000, 700]
    b = W.make_batch(q_lens, seq_lens, Hq, Hkv, D, seed=80 + G, max_pages=320)
    ref = oracle.batch_attention(b)
    for chunk in (0, 64):
        assert_close(run(b, kv_chunk=chunk), ref, f"G {G} chunk {chunk}")


def test_multi_token_decode_spikes_bit_exact():
    b, exp = W.spike_batch([2, 3, 4, 1, 4], [40, 1000, 5000, 17, 4], 32, 8, 128, seed=26, max_pages=320)
    want = _codes(exp, 128)
    for chunk in (0, 64, 1024):
        got = run(b, kv_chunk=chunk)
        bad = (got.view(torch.int16) != want.view(torch.int16)).any(-1)
        assert not bad.any(), (chunk, torch.nonzero(bad)[:5].tolist())


def test_workspace_reuse_across_growing_batches():
    """Calls on one stream whose split-ticket counter area grows (more sequences)
    after calls that wrote partials: the counters must never land on bytes that
    held partials."""
    s = torch.cuda.Stream()
    for B in (2, 9, 40, 3, 64):
        g = torch.Generator().manual_seed(200 + B)
        lens = torch.randint(600, 3000, (B,), generator=g).tolist()
        b = W.make_batch([1] * B, lens, 32, 8, 128, seed=200 + B, max_pages=200)
        d = b.to("cuda")
        out = torch.full_like(d.q, float("nan"))
        torch.cuda.synchronize()  # the inputs were made on the default stream
        with torch.cuda.stream(s):
            pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out,
                       scale=b.scale, kv_chunk=256)
        s.synchronize()
        assert pa.device_error(s) == 0
        assert_close(out.cpu(), oracle.batch_attention(b), f"B {B}")


def test_launch_only_writes_one_kernels_rows():
    """pa_options.launch_only (timing and tests): 1 launches only the decode
    kernel, 2 only the prefill kernel; each writes exactly its own rows, equal
    bit for bit to the rows of a full call."""
    b = W.make_batch([300, 1, 3, 150, 1], [800, 2000, 40, 150, 9000], 32, 8, 128, seed=81)
    full = run(b)
    qsl = b.query_start_loc.tolist()
    decode_rows = torch.zeros(b.num_tokens, dtype=torch.bool)
    for s, n in enumerate(b.q_lens()):
        if 1 <= n <= 4:  # G = 4: up to 4 new tokens take the decode kernel
            decode_rows[qsl[s]:qsl[s + 1]] = True
    d = b.to("cuda")
    for only, mine in ((1, decode_rows), (2, ~decode_rows)):
        out = torch.full_like(d.q, float("nan"))
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale,
                   launch_only=only)
        torch.cuda.synchronize()
        assert pa.device_error() == 0
        got = out.cpu()
        assert torch.equal(got[mine].view(torch.int16), full[mine].view(torch.int16)), only
        assert torch.isnan(got[~mine].float()).all(), only


def test_back_to_back_calls_see_the_previous_output():
    """Two decode calls in a row on one stream, the second reading the first's
    output as its queries: the second call (scheduled early by programmatic
    dependent launch) must not read q before the first call has written it.
    Eager and in a CUDA graph, against the same two calls with a device
    synchronisation between them."""
    b = W.llama_decode(8192, seed=82)
    d = b.to("cuda")
    pl = pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens)
    assert pl["decode_ctas"] <= torch.cuda.get_device_properties(0).multi_processor_count
    mid = torch.empty_like(d.q)
    ref = torch.empty_like(d.q)
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, mid, scale=b.scale)
    torch.cuda.synchronize()
    pa.forward(mid, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, ref, scale=b.scale)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s)
    torch.cuda.synchronize()
    for mode in ("eager", "graph"):
        mid.fill_(float("nan"))
        out = torch.full_like(d.q, float("nan"))

        def two_calls():
            pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, mid, scale=b.scale,
                       stream=s)
            pa.forward(mid, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale,
                       stream=s)

        if mode == "eager":
            with torch.cuda.stream(s):
                two_calls()
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                two_calls()
            mid.fill_(float("nan"))
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                g.replay()
        s.synchronize()
        assert pa.device_error(s) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), mode


_EARLY_CASES = {
    "decode_1024": lambda: W.llama_decode(1024, seed=84),
    "decode_8192": lambda: W.llama_decode(8192, seed=85),
    "multi_token": lambda: W.make_batch([4, 1, 2, 3], [700, 5000, 33, 1600], 32, 8, 128, seed=86),
    "batched": lambda: W.batched_decode(seed=87),
    "mixed": lambda: W.make_batch([300, 1, 3, 150, 1], [800, 2000, 40, 150, 9000], 32, 8, 128, seed=88),
    "d64": lambda: W.make_batch([1, 1, 1], [3000, 17, 900], 16, 4, 64, seed=89),
    "d256": lambda: W.make_batch([1, 2, 1], [2500, 700, 31], 16, 2, 256, seed=90),
}


@pytest.mark.parametrize("case", sorted(_EARLY_CASES))
@pytest.mark.parametrize("cluster", [0, 4])
def test_early_metadata_is_bit_identical(case, cluster):
    """pa_options.early_metadata only moves the metadata loads (and L2 prefetches
    of the first KV pages) ahead of the wait for the previous kernel: the output
    equals, bit for bit, that of the same call without it, in every path (single
    and split decode, cluster merge, multi-token decode, the mixed batch)."""
    b = _EARLY_CASES[case]()
    d = b.to("cuda")
    outs = []
    for early in (0, 1):
        out = torch.full_like(d.q, float("nan"))
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out, scale=b.scale,
                   decode_cluster=cluster, early_metadata=early)
        torch.cuda.synchronize()
        assert pa.device_error() == 0
        outs.append(out.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), case
    assert_close(outs[1], oracle.batch_attention(b), f"{case} cluster {cluster}")


def test_early_metadata_still_waits_for_q_and_kv_written_just_before():
    """With early_metadata the second of two back-to-back decode calls reads its
    metadata while the first may still run, but q and KV values still wait:
    here the first call's output is the second call's q and also overwrites the
    first four rows of a KV page that the second call reads (one of the pages it
    prefetches).  Eager and in a CUDA graph, the result equals the two calls with
    a device synchronisation between them."""
    b = W.llama_decode(8192, seed=91)
    d = b.to("cuda")
    pl = pa.plan_for(d.q, d.k_cache, d.block_table, d.seq_lens)
    assert pl["decode_ctas"] <= torch.cuda.get_device_properties(0).multi_processor_count
    X = int(b.block_table[0, 0])  # the first page of split 0's first warp
    orig = d.k_cache[X].clone()
    mid = torch.empty_like(d.q)
    spill = d.k_cache[X, 0:4].view(1, b.num_q_heads, b.head_dim)  # 4 tokens x Hkv x D = Hq x D

    def two_calls(early, stream=None):
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, spill, scale=b.scale,
                   stream=stream, early_metadata=early)
        pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, mid, scale=b.scale,
                   stream=stream, early_metadata=early)

    def reset():
        d.k_cache[X].copy_(orig)
        torch.cuda.synchronize()

    reset()
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, spill, scale=b.scale)
    torch.cuda.synchronize()
    ref = torch.empty_like(d.q)
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, ref, scale=b.scale)
    torch.cuda.synchronize()
    # the first call changed a page the second one reads, so a stale read would show
    reset()
    unchanged = torch.empty_like(d.q)
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, unchanged, scale=b.scale)
    torch.cuda.synchronize()
    assert not torch.equal(unchanged.view(torch.int16), ref.view(torch.int16))
    s = torch.cuda.Stream()
    pa.prepare(d.q, d.k_cache, d.block_table, d.seq_lens, stream=s)
    torch.cuda.synchronize()
    for mode in ("eager", "graph"):
        reset()
        mid.fill_(float("nan"))
        torch.cuda.synchronize()
        if mode == "eager":
            with torch.cuda.stream(s):
                two_calls(1, s)
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                two_calls(1, s)
            reset()
            mid.fill_(float("nan"))
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                g.replay()
        s.synchronize()
        assert pa.device_error(s) == 0
        assert torch.equal(mid.view(torch.int16), ref.view(torch.int16)), mode
    reset()
