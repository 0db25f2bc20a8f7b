"""The C-ABI library without a GPU: it loads, exports every declared symbol,
plans on the host, and rejects bad arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

from paged_kv_cache_forward_gb300 import binding as B
from paged_kv_cache_forward_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_what_binding_knows():
    assert declared_functions() == sorted(B.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for st in range(5):
        assert lib.pa_status_string(st)
    assert lib.pa_version() == 102


def llama_dims(**kw):
    d = dict(num_tokens=1, num_blocks=3072, num_seqs=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
             page_size=16, max_pages=2048)
    d.update(kw)
    return B.Dims(**d)


def test_plan_shapes_only(lib):
    p = B.plan(llama_dims())
    assert p["kv_chunk"] % 16 == 0
    assert p["splits"] == -(-2048 * 16 // p["kv_chunk"])
    assert p["decode_ctas"] == 1 * 8 * 1 * p["splits"]
    assert p["workspace_bytes"] >= 256
    # static grid: a plan never depends on anything but the dims
    assert B.plan(llama_dims()) == p


def test_plan_forced_chunk(lib):
    p = B.plan(llama_dims(), kv_chunk=1024)
    assert p["kv_chunk"] == 1024 and p["splits"] == 32
    p = B.plan(llama_dims(), kv_chunk=1 << 20)
    assert p["splits"] == 1 and p["combine_ctas"] == 0


def test_plan_row_groups(lib):
    # G = 32 query heads per KV head: two decode row groups of 16
    p = B.plan(llama_dims(num_kv_heads=1))
    assert p["decode_ctas"] == 1 * 1 * 2 * p["splits"]


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), B.PA_ERR_UNSUPPORTED),
    (dict(head_dim=512), B.PA_ERR_UNSUPPORTED),
    (dict(page_size=32), B.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=30), B.PA_ERR_INVALID_ARG),
    (dict(num_kv_heads=0), B.PA_ERR_INVALID_ARG),
    (dict(num_blocks=0), B.PA_ERR_INVALID_ARG),
    (dict(max_pages=0), B.PA_ERR_INVALID_ARG),
    (dict(num_tokens=-1), B.PA_ERR_INVALID_ARG),
    (dict(num_q_heads=128, num_kv_heads=1), B.PA_ERR_UNSUPPORTED),
])
def test_plan_rejects(lib, kw, status):
    with pytest.raises(B.PagedAttnError) as e:
        B.plan(llama_dims(**kw))
    assert e.value.status == status
    assert lib.pa_last_error().decode()


DECODE_VARIANTS = [(4, 2), (4, 3), (4, 4), (8, 2), (8, 3), (12, 2)]  # (warps, stages)


def test_decode_variant_option(lib):
    p = B.plan(llama_dims())
    assert (p["decode_warps"], p["decode_stages"]) in DECODE_VARIANTS
    for w, st in DECODE_VARIANTS:
        p = B.plan(llama_dims(), decode_stages=st, decode_warps=w)
        assert (p["decode_warps"], p["decode_stages"]) == (w, st)
    # one field alone: the other takes its default (4 warps / 2 stages)
    assert B.plan(llama_dims(), decode_stages=3)["decode_warps"] == 4
    assert B.plan(llama_dims(), decode_warps=8)["decode_stages"] == 2
    for w, st in [(4, 1), (4, 5), (8, 4), (12, 3), (16, 2), (2, 2), (-4, 2)]:
        with pytest.raises(B.PagedAttnError) as e:
            B.plan(llama_dims(), decode_stages=st, decode_warps=w)
        assert e.value.status == B.PA_ERR_INVALID_ARG


def test_head_dim_256_plan(lib):
    p = B.plan(llama_dims(head_dim=256))
    assert (p["decode_warps"], p["decode_stages"]) in [(4, 2), (4, 3)]  # table variant mapped to a D=256 one
    # static prefill grid: T / (tiles per CTA x 32 tokens) + B CTAs per KV head
    assert B.plan(llama_dims(head_dim=256, num_tokens=64))["prefill_ctas"] == (64 // 32 + 1) * 8  # one tile
    assert B.plan(llama_dims(head_dim=128, num_tokens=64))["prefill_ctas"] == (64 // 64 + 1) * 8  # a pair
    with pytest.raises(B.PagedAttnError) as e:
        B.plan(llama_dims(head_dim=256), decode_warps=8, decode_stages=3)
    assert e.value.status == B.PA_ERR_INVALID_ARG


def test_decode_cluster_option(lib):
    for c in (2, 4, 8, 16, 3):
        p = B.plan(llama_dims(), decode_cluster=c)
        assert p["decode_cluster"] == c and p["splits"] == c
        assert p["decode_ctas"] == 8 * c
        assert p["kv_chunk"] * c >= 2048 * 16 and p["kv_chunk"] % 16 == 0
        # partials merge in distributed shared memory: only the error word
        assert p["workspace_bytes"] == 256
    assert B.plan(llama_dims(), kv_chunk=1024)["decode_cluster"] == 1
    assert B.plan(llama_dims(), decode_cluster=1, decode_warps=8)["decode_cluster"] == 1
    for kw in (dict(decode_cluster=17), dict(decode_cluster=-1), dict(decode_cluster=4, kv_chunk=1024)):
        with pytest.raises(B.PagedAttnError) as e:
            B.plan(llama_dims(), **kw)
        assert e.value.status == B.PA_ERR_INVALID_ARG


def test_bad_chunk_rejected(lib):
    with pytest.raises(B.PagedAttnError) as e:
        B.plan(llama_dims(), kv_chunk=24)
    assert e.value.status == B.PA_ERR_INVALID_ARG


def test_forward_rejects_before_cuda(lib):
    d = llama_dims()
    # NULL dims, NULL pointers and misaligned pointers are refused on the host
    st = lib.pa_forward(None, None, None, None, None, None, None, ctypes.c_float(1.0), None, None)
    assert st == B.PA_ERR_INVALID_ARG
    st = lib.pa_forward(None, None, None, None, None, None, None, ctypes.c_float(1.0), ctypes.byref(d), None)
    assert st == B.PA_ERR_INVALID_ARG
    buf = (ctypes.c_uint8 * 64)()
    base = ctypes.addressof(buf)
    a16 = (base + 15) & ~15
    st = lib.pa_forward(a16 + 2, a16, a16, a16, a16, a16, a16, ctypes.c_float(1.0), ctypes.byref(d), None)
    assert st == B.PA_ERR_INVALID_ARG
    assert "aligned" in lib.pa_last_error().decode()


def test_empty_batch_is_noop(lib):
    d = llama_dims(num_tokens=0, num_seqs=0)
    st = lib.pa_forward(None, None, None, None, None, None, None, ctypes.c_float(1.0), ctypes.byref(d), None)
    assert st == B.PA_OK


def test_library_has_no_oracle_dependency():
    # the product library must not link or name the test oracle
    data = open(B.LIB_PATH, "rb").read()
    assert b"oracle_attention" not in data
    for f in os.listdir(os.path.join(ROOT, "paged_kv_cache_forward_gb300")):
        if f.endswith(".py") and f != "workloads.py":
            src = open(os.path.join(ROOT, "paged_kv_cache_forward_gb300", f)).read()
            assert "import oracle" not in src and "from oracle" not in src, f


def test_cache_write_rejects_before_cuda(lib):
    d = B.CacheDims(num_tokens=4, num_blocks=0, num_kv_heads=8, head_dim=128, page_size=16)
    assert lib.pa_cache_write(None, None, None, None, None, ctypes.byref(d), None) == B.PA_ERR_INVALID_ARG
    d = B.CacheDims(num_tokens=4, num_blocks=8, num_kv_heads=1, head_dim=12, page_size=16)
    assert lib.pa_cache_write(None, None, None, None, None, ctypes.byref(d), None) == B.PA_ERR_UNSUPPORTED
    d = B.CacheDims(num_tokens=0, num_blocks=8, num_kv_heads=8, head_dim=128, page_size=16)
    assert lib.pa_cache_write(None, None, None, None, None, ctypes.byref(d), None) == B.PA_OK
    d = B.CacheDims(num_tokens=4, num_blocks=8, num_kv_heads=8, head_dim=128, page_size=16)
    assert lib.pa_cache_write(None, None, None, None, None, ctypes.byref(d), None) == B.PA_ERR_INVALID_ARG


def test_early_metadata_option(lib):
    """pa_options.early_metadata takes 0 or 1 and does not change the plan."""
    base = B.plan(llama_dims())
    for v, ok in ((0, True), (1, True), (2, False), (-1, False)):
        info = B.PlanInfo()
        opts = B.options(early_metadata=v)
        st = lib.pa_plan(ctypes.byref(llama_dims()), ctypes.byref(opts), ctypes.byref(info))
        if ok:
            assert st == B.PA_OK and info.as_dict() == base
        else:
            assert st == B.PA_ERR_INVALID_ARG and lib.pa_last_error().decode()


def test_wide_groups_take_the_second_table(lib):
    """More than 16 query heads per KV head (several row groups reading the same
    pages): the plan takes the kSplitTableWide cell the call falls in; 16 or fewer
    take the first table."""
    from paged_kv_cache_forward_gb300 import sweep as S
    table = os.path.join(os.path.dirname(B.__file__), "csrc", "lut_gb300.inc")
    wide, first = S.read_table(table, S.WIDE_NAME), S.read_table(table)
    assert wide, "no wide-group rows"
    for (d, bound, units), (chunk, st, w, cl) in sorted(wide.items())[:12]:
        seqs = units // 2  # Hq 32 / Hkv 1: two row groups per sequence
        p = B.plan(llama_dims(num_q_heads=32, num_kv_heads=1, head_dim=d, num_seqs=seqs, num_tokens=seqs,
                              max_pages=bound // 16, num_blocks=seqs * bound // 16 + 1))
        assert (p["decode_warps"], p["decode_stages"], p["decode_cluster"]) == (w, st, max(cl, 1)), (bound, units)
        if cl <= 1:
            assert p["kv_chunk"] == min(chunk, bound), (bound, units)
    # 4 query heads per KV head, same decode units: the first table
    (d, bound, units), (chunk, st, w, cl) = sorted(first.items())[0]
    p = B.plan(llama_dims(num_q_heads=4 * units, num_kv_heads=units, head_dim=d, max_pages=bound // 16))
    assert (p["decode_warps"], p["decode_stages"], p["decode_cluster"]) == (w, st, max(cl, 1))


def test_binding_host_tensor_rules(monkeypatch):
    """Host tensors: q, the metadata and out may be pinned host memory (the
    library checks q against the shapes); the caches must be on the device; a
    pageable host tensor is refused before the library is called."""
    import torch

    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    kv = torch.zeros(3, 16, 1, 64, dtype=torch.bfloat16)
    bt = torch.zeros(2, 1, dtype=torch.int32)
    sl = torch.ones(2, dtype=torch.int32)
    qsl = torch.arange(3, dtype=torch.int32)
    assert set(B._HOST_OK) == {"q", "block_table", "seq_lens", "query_start_loc", "out"}
    with pytest.raises(ValueError, match="q must be a CUDA tensor or a pinned host tensor"):
        B._check_tensors(q, kv, kv, bt, sl, qsl, q)
    # every host tensor taken as pinned: the first refusal is the KV cache's
    monkeypatch.setattr(torch.Tensor, "is_pinned", lambda self: True)
    with pytest.raises(ValueError, match="k_cache must be a CUDA tensor$"):
        B._check_tensors(q, kv, kv, bt, sl, qsl, q)
