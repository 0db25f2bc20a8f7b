"""ctypes binding of libpagedattn (include/pagedattn.h): argument marshalling only.

Every step of the attention runs in the library's CUDA kernels.  Tensors are
PyTorch CUDA tensors (PyTorch provides the device memory and the stream); q, the
metadata and out may also be pinned host tensors, which the decode kernel reads
and writes in place (the library rejects a host q when the shapes allow prefill
rows).  This module checks dtypes, shapes and contiguity, fills a ``pa_dims``
and passes raw pointers.  There is no fallback: if the library is missing, or a
call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedattn.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_NOT_PREPARED, PA_ERR_CUDA = range(5)

# Every symbol include/pagedattn.h declares.
EXPORTED = (
    "pa_forward", "pa_forward_ex", "pa_plan", "pa_prepare", "pa_device_error",
    "pa_release_workspaces", "pa_status_string", "pa_last_error", "pa_version", "pa_forward_noalloc",
    "pa_cache_write",
)

DEVICE_ERRORS = {
    0: "none",
    1: "block-table entry outside [0, num_blocks)",
    2: "seq_len above max_pages * page_size",
    3: "more new tokens than seq_len",
    4: "a bounded wait in a kernel gave up",
    5: "query_start_loc outside [0, num_tokens]",
}


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"libpagedattn: status {status}: {detail}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int64),
        ("num_blocks", ctypes.c_int64),
        ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
    ]


class Options(ctypes.Structure):
    _fields_ = [
        ("kv_chunk", ctypes.c_int32),
        ("decode_stages", ctypes.c_int32),
        ("decode_warps", ctypes.c_int32),
        ("decode_cluster", ctypes.c_int32),
        ("decode_start_event", ctypes.c_void_p),
        ("decode_stop_event", ctypes.c_void_p),
        ("prefill_start_event", ctypes.c_void_p),
        ("prefill_stop_event", ctypes.c_void_p),
        ("test_stall_prefill", ctypes.c_int32),
        ("launch_only", ctypes.c_int32),
        ("early_metadata", ctypes.c_int32),
    ]


class CacheDims(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int64),
        ("num_blocks", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("kv_chunk", ctypes.c_int32),
        ("splits", ctypes.c_int32),
        ("decode_ctas", ctypes.c_int64),
        ("combine_ctas", ctypes.c_int64),
        ("prefill_ctas", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
        ("launches", ctypes.c_int32),
        ("decode_stages", ctypes.c_int32),
        ("decode_warps", ctypes.c_int32),
        ("decode_cluster", ctypes.c_int32),
    ]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libpagedattn.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with paged_kv_cache_forward_gb300.build.build() "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    P, I32 = ctypes.c_void_p, ctypes.c_int
    fwd = [P, P, P, P, P, P, P, ctypes.c_float, ctypes.POINTER(Dims)]
    lib.pa_forward.argtypes = fwd + [P]
    lib.pa_forward_ex.argtypes = fwd + [ctypes.POINTER(Options), P]
    lib.pa_forward_noalloc.argtypes = fwd + [P, P]
    lib.pa_cache_write.argtypes = [P, P, P, P, P, ctypes.POINTER(CacheDims), P]
    lib.pa_plan.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Options), ctypes.POINTER(PlanInfo)]
    lib.pa_prepare.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Options), P]
    lib.pa_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
    lib.pa_release_workspaces.argtypes = []
    lib.pa_status_string.argtypes = [I32]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_error.argtypes = []
    lib.pa_last_error.restype = ctypes.c_char_p
    lib.pa_version.argtypes = []
    for name in ("pa_forward", "pa_forward_ex", "pa_plan", "pa_prepare", "pa_device_error",
                 "pa_release_workspaces", "pa_version", "pa_forward_noalloc", "pa_cache_write"):
        getattr(lib, name).restype = I32
    _lib = lib
    return lib


def _check(status: int):
    if status != PA_OK:
        lib = load()
        raise PagedAttnError(status, f"{lib.pa_status_string(status).decode()}: {lib.pa_last_error().decode()}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_dims(q_shape, k_shape, bt_shape, num_seqs) -> Dims:
    T, Hq, D = q_shape
    NB, P, Hkv, D2 = k_shape
    if D2 != D:
        raise ValueError(f"head_dim of q ({D}) and cache ({D2}) differ")
    max_pages = bt_shape[1]
    return Dims(num_tokens=T, num_blocks=NB, num_seqs=num_seqs, num_q_heads=Hq, num_kv_heads=Hkv,
                head_dim=D, page_size=P, max_pages=max_pages)


# Arguments the decode kernel reads (or writes) with plain loads and stores, so
# they may also be pinned host memory (pa_forward's pointer rules: decode-only
# dims for q).
_HOST_OK = ("q", "block_table", "seq_lens", "query_start_loc", "out")


def _out_like(q):
    # out where q is: on the device, or in pinned host memory
    return torch.empty_like(q) if q.is_cuda else torch.empty(q.shape, dtype=q.dtype, pin_memory=True)


def _check_tensors(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out):
    for name, t, dt, nd in (("q", q, torch.bfloat16, 3), ("k_cache", k_cache, torch.bfloat16, 4),
                            ("v_cache", v_cache, torch.bfloat16, 4), ("block_table", block_table, torch.int32, 2),
                            ("seq_lens", seq_lens, torch.int32, 1),
                            ("query_start_loc", query_start_loc, torch.int32, 1), ("out", out, torch.bfloat16, 3)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if t.dim() != nd:
            raise ValueError(f"{name} must have {nd} dims, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not (name in _HOST_OK and t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor" +
                             (" or a pinned host tensor" if name in _HOST_OK else ""))
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if out.shape != q.shape:
        raise ValueError("out must have the shape of q")
    B = seq_lens.shape[0]
    if query_start_loc.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("seq_lens [B], query_start_loc [B+1] and block_table [B, max_pages] disagree on B")


def options(kv_chunk: int = 0, events=None, decode_stages: int = 0, decode_warps: int = 0,
            decode_cluster: int = 0, test_stall_prefill: int = 0, launch_only: int = 0,
            early_metadata: int = 0) -> Options:
    o = Options()
    o.launch_only = launch_only
    o.early_metadata = early_metadata
    o.kv_chunk = kv_chunk
    o.decode_stages = decode_stages
    o.decode_warps = decode_warps
    o.decode_cluster = decode_cluster
    o.test_stall_prefill = test_stall_prefill
    if events:
        for key in ("decode_start_event", "decode_stop_event", "prefill_start_event", "prefill_stop_event"):
            ev = events.get(key)
            if ev is not None and not ev.cuda_event:
                raise ValueError(f"{key}: the torch event has no CUDA event yet (record it once first)")
            setattr(o, key, ev.cuda_event if ev is not None else None)
    return o


def forward(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out=None,
            scale: Optional[float] = None, kv_chunk: int = 0, events=None, stream=None,
            decode_stages: int = 0, decode_warps: int = 0, decode_cluster: int = 0,
            test_stall_prefill: int = 0, launch_only: int = 0, early_metadata: int = 0) -> torch.Tensor:
    """Paged attention forward (pa_forward).  Returns ``out`` ([T, Hq, D] bf16).

    ``events`` (optional) maps decode_start_event / decode_stop_event /
    prefill_start_event / prefill_stop_event to torch.cuda.Event objects, recorded
    around the corresponding kernels on the stream.  ``test_stall_prefill``
    (tests only) makes a wait of the prefill kernel run out; ``launch_only``
    (timing and tests) launches only the decode (1) or the prefill (2) kernel;
    ``early_metadata`` promises that the metadata is not written by the kernel
    just before the call (pa_options).
    """
    if out is None:
        out = _out_like(q)
    _check_tensors(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    dims = make_dims(q.shape, k_cache.shape, block_table.shape, seq_lens.shape[0])
    lib = load()
    s = _stream_handle(stream)
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(query_start_loc),
            _ptr(out), ctypes.c_float(scale), ctypes.byref(dims))
    if (kv_chunk or events or decode_stages or decode_warps or decode_cluster or test_stall_prefill or launch_only
            or early_metadata):
        opts = options(kv_chunk, events, decode_stages, decode_warps, decode_cluster, test_stall_prefill,
                       launch_only, early_metadata)
        _check(lib.pa_forward_ex(*args, ctypes.byref(opts), s))
    else:
        _check(lib.pa_forward(*args, s))
    return out


def forward_noalloc(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out=None,
                    scale: Optional[float] = None, device_error=None, stream=None) -> torch.Tensor:
    """pa_forward_noalloc: the forward pass using the library's fixed scratch
    array instead of an allocated workspace (for callers that cannot allocate).
    ``device_error`` (optional) is a CUDA int32 tensor of one element that
    receives the first device-side error code; the caller zeroes it."""
    if out is None:
        out = _out_like(q)
    _check_tensors(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out)
    if device_error is not None and (device_error.dtype != torch.int32 or not device_error.is_cuda):
        raise TypeError("device_error must be a CUDA int32 tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    dims = make_dims(q.shape, k_cache.shape, block_table.shape, seq_lens.shape[0])
    _check(load().pa_forward_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(query_start_loc),
        _ptr(out), ctypes.c_float(scale), ctypes.byref(dims), _ptr(device_error), _stream_handle(stream)))
    return out


def cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None):
    """pa_cache_write: copy each new token's K and V ([T, Hkv, D] bf16) to page
    slot_mapping[t] // P, slot slot_mapping[t] % P of the caches (int64 slots;
    negative = padding, no write).  The caches are updated in place."""
    for name, t, dt in (("k_new", k_new, torch.bfloat16), ("v_new", v_new, torch.bfloat16),
                        ("slot_mapping", slot_mapping, torch.int64), ("k_cache", k_cache, torch.bfloat16),
                        ("v_cache", v_cache, torch.bfloat16)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k_new.dim() != 3 or v_new.shape != k_new.shape or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("k_new, v_new must be [T, Hkv, D] and the caches [NB, P, Hkv, D]")
    T, Hkv, D = k_new.shape
    if tuple(k_cache.shape[2:]) != (Hkv, D) or tuple(slot_mapping.shape) != (T,):
        raise ValueError("shapes of the new rows, the caches and slot_mapping disagree")
    dims = CacheDims(num_tokens=T, num_blocks=k_cache.shape[0], num_kv_heads=Hkv, head_dim=D,
                     page_size=k_cache.shape[1])
    _check(load().pa_cache_write(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                 ctypes.byref(dims), _stream_handle(stream)))


def plan(dims: Dims, kv_chunk: int = 0, decode_stages: int = 0, decode_warps: int = 0,
         decode_cluster: int = 0) -> dict:
    info = PlanInfo()
    opts = options(kv_chunk, decode_stages=decode_stages, decode_warps=decode_warps, decode_cluster=decode_cluster)
    _check(load().pa_plan(ctypes.byref(dims), ctypes.byref(opts), ctypes.byref(info)))
    return info.as_dict()


def plan_for(q, k_cache, block_table, seq_lens, kv_chunk: int = 0, decode_stages: int = 0,
             decode_warps: int = 0, decode_cluster: int = 0) -> dict:
    return plan(make_dims(q.shape, k_cache.shape, block_table.shape, seq_lens.shape[0]), kv_chunk, decode_stages,
                decode_warps, decode_cluster)


def prepare(q, k_cache, block_table, seq_lens, kv_chunk: int = 0, stream=None, decode_stages: int = 0,
            decode_warps: int = 0, decode_cluster: int = 0):
    """Allocates the workspace for these shapes on the stream (call before capture)."""
    dims = make_dims(q.shape, k_cache.shape, block_table.shape, seq_lens.shape[0])
    opts = options(kv_chunk, decode_stages=decode_stages, decode_warps=decode_warps, decode_cluster=decode_cluster)
    _check(load().pa_prepare(ctypes.byref(dims), ctypes.byref(opts), _stream_handle(stream)))


def device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) its sticky device error code."""
    code = ctypes.c_int32(0)
    _check(load().pa_device_error(_stream_handle(stream), ctypes.byref(code)))
    return int(code.value)


def release_workspaces():
    _check(load().pa_release_workspaces())


def version() -> int:
    return int(load().pa_version())
