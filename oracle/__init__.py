"""Python marshalling for the fp64 CPU oracle in ``oracle.c``.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use this module; the CUDA library and its
binding never import it.  It shares no code with the CUDA path.

``build()`` compiles ``oracle.c`` with the host C compiler (OpenMP, -O2, strict
IEEE double: no fast-math).  Inputs are passed as the bf16 bit patterns, which the
C code widens to double exactly.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

ERRORS = {
    0: "ok",
    1: "bad dimensions",
    2: "bad query_start_loc",
    3: "bad lengths (need q_len <= seq_len <= max_pages * page_size)",
    4: "block id out of range",
    5: "row index out of range",
    6: "out of memory",
}


class OracleError(RuntimeError):
    pass


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "num_tokens", "num_seqs", "num_q_heads", "num_kv_heads",
        "head_dim", "page_size", "num_blocks", "max_pages")]


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra=()) -> str:
    """Compile an oracle source file to a shared library; returns the path."""
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", *extra, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_oracle()
    return _LIB_PATH


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed) or a given copy of it."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    lib.oracle_attention.argtypes = [P, P, P, P, P, P, ctypes.POINTER(_Dims), ctypes.c_double, P, P, ctypes.c_int]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [P, P, P, P, P, P, ctypes.POINTER(_Dims), ctypes.c_double,
                                          P, ctypes.c_int64, P, P, ctypes.c_int]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention_weights.argtypes = [P, P, P, P, P, P, ctypes.POINTER(_Dims), ctypes.c_double,
                                             ctypes.c_int64, ctypes.c_int64, P, P]
    lib.oracle_attention_weights.restype = ctypes.c_int
    lib.oracle_validate.argtypes = [ctypes.POINTER(_Dims), P, P, P]
    lib.oracle_validate.restype = ctypes.c_int
    lib.oracle_cache_write.argtypes = [P, P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int64]
    lib.oracle_cache_write.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _bf16_bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 numpy array."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x.astype(np.int32, copy=False))
    return np.ascontiguousarray(x.detach().cpu().numpy().astype(np.int32, copy=False))


def _scale64(scale: float) -> float:
    # The kernel receives scale as an fp32; widen exactly that value.
    return float(np.float32(scale))


class _Args:
    def __init__(self, q, k_cache, v_cache, block_table, seq_lens, query_start_loc):
        self.q = _bf16_bits(q)
        self.k = _bf16_bits(k_cache)
        self.v = _bf16_bits(v_cache)
        self.bt = _i32(block_table)
        self.sl = _i32(seq_lens)
        self.qsl = _i32(query_start_loc)
        T, Hq, D = self.q.shape
        NB, P, Hkv, D2 = self.k.shape
        assert D == D2 and self.v.shape == self.k.shape
        B = self.sl.shape[0]
        assert self.qsl.shape[0] == B + 1
        mp = self.bt.shape[1] if self.bt.ndim == 2 else 0
        if B:
            assert self.bt.shape[0] == B
        self.dims = _Dims(T, B, Hq, Hkv, D, P, NB, mp)
        if self.bt.size == 0:
            self.bt = np.zeros(1, dtype=np.int32)

    def ptrs(self):
        return [a.ctypes.data for a in (self.q, self.k, self.v, self.bt, self.sl, self.qsl)]


def _check(rc: int):
    if rc != 0:
        raise OracleError(f"oracle: {ERRORS.get(rc, rc)}")


def attention(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, scale: float,
              threads: int = 0, return_lse: bool = False, lib=None):
    """Every output row in fp64: returns out [T, Hq, D] (and lse [T, Hq])."""
    a = _Args(q, k_cache, v_cache, block_table, seq_lens, query_start_loc)
    T, Hq, D = a.q.shape
    out = np.empty((T, Hq, D), dtype=np.float64)
    lse = np.empty((T, Hq), dtype=np.float64) if return_lse else None
    rc = (lib or load()).oracle_attention(*a.ptrs(), ctypes.byref(a.dims), _scale64(scale), out.ctypes.data,
                                 lse.ctypes.data if lse is not None else None, int(threads))
    _check(rc)
    return (out, lse) if return_lse else out


def attention_rows(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, scale: float,
                   rows: Sequence, threads: int = 0, return_lse: bool = False, lib=None):
    """Selected rows: ``rows`` is a list/array of (token, q_head); returns [n, D] fp64."""
    a = _Args(q, k_cache, v_cache, block_table, seq_lens, query_start_loc)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    D = a.q.shape[2]
    out = np.empty((r.shape[0], D), dtype=np.float64)
    lse = np.empty((r.shape[0],), dtype=np.float64) if return_lse else None
    rc = (lib or load()).oracle_attention_rows(*a.ptrs(), ctypes.byref(a.dims), _scale64(scale), r.ctypes.data,
                                               r.shape[0], out.ctypes.data,
                                               lse.ctypes.data if lse is not None else None, int(threads))
    _check(rc)
    return (out, lse) if return_lse else out


def attention_weights(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, scale: float,
                      token: int, head: int, lib=None):
    """Softmax weights of one row over positions 0..L_b-1, and the row's output."""
    a = _Args(q, k_cache, v_cache, block_table, seq_lens, query_start_loc)
    qsl = a.qsl
    b = int(np.searchsorted(qsl, token, side="right") - 1)
    L = max(int(a.sl[b]), 1)
    w = np.zeros(L, dtype=np.float64)
    out = np.empty(a.q.shape[2], dtype=np.float64)
    rc = (lib or load()).oracle_attention_weights(*a.ptrs(), ctypes.byref(a.dims), _scale64(scale),
                                                  int(token), int(head), w.ctypes.data, out.ctypes.data)
    _check(rc)
    return w, out


def validate(block_table, seq_lens, query_start_loc, dims: dict) -> int:
    d = _Dims(*[int(dims[k]) for k, _ in _Dims._fields_])
    bt, sl, qsl = _i32(block_table), _i32(seq_lens), _i32(query_start_loc)
    if bt.size == 0:
        bt = np.zeros(1, dtype=np.int32)
    return load().oracle_validate(ctypes.byref(d), bt.ctypes.data, sl.ctypes.data, qsl.ctypes.data)


def batch_attention(batch, rows=None, threads: int = 0, lib=None):
    """Convenience: run the oracle on a workloads.Batch (all rows or selected rows)."""
    args = (batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.seq_lens,
            batch.query_start_loc, batch.scale)
    if rows is None:
        return attention(*args, threads=threads, lib=lib)
    return attention_rows(*args, rows=rows, threads=threads, lib=lib)


def max_threads() -> int:
    return int(load().oracle_max_threads())


def cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, lib=None):
    """Paged KV-cache write on copies of the caches; returns (k_cache, v_cache) as
    uint16 (bf16 bit) arrays.  Negative slots write nothing."""
    kn, vn = _bf16_bits(k_new), _bf16_bits(v_new)
    kc, vc = _bf16_bits(k_cache).copy(), _bf16_bits(v_cache).copy()
    sm = slot_mapping if isinstance(slot_mapping, np.ndarray) else slot_mapping.detach().cpu().numpy()
    sm = np.ascontiguousarray(sm.astype(np.int64))
    T = kn.shape[0]
    NB, P, Hkv, D = kc.shape
    assert kn.shape == (T, Hkv, D) and vn.shape == kn.shape and vc.shape == kc.shape and sm.shape == (T,)
    rc = (lib or load()).oracle_cache_write(kn.ctypes.data, vn.ctypes.data, sm.ctypes.data, kc.ctypes.data,
                                            vc.ctypes.data, T, NB, P, Hkv, D)
    _check(rc)
    return kc, vc
