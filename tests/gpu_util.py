"""Helpers for the GPU parity tests: run the CUDA path, compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_forward_gb300 as pa
from paged_kv_cache_forward_gb300 import build as build_mod
from paged_kv_cache_forward_gb300 import workloads as W

# Tolerance of the GPU bf16 output against the fp64 oracle, over all compared
# elements: max-abs error 1.5e-2 and mean-abs error 2e-3.  The output is bf16,
# so an element whose exact value has magnitude >= 4 cannot always be written
# within 1.5e-2 (half a bf16 ulp there is 2^-6 = 0.0156); such an element is
# held to half an ulp of its exact value plus 1e-3 instead (the larger bound).
TOL_MAX = 1.5e-2
TOL_MEAN = 2e-3
TOL_ARITH = 1e-3  # fp32 arithmetic on top of the output rounding, for |exact| >= 4


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) at |x|."""
    _, e = np.frexp(np.abs(x))  # |x| = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 9)


def max_abs_bound(ref: np.ndarray) -> np.ndarray:
    return np.maximum(TOL_MAX, bf16_half_ulp(ref) + TOL_ARITH)

_built = False


def ensure_built():
    global _built
    if not _built:
        build_mod.build()
        pa.load()
        _built = True


def run(b: W.Batch, kv_chunk: int = 0, device="cuda", check_errors: bool = True,
        decode_stages: int = 0, decode_warps: int = 0, decode_cluster: int = 0,
        test_stall_prefill: int = 0) -> torch.Tensor:
    """pa_forward on the batch; returns the output on the CPU (bf16).  The output
    buffer starts as NaN so that an unwritten row cannot pass."""
    ensure_built()
    d = b.to(device)
    out = torch.full_like(d.q, float("nan"))
    pa.forward(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.query_start_loc, out,
               scale=b.scale, kv_chunk=kv_chunk, decode_stages=decode_stages,
               decode_warps=decode_warps, decode_cluster=decode_cluster, test_stall_prefill=test_stall_prefill)
    torch.cuda.synchronize()
    if check_errors:
        assert pa.device_error() == 0
    return out.cpu()


def errors(got_bf16: torch.Tensor, ref: np.ndarray):
    g = got_bf16.double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), "non-finite GPU output"
    e = np.abs(g - ref)
    return float(e.max()), float(e.mean())


def assert_close(got_bf16, ref, what=""):
    mx, mean = errors(got_bf16, ref)
    g = got_bf16.double().numpy()
    worst = float((np.abs(g - ref) / max_abs_bound(ref)).max()) if ref.size else 0.0
    assert worst <= 1.0 and mean <= TOL_MEAN, (
        f"{what}: max_abs {mx:.3e} mean_abs {mean:.3e} (worst element at {worst:.3f} of its bound)")
    return mx, mean


def sample_rows(b: W.Batch, n_random: int, seed: int = 0):
    """(token, head) rows to check on a batch too large for a full oracle pass:
    the first and last new token of every sequence (all heads of one, one head of
    the rest), plus random rows."""
    g = torch.Generator().manual_seed(seed)
    Hq = b.num_q_heads
    qsl = b.query_start_loc.tolist()
    rows = set()
    for s in range(b.num_seqs):
        if qsl[s + 1] == qsl[s]:
            continue
        first, last = qsl[s], qsl[s + 1] - 1
        if s == 0:
            for h in range(Hq):
                rows.add((first, h))
                rows.add((last, h))
        else:
            rows.add((first, s % Hq))
            rows.add((last, (s * 7 + 3) % Hq))
    T = b.num_tokens
    for _ in range(n_random):
        rows.add((int(torch.randint(0, T, (1,), generator=g)), int(torch.randint(0, Hq, (1,), generator=g))))
    return sorted(rows)
