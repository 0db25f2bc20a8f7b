"""The benchmark's N > 1 host logic on CPU with two gloo ranks: each rank draws
its own batch (weak scaling, no data-path collective), the timing is the max
over ranks and the work is summed over ranks."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_forward_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        b = W.batched_decode(seed=bench.rank_seed(0, r), batch=4, lo=16, hi=64)
        work = bench.work_of(b)
        t_ms = 10.0 + 5.0 * r  # rank 1 is the slow one
        bench.barrier(w)
        mx = bench.reduce_max(t_ms, w)
        total = bench.reduce_sum(work["kv_bytes"], w)
        q.put((r, w, local, mx, total, work["kv_bytes"], b.seq_lens.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, mx0, tot0, kv0, sl0), (r1, w1, l1, mx1, tot1, kv1, sl1) = res
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert mx0 == mx1 == 15.0          # max over ranks
    assert tot0 == tot1 == kv0 + kv1   # whole-job work
    assert sl0 != sl1                  # independent batches per rank


def test_single_rank_helpers_are_identity():
    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.reduce_sum(4.0, 1) == 4.0
    assert bench.rank_seed(5, 0) == 5


def test_metric_selection():
    assert bench.metric_of("varlen_prefill")[1] == "TFLOP/s"
    assert bench.metric_of("llama_decode_32768")[1] == "GB/s"
    b = W.llama_decode(1024, seed=0)
    w = bench.work_of(b)
    assert w["kv_bytes"] == 1024 * 2 * 8 * 128 * 2
    assert w["flops"] == 4 * 128 * 32 * 1024


@pytest.mark.parametrize("cfg", ["tiny_decode"])
def test_reference_arm_prints_one_line(cfg, capsys):
    assert bench.main(["--impl", "reference", "--config", cfg, "--steps", "1", "--warmup", "0",
                       "--cpu-seconds", "0.5"]) == 0
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
