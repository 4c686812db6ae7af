"""Host logic of bench.py without a GPU: byte accounting, aggregation over ranks,
and the multi-rank timing reduction on two gloo ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_119_gb300 import workloads


def test_aggregate_uses_slowest_rank():
    value, t = bench.aggregate([1.0, 2.0, 1.5], [10, 10, 10])
    assert t == 2.0 and value == 15.0


def test_algorithmic_bytes_tiny():
    w = workloads.make("tiny")
    b = bench.algorithmic_bytes(w)
    # 69 cached tokens x 2 heads x (K + V) x 64 dims x 4 bytes
    assert b["kv"] == 69 * 2 * 2 * 64 * 4
    assert b["decode"] == b["kv"] + 2 * 4 * 2 * 64 * 4 + 4 * (1 + 1 + 1 + 3) + 4 * 4
    assert b["step"] == b["decode"] + b["reshape"]


def test_parse_defaults():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.config == "llama13b"
    assert a.warmup >= 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sec = bench.max_over_ranks(0.5 + rank, torch.device("cpu"))
    value, t = bench.aggregate([sec], [100 * world])
    q.put((rank, sec, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [1.5, 1.5]
    assert all(abs(r[2] - 200 / 1.5) < 1e-9 for r in res)
