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


def test_chunk_oracle_sample_runs_on_e4m3_caches():
    """The CPU baseline of a chunk workload over E4M3 caches passes the per-head scales
    (the oracle refuses an E4M3 cache without them)."""
    w = workloads.to_fp8(workloads.make("long16_chunk512", num_seqs=1, context=300,
                                        query_len=40))
    value, unit, desc = bench._chunk_sample(w, bench._host_inputs(w), 0.2, 1)
    assert value > 0 and unit in ("TFLOP/s", "GB/s") and "oracle" in desc


def test_dominant_kernel_is_the_library_routing():
    """The roofline's kernel label comes from the library's own routing query."""
    from paged_kv_cache_119_gb300 import build
    build.build()
    import paged_kv_cache_119_gb300 as pa

    def label(config, **kw):
        return bench.dominant_kernel(pa, bench.make_workload(config, "cpu", **kw))
    assert label("llama13b", num_seqs=2) == "decode_kernel"                 # MHA, CUDA cores
    assert label("long16", num_seqs=1) == "decode_mma_kernel"               # group 8
    assert label("llama13b_fp8", num_seqs=2) == "decode_tc8_kernel"         # E4M3 MHA
    assert label("long16_fp8", num_seqs=1) == "decode_mma_kernel"           # E4M3, 8 rows
    assert label("llama13b_verify4_fp8", num_seqs=2) == "decode_tc8_kernel (chunk rows)"
    assert label("llama13b_verify4", num_seqs=2) == "decode_mma_kernel (chunk rows)"
    assert label("long16_chunk512", num_seqs=1) == "chunk_attn_kernel"
    assert label("long16_chunk512_fp8", num_seqs=1) == \
        "chunk_attn_kernel (E4M3 tiles converted to f16)"
    assert pa.pa_decode_kernel_name(torch.float32, 64, 8, 128) == "decode_kernel"


def test_percentiles_nearest_rank():
    p = bench.percentiles(list(range(1, 21)))
    assert (p["p10"], p["p50"], p["p90"]) == (2, 10, 18)
    assert bench.percentiles([7.0]) == {"p10": 7.0, "p50": 7.0, "p90": 7.0}


def test_traffic_rows_count_only_for_current_sources(tmp_path, monkeypatch):
    import json
    f = tmp_path / "t.json"
    f.write_text(json.dumps({"rows": {"a": {"kernel_hash": bench.kernel_hash(),
                                            "dram_bytes_per_launch": 123},
                                      "b": {"kernel_hash": "0" * 16,
                                            "dram_bytes_per_launch": 456}}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("a") == 123
    assert bench.recorded_traffic("b") is None           # stale: captured from other sources
    assert bench.recorded_traffic("c") is None


def test_bench_reads_no_markdown():
    src = open(bench.__file__, encoding="utf-8").read()
    assert ".md" not in src
