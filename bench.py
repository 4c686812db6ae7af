#!/usr/bin/env python3
"""Benchmark of one paged decode step on GB300.

A step is the whole hot path over one batch: pa_reshape_and_cache of the new
tokens' K/V (plus pa_copy_blocks where the workload has copy-on-write pairs),
then pa_decode (and its merge pass when the call splits contexts).

Default workload: the LLaMA-13B-shaped batched decode (256 sequences, 40 query
/ 40 kv heads, head_dim 128, bf16, block_size 16, lognormal context lengths with
median 400 clipped to [16, 2048], 256 new tokens per step).  Its KV pool is
about 3 GB, far larger than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle instead,
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

WORKLOADS = {
    "llama13b": "LLaMA-13B-shaped batched decode: 256 seqs, 40 q / 40 kv heads, head_dim 128, "
                "bf16, block_size 16, context lognormal(median 400, sigma 0.8) in [16, 2048], "
                "N(0, 0.5), reshape_and_cache of 256 new tokens per step",
    "opt13b": "OPT-13B-shaped decode layer: 64 seqs, 40 q / 40 kv heads, head_dim 128, fp16, "
              "block_size 16, context uniform in [1, 2048], N(0, 1)",
    "long16": "long-context split decode: 8 seqs x 32768 tokens, 64 q / 8 kv heads, head_dim 128, "
              "bf16, block_size 16, split into partitions by the library + reduce",
    "long32": "long-context split decode: 8 seqs x 32768 tokens, 64 q / 8 kv heads, head_dim 128, "
              "bf16, block_size 32, split into partitions by the library + reduce",
    "prefix": "shared-prefix decode: 16 groups x 8 seqs, 32 q / 8 kv heads, head_dim 128, bf16, "
              "block_size 16, 1024-token shared prefix, CoW tail copies each step",
}
# the same shapes over E4M3 caches with per-kv-head scales (queries and new K/V in the
# model dtype; the step's cache write quantises)
for _name in ("llama13b", "opt13b", "long16", "long32", "prefix"):
    WORKLOADS[_name + "_fp8"] = WORKLOADS[_name] + "; KV cache in FP8 E4M3 with per-head scales"
# multi-token queries (pa_chunk_attention): the step writes every new token's K/V and
# attends each new token causally over its sequence's cache
WORKLOADS["llama13b_verify4"] = (
    "speculative verification on the LLaMA-13B batch: 256 seqs, 4 new tokens each (1024 query "
    "rows) attended causally, 40 q / 40 kv heads, head_dim 128, bf16, block_size 16, context "
    "lognormal(median 400, sigma 0.8) in [16, 2048], N(0, 0.5)")
WORKLOADS["long16_chunk512"] = (
    "chunked prefill: 8 seqs x 32768-token contexts whose last 512 tokens are new (4096 query "
    "rows), 64 q / 8 kv heads, head_dim 128, bf16, block_size 16, N(0, 1)")
WORKLOADS["llama13b_verify4_fp8"] = WORKLOADS["llama13b_verify4"] + \
    "; KV cache in FP8 E4M3 with per-head scales"
WORKLOADS["long16_chunk512_fp8"] = WORKLOADS["long16_chunk512"] + \
    "; KV cache in FP8 E4M3 with per-head scales"
CHUNK_METRIC = {"llama13b_verify4": "paged verify attention KV GB/s",
                "llama13b_verify4_fp8": "paged verify attention KV GB/s",
                "long16_chunk512": "paged chunk attention TFLOP/s",
                "long16_chunk512_fp8": "paged chunk attention TFLOP/s"}
# swapping (pa_swap_blocks): a preempted group's blocks out to pinned CPU memory and back
WORKLOADS["llama13b_swap"] = (
    "KV swapping on the LLaMA-13B batch: every block of the last 64 of 256 sequences "
    "(all-or-nothing per sequence), one layer's K and V pools (160 KB blocks), out to a "
    "pinned CPU pool and back into the GPU pool, one pa_swap_blocks launch each way")
SWAP_METRIC = "paged KV swap GB/s (out + in)"
# every workload above, each measured briefly in the default run's `configs` object
CONFIG_ROWS = ("opt13b", "llama13b", "prefix", "long16", "long32", "opt13b_fp8",
               "llama13b_fp8", "prefix_fp8", "long16_fp8", "long32_fp8", "llama13b_verify4",
               "llama13b_verify4_fp8", "long16_chunk512", "long16_chunk512_fp8",
               "llama13b_swap")
DTYPE_NAME = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32",
              torch.float8_e4m3fn: "fp8_e4m3"}
METRIC = "paged decode attention KV GB/s"
KERNEL_SRC = os.path.join(ROOT, "paged_kv_cache_119_gb300", "csrc", "decode_kernel.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")
# nominal GB300 HBM3e bandwidth, context for the measured fractions
NOMINAL_HBM_GBS = 7900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(WORKLOADS), default="llama13b")
    ap.add_argument("--partition-size", type=int, default=None,
                    help="pa_decode partition_size (default 0: the library's automatic split)")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="shrink the workload to this many sequences (profiling cases)")
    ap.add_argument("--flush-l2", action="store_true",
                    help="write a 512 MB buffer between timed steps (outside the events)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the short runs of the other workloads (the `configs` object)")
    ap.add_argument("--config-steps", type=int, default=10,
                    help="timed steps of each workload in the `configs` object")
    ap.add_argument("--config-warmup", type=int, default=3)
    ap.add_argument("--eager", action="store_true",
                    help="time eager steps instead of replays of the captured step graph")
    ap.add_argument("--run-probe", action="store_true",
                    help="print the read rate of randomly ordered fixed-size runs (1-16 KB, the "
                         "granularity of one kv head's block) instead of a bench line")
    ap.add_argument("--no-read-probe", action="store_true",
                    help="skip the read-only bandwidth probe reported beside the copy peak")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(per_rank_seconds, per_rank_units):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = max(per_rank_seconds)
    return sum(per_rank_units) / t, t


def max_over_ranks(seconds: float, device) -> float:
    """The slowest rank's time (an all-reduce MAX over the default process group)."""
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def load_tensor_peak():
    """Dense bf16 tensor TFLOP/s: the sustained measurement (the chunk kernel is timed
    inside a seconds-long loop of steps), else the recipe's fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops_sustained"]), "measured sustained"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback sustained"


def kernel_hash() -> str:
    """Hash of every kernel source (csrc/*.cuh, *.cu, *.h) but the bandwidth probe, which
    no attention kernel includes: a recorded traffic row counts only for the exact
    sources it was captured from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_119_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cuh", ".cu", ".h")) and name != "probe.cu":
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str):
    """ncu DRAM bytes per attention launch, if recorded for the current kernel sources
    (profiles/decode_traffic.json, one row per config)."""
    try:
        with open(TRAFFIC_FILE, encoding="utf-8") as f:
            row = json.load(f)["rows"][config]
    except (OSError, KeyError, ValueError):
        return None
    if row.get("kernel_hash") != kernel_hash():
        return None
    return int(row["dram_bytes_per_launch"])


def algorithmic_bytes(w) -> dict:
    """Bytes a decode step must move at minimum (each cached K/V byte read once)."""
    esz = torch.tensor([], dtype=w.dtype).element_size()       # q, out, new K/V
    csz = w.k_cache.element_size()                              # cache elements
    lens = w.context_lens.tolist()
    kv = w.kv_bytes()
    qo = 2 * w.num_seqs * w.num_q_heads * w.head_dim * esz
    tables = 4 * sum(math.ceil(L / w.block_size) for L in lens) + 4 * w.num_seqs
    T = w.slot_mapping.numel()
    reshape = 2 * T * w.num_kv_heads * w.head_dim * (esz + csz) + 8 * T
    copies = 0
    if w.copy_pairs is not None:
        copies = 2 * 2 * len(w.copy_pairs) * w.num_kv_heads * w.block_size * w.head_dim * csz
    if w.query_start is not None:                  # one q and out row per new token
        qo = 2 * int(w.q.shape[0]) * w.num_q_heads * w.head_dim * esz + 4 * (w.num_seqs + 1)
    return {"kv": kv, "decode": kv + qo + tables, "reshape": reshape, "copy": copies,
            "step": kv + qo + tables + reshape + copies}


def algorithmic_flops(w) -> int:
    """Multiply-adds x 2 of the attention a step must do: q.k and p.v over every
    (query row, head, visible token), 4 * head_dim flops each; chunk token j of a
    sequence with n new tokens and context L sees L - n + j + 1 tokens."""
    lens = w.context_lens.tolist()
    if w.query_start is None:
        return 4 * w.head_dim * w.num_q_heads * int(sum(lens))
    qs = w.query_start.tolist()
    total = 0
    for s, L in enumerate(lens):
        n = qs[s + 1] - qs[s]
        total += n * (L - n) + n * (n + 1) // 2
    return 4 * w.head_dim * w.num_q_heads * total


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0_wall: float, t1_wall: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + r[0].strip().split(".")[1]) if "." in r[0] else 0.0
                rows.append((ts, float(r[1]), float(r[2]), r[4].strip(),
                             [x.strip() for x in r[5:9]]))
            except (ValueError, IndexError):
                continue
        inside = [x for x in rows if t0_wall - 0.05 <= x[0] <= t1_wall + 0.05]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(x[1] for x in use)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for x in use for i, v in enumerate(x[4]) if v == "Active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(x[2] for x in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


def make_workload(config: str, device, num_seqs=None):
    from paged_kv_cache_119_gb300 import workloads
    kw = {} if num_seqs is None else {"num_seqs": num_seqs}
    if config.endswith("_fp8"):
        return workloads.to_fp8(workloads.make(config[:-4], device=device, **kw))
    return workloads.make(config, device=device, **kw)


def launched_split(pa, w) -> bool:
    """Whether the library's automatic choice splits this workload (one more launch)."""
    if w.query_start is not None:
        return pa.pa_chunk_partition_tokens(w.k_cache.dtype if w.fp8 else w.dtype, w.num_seqs,
                                            w.num_q_heads, w.num_kv_heads,
                                            w.head_dim, w.block_size, w.max_query_len,
                                            w.max_context_len, 0) > 0
    return pa.pa_decode_partition_tokens(w.q.dtype, w.k_cache.dtype, w.num_seqs, w.num_q_heads,
                                         w.num_kv_heads, w.head_dim, w.block_size,
                                         w.max_context_len, 0) > 0


def dominant_kernel(pa, w) -> str:
    """The attention kernel the library runs for this workload, as the library itself
    reports it (pa_decode_kernel_name / pa_chunk_kernel_name: the launchers' own rule)."""
    kv = w.k_cache.dtype
    if w.query_start is not None:
        return pa.pa_chunk_kernel_name(kv, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                       w.max_query_len)
    return pa.pa_decode_kernel_name(kv, w.num_q_heads, w.num_kv_heads, w.head_dim)


def percentiles(vals) -> dict:
    """p10 / p50 / p90 of a list (nearest rank)."""
    v = sorted(vals)
    pick = lambda f: v[min(len(v) - 1, max(0, int(math.ceil(f * len(v))) - 1))]
    return {"p10": pick(0.1), "p50": pick(0.5), "p90": pick(0.9)}


def read_probe_gbs(pa, dev, nbytes=4 << 30, reps=10) -> float:
    """Read-only bandwidth of this GPU: pa_stream_read over a 4 GiB buffer (larger than
    L2), median of `reps` launches timed with CUDA events on the current stream."""
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        pa.pa_stream_read(buf, sink)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for b, e in ev:
        b.record()
        pa.pa_stream_read(buf, sink)
        e.record()
    torch.cuda.synchronize()
    ms = percentiles([b.elapsed_time(e) for b, e in ev])["p50"]
    del buf
    return nbytes / (ms / 1e3) / 1e9


def run_probe(dev, nbytes=4 << 30, reps=10) -> dict:
    """Read rate of a 4 GiB buffer read as fixed-size runs in a seeded random order
    (pa_stream_read_runs; best of `reps` launches, CUDA events): the ceiling for a paged
    cache whose blocks of one kv head are runs of block_size x head_dim x element bytes
    scattered through the pool.  Sequential pa_stream_read beside it."""
    import paged_kv_cache_119_gb300 as pa
    from paged_kv_cache_119_gb300 import build as pa_build
    pa_build.build()
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros(2, dtype=torch.int32, device=dev)
    gen = torch.Generator().manual_seed(119)
    out = {"metric": "random-run read GB/s", "unit": "GB/s", "bytes": nbytes,
           "order": "seeded random permutation of all runs; CTAs take consecutive entries"}
    for run in (1024, 2048, 4096, 8192, 16384):
        order = torch.randperm(nbytes // run, generator=gen, dtype=torch.int32).to(dev)
        for _ in range(3):
            pa.pa_stream_read_runs(buf, run, order, sink)
        best = float("inf")
        for _ in range(reps):
            b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b.record()
            pa.pa_stream_read_runs(buf, run, order, sink)
            e.record()
            torch.cuda.synchronize()
            best = min(best, b.elapsed_time(e))
        out[f"run_{run // 1024}KB_gbs"] = round(nbytes / (best / 1e3) / 1e9, 1)
        del order
    if int(sink[1].item()) != 0:
        raise RuntimeError("run probe: entries outside the buffer")
    out["sequential_gbs"] = round(read_probe_gbs(pa, dev, nbytes, reps), 1)
    return out


def step_ops(pa, w):
    """(cache write, decode) callables of the library for this workload's cache type
    (for a chunk workload the attention call is pa_chunk_attention)."""
    if w.query_start is not None and w.fp8:
        ks, vs = w.meta["k_scale"], w.meta["v_scale"]

        def write(k, v, slots):
            pa.pa_reshape_and_cache_fp8(k, v, w.k_cache, w.v_cache, slots, ks, vs)

        def decode(out, q, bt, cl, part, ws, qs=None):
            pa.pa_chunk_attention_fp8(out, q, w.k_cache, w.v_cache, ks, vs, bt, cl,
                                      w.query_start if qs is None else qs, w.scale,
                                      w.num_kv_heads, w.block_size, max_query_len=w.max_query_len,
                                      max_context_len=w.max_context_len, partition_size=part,
                                      workspace=ws)
        return write, decode
    if w.query_start is not None:
        def write(k, v, slots):
            pa.pa_reshape_and_cache(k, v, w.k_cache, w.v_cache, slots)

        def decode(out, q, bt, cl, part, ws, qs=None):
            pa.pa_chunk_attention(out, q, w.k_cache, w.v_cache, bt, cl,
                                  w.query_start if qs is None else qs, w.scale, w.num_kv_heads,
                                  w.block_size, max_query_len=w.max_query_len,
                                  max_context_len=w.max_context_len, partition_size=part,
                                  workspace=ws)
        return write, decode
    if w.fp8:
        ks, vs = w.meta["k_scale"], w.meta["v_scale"]

        def write(k, v, slots):
            pa.pa_reshape_and_cache_fp8(k, v, w.k_cache, w.v_cache, slots, ks, vs)

        def decode(out, q, bt, cl, part, ws):
            pa.pa_decode_fp8(out, q, w.k_cache, w.v_cache, ks, vs, bt, cl, w.scale,
                             w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                             partition_size=part, workspace=ws)
    else:
        def write(k, v, slots):
            pa.pa_reshape_and_cache(k, v, w.k_cache, w.v_cache, slots)

        def decode(out, q, bt, cl, part, ws):
            pa.pa_decode(out, q, w.k_cache, w.v_cache, bt, cl, w.scale, w.num_kv_heads,
                         w.block_size, max_context_len=w.max_context_len, partition_size=part,
                         workspace=ws)
    return write, decode


# ------------------------------------------------------------------------------ our arm

def swap_plan(w, victims=64):
    """(GPU block ids of the last `victims` sequences, bytes of one block)."""
    bt = w.block_tables.cpu()
    lens = w.context_lens.tolist()
    blocks = []
    for s in range(w.num_seqs - victims, w.num_seqs):
        n = (lens[s] + w.block_size - 1) // w.block_size
        blocks += [int(b) for b in bt[s, :n]]
    bb = w.k_cache[0].numel() * w.k_cache.element_size()
    return blocks, bb


def link_peak_gbs(dev, nbytes=1 << 30, reps=5):
    """Best 1 GiB pinned-host <-> device copy rates, each way, in GB/s: by the copy
    engines (cudaMemcpyAsync) and by the SMs (the swap kernel moving 64 contiguous
    16 MiB blocks in one launch, the plainest SM-driven streaming copy)."""
    import paged_kv_cache_119_gb300 as pa
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    devb = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    nblk = 64
    ident = torch.stack([torch.arange(nblk), torch.arange(nblk)], 1).contiguous()
    best = {}
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, (dst, src) in (("d2h", (host, devb)), ("h2d", (devb, host))):
        for how in ("dma", "sm"):
            t = []
            for _ in range(reps):
                b.record()
                if how == "dma":
                    dst.copy_(src, non_blocking=True)
                else:
                    pa.pa_swap_blocks(src.view(nblk, -1), dst.view(nblk, -1), ident)
                e.record()
                torch.cuda.synchronize()
                t.append(b.elapsed_time(e))
            best[f"{name}_{how}"] = nbytes / (min(t) / 1e3) / 1e9
    return best


def run_swap(args, rank, world, local):
    """The swap step: every block of the victim sequences, K and V, out to a pinned CPU
    pool (one launch) and back into its GPU blocks (one launch)."""
    import paged_kv_cache_119_gb300 as pa
    from paged_kv_cache_119_gb300 import build as pa_build
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa_build.build()
    w = make_workload("llama13b", dev, args.num_seqs)
    blocks, bb = swap_plan(w, min(64, w.num_seqs))
    n = len(blocks)
    cpu_k = torch.empty((n,) + tuple(w.k_cache.shape[1:]), dtype=w.dtype).pin_memory()
    cpu_v = torch.empty_like(cpu_k).pin_memory()
    # the pairs are host int64 tensors built once (the binding takes them as they are)
    out_pairs = torch.tensor([(b, i) for i, b in enumerate(blocks)], dtype=torch.int64)
    in_pairs = out_pairs.flip(1).contiguous()
    moved = 2 * 2 * n * bb                       # K and V, out and in

    def step(e=None):
        if e is not None:
            e[0].record()
        pa.pa_swap_blocks([w.k_cache, w.v_cache], [cpu_k, cpu_v], out_pairs)
        if e is not None:
            e[1].record()
        pa.pa_swap_blocks([cpu_k, cpu_v], [w.k_cache, w.v_cache], in_pairs)
        if e is not None:
            e[2].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    begin, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0_wall = time.time()
    begin.record()
    for i in range(args.steps):
        step(ev[i])
    end.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1_wall = time.time()
    clocks = sampler.stop(t0_wall, t1_wall) if rank == 0 else None
    total_ms = begin.elapsed_time(end)
    out_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    in_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    sec = max_over_ranks(total_ms / 1e3, dev) if world > 1 else total_ms / 1e3
    value = moved * args.steps * world / sec / 1e9

    # the same moves as one cudaMemcpyAsync per block and pool (the per-block transfers
    # whose small size the pages' Figure 19a blames), for comparison
    pair_list = out_pairs.tolist()

    def per_block():
        for (g, c) in pair_list:
            cpu_k[c].copy_(w.k_cache[g], non_blocking=True)
            cpu_v[c].copy_(w.v_cache[g], non_blocking=True)
        for (g, c) in pair_list:
            w.k_cache[g].copy_(cpu_k[c], non_blocking=True)
            w.v_cache[g].copy_(cpu_v[c], non_blocking=True)
    per_block()
    torch.cuda.synchronize()
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b.record()
    for _ in range(3):
        per_block()
    e.record()
    torch.cuda.synchronize()
    per_block_gbs = 3 * moved / (b.elapsed_time(e) / 1e3) / 1e9

    # end to end through the public API: each step waits for its moves on the host
    def e2e_step():
        pa.pa_swap_blocks([w.k_cache, w.v_cache], [cpu_k, cpu_v], out_pairs)
        pa.pa_swap_blocks([cpu_k, cpu_v], [w.k_cache, w.v_cache], in_pairs)
        torch.cuda.current_stream().synchronize()
    for _ in range(args.warmup):
        e2e_step()
    t = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    e2e_ms = (time.perf_counter() - t) / args.steps * 1e3
    peaks = link_peak_gbs(dev)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None
    peak = max((peaks["d2h_dma"] + peaks["h2d_dma"]) / 2, (peaks["d2h_sm"] + peaks["h2d_sm"]) / 2)
    achieved = moved / ((out_ms + in_ms) / 1e3) / 1e9
    line = {
        "metric": SWAP_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[w.k_cache.dtype],
        "data": "synthetic",
        "config": {"workload": WORKLOADS[args.config], "name": args.config,
                   "swapped_blocks": n, "block_bytes": bb, "bytes_per_step": moved,
                   "l2": "no flush: each direction moves "
                         f"{2 * n * bb / 1e9:.2f} GB, larger than the 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "swap_out_us": round(out_ms * 1e3, 2), "swap_in_us": round(in_ms * 1e3, 2),
        "swap_out_gbs": round(2 * n * bb / (out_ms / 1e3) / 1e9, 1),
        "swap_in_gbs": round(2 * n * bb / (in_ms / 1e3) / 1e9, 1),
        "per_block_memcpy_gbs": round(per_block_gbs, 1),
        "roofline": {"bound": "link", "achieved": round(achieved, 1), "peak": round(peak, 1),
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "swap_blocks_kernel",
                     "peak_kind": "measured in this run: the faster of the mean best "
                                  "1 GiB pinned<->device copy each way by the copy engines "
                                  f"(d2h {peaks['d2h_dma']:.0f}, h2d {peaks['h2d_dma']:.0f} GB/s) "
                                  "and by the SMs in one contiguous streaming launch "
                                  f"(d2h {peaks['d2h_sm']:.0f}, h2d {peaks['h2d_sm']:.0f} GB/s)",
                     "algorithmic_bytes_per_launch": 2 * n * bb},
        # one launch per 1024 pairs (and per 64 caches) in each direction
        "gpu_launches": 2 * math.ceil(n / 1024) * args.steps,
        "clocks": clocks,
        "e2e": {"value": round(moved / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": moved // 2,
                "d2h_bytes_per_step": moved // 2},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = swap_cpu_baseline(w, blocks, bb, args.cpu_budget)
    return line


def swap_row(pa, dev, steps, warmup, local) -> dict:
    """The swap step of the LLaMA-13B batch (last 64 sequences' blocks out to a pinned
    CPU pool and back, one launch each way) for the `configs` object."""
    w = make_workload("llama13b", dev)
    blocks, bb = swap_plan(w, 64)
    n = len(blocks)
    cpu_k = torch.empty((n,) + tuple(w.k_cache.shape[1:]), dtype=w.dtype).pin_memory()
    cpu_v = torch.empty_like(cpu_k).pin_memory()
    out_pairs = torch.tensor([(b, i) for i, b in enumerate(blocks)], dtype=torch.int64)
    in_pairs = out_pairs.flip(1).contiguous()
    for _ in range(warmup):
        pa.pa_swap_blocks([w.k_cache, w.v_cache], [cpu_k, cpu_v], out_pairs)
        pa.pa_swap_blocks([cpu_k, cpu_v], [w.k_cache, w.v_cache], in_pairs)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    sampler = ClockSampler(local)
    sampler.start()
    torch.cuda.synchronize()
    t0 = time.time()
    for e in ev:
        e[0].record()
        pa.pa_swap_blocks([w.k_cache, w.v_cache], [cpu_k, cpu_v], out_pairs)
        e[1].record()
        pa.pa_swap_blocks([cpu_k, cpu_v], [w.k_cache, w.v_cache], in_pairs)
        e[2].record()
    torch.cuda.synchronize()
    clocks = sampler.stop(t0, time.time())
    step = percentiles([e[0].elapsed_time(e[2]) for e in ev])
    mean_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / steps
    peaks = link_peak_gbs(dev)
    peak = max((peaks["d2h_dma"] + peaks["h2d_dma"]) / 2, (peaks["d2h_sm"] + peaks["h2d_sm"]) / 2)
    achieved = 4 * n * bb / (mean_ms / 1e3) / 1e9
    del w, cpu_k, cpu_v
    torch.cuda.empty_cache()
    return {"kernel": "swap_blocks_kernel", "bound": "link", "achieved": round(achieved, 1),
            "unit": "GB/s", "peak": round(peak, 1), "frac": round(achieved / peak, 4),
            "traffic": None, "step_us_p50": round(step["p50"] * 1e3, 2),
            "step_us_p10": round(step["p10"] * 1e3, 2), "step_us_p90": round(step["p90"] * 1e3, 2),
            "step_us_mean": round(mean_ms * 1e3, 2), "steps": steps, "warmup": warmup,
            "peak_kind": "measured in this run: faster of the copy engines' and one SM streaming "
                         "launch's pinned<->device rate, mean of both directions",
            "clocks": clocks}


def swap_cpu_baseline(w, blocks, bb, budget_s):
    """The oracle's byte moves on host copies of the same pools and pairs."""
    import oracle
    k, v = w.k_cache.cpu(), w.v_cache.cpu()
    ck = torch.empty((len(blocks),) + tuple(k.shape[1:]), dtype=k.dtype)
    cv = torch.empty_like(ck)
    out_pairs = [(b, i) for i, b in enumerate(blocks)]
    in_pairs = [(i, b) for i, b in enumerate(blocks)]
    reps, t = 0, time.perf_counter()
    while time.perf_counter() - t < budget_s / 2 or reps == 0:
        oracle.swap_blocks([k, v], [ck, cv], out_pairs)
        oracle.swap_blocks([ck, cv], [k, v], in_pairs)
        reps += 1
    el = time.perf_counter() - t
    return {"value": round(reps * 4 * len(blocks) * bb / el / 1e9, 2), "unit": "GB/s",
            "cores": 1, "kind": "oracle",
            "sample": f"C oracle memcpy, 1 thread: {reps} swap out + in rounds of "
                      f"{len(blocks)} blocks x K, V, {el:.1f} s"}


def workspace_for(pa, w, part, dev):
    """The workspace a call with this partition_size needs (one byte when none)."""
    if w.query_start is not None:
        n = pa.pa_chunk_workspace_bytes(w.q.shape[0], w.num_q_heads, w.head_dim,
                                        w.max_context_len, max(part, 0)) if part >= 0 else 0
    else:
        n = pa.pa_decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                         w.max_context_len, w.block_size, max(part, 0)) \
            if part >= 0 else 0
    return torch.empty(max(n, 1), dtype=torch.uint8, device=dev)


def timed_steps(pa, w, steps, warmup, part, dev, flush=None, barrier=None, sampler=None,
                graph=True):
    """Runs `warmup` untimed steps, then exactly `steps` timed ones bracketed by CUDA
    events on the launching stream.  With `graph`, the step (its kernels, in order) is
    captured once into a CUDA graph and the timed steps are replays of it, as a serving
    loop replays its captured step; the per-kernel times then come from `steps` more
    eager steps with events between the kernels.  Returns the total time, per-step times
    and the buffers the e2e leg reuses."""
    out = torch.empty(w.q.shape, dtype=w.dtype, device=dev)
    ws = workspace_for(pa, w, part, dev)
    cow_src = None
    if w.copy_pairs is not None:
        # the CoW copy reads the original tails and writes scratch destinations each step,
        # so the decoded state stays the same from step to step
        pa.pa_copy_blocks([w.k_cache], [w.v_cache], w.copy_pairs)
        cow_src = w.copy_pairs.copy()
    write, decode = step_ops(pa, w)

    def step(e=None):
        if e is not None:
            e[0].record()
        if cow_src is not None:
            pa.pa_copy_blocks([w.k_cache], [w.v_cache], cow_src)
        if e is not None:
            e[1].record()
        write(w.k_new, w.v_new, w.slot_mapping)
        if e is not None:
            e[2].record()
        decode(out, w.q, w.block_tables, w.context_lens, part, ws)
        if e is not None:
            e[3].record()

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    if pa.pa_get_device_error():
        raise RuntimeError("device error word set during warm-up")
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        g.replay()                                   # one untimed replay
        torch.cuda.synchronize()
    run = g.replay if g is not None else step
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    if sampler is not None:
        sampler.start()
    if barrier is not None:
        barrier()
    torch.cuda.synchronize()
    t0_wall = time.time()
    if flush is None:
        for i in range(steps):
            marks[i].record()
            run()
        marks[steps].record()
        torch.cuda.synchronize()
        step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    else:
        end = torch.cuda.Event(enable_timing=True)
        step_ms = []
        for i in range(steps):
            flush.fill_(i & 0xff)
            marks[i].record()
            run()
            end.record()
            torch.cuda.synchronize()
            step_ms.append(marks[i].elapsed_time(end))
    if barrier is not None:
        barrier()
    t1_wall = time.time()
    clocks = sampler.stop(t0_wall, t1_wall) if sampler is not None else None
    torch.cuda.synchronize()
    if pa.pa_get_device_error():
        raise RuntimeError("device error word set during the timed steps")
    # per-kernel times: eager steps with events between the kernels
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        step(ev[i])
    torch.cuda.synchronize()
    if pa.pa_get_device_error():
        raise RuntimeError("device error word set during the per-kernel steps")
    return {"total_ms": sum(step_ms), "step_ms": step_ms, "graph": g is not None,
            "copy_ms": [e[0].elapsed_time(e[1]) for e in ev],
            "reshape_ms": [e[1].elapsed_time(e[2]) for e in ev],
            "decode_ms": [e[2].elapsed_time(e[3]) for e in ev],
            "eager_step_ms": [e[0].elapsed_time(e[3]) for e in ev],
            "clocks": clocks, "out": out, "ws": ws, "copies": cow_src is not None}


def attention_summary(pa, w, config, part, t) -> dict:
    """Roofline of the attention launch and the step's launch count, from one
    timed_steps result: achieved bytes (or flops for long chunks) per average launch."""
    nbytes = algorithmic_bytes(w)
    chunk = w.query_start is not None
    decode_ms = sum(t["decode_ms"]) / len(t["decode_ms"])
    peak, peak_kind = load_peaks()
    achieved = nbytes["decode"] / (decode_ms / 1e3) / 1e9
    split = part > 0 and w.max_context_len > part
    if part == 0:
        split = launched_split(pa, w)
    # an automatic one-pass decode of several waves first builds its longest-first order
    ordered = (not chunk and part == 0 and not split and
               pa.pa_decode_orders_sequences(w.q.dtype, w.k_cache.dtype, w.num_seqs,
                                             w.num_q_heads, w.num_kv_heads, w.head_dim,
                                             w.block_size, w.max_context_len, 0))
    launches = 2 + (1 if split else 0) + (1 if ordered else 0) + (1 if t["copies"] else 0)
    kernel = (dominant_kernel(pa, w) + (" + reduce kernel" if split else "")
              + (" (after the order kernel)" if ordered else ""))
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(config), "kernel": kernel,
                "peak_kind": ("measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs: read + "
                              "write)" if peak_kind == "measured" else "fallback 6.8 TB/s"),
                "algorithmic_bytes_per_launch": nbytes["decode"],
                "nominal_gbs": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4)}
    flops = algorithmic_flops(w)
    tpeak, tpeak_kind = load_tensor_peak()
    if chunk and flops / (tpeak * 1e12) > nbytes["decode"] / (peak * 1e9):
        # bound by the tensor cores: a long chunk makes every K/V byte feed many rows
        tflops = flops / (decode_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(tflops, 1), "peak": tpeak,
                    "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4),
                    "traffic": recorded_traffic(config), "kernel": kernel,
                    "peak_kind": f"{tpeak_kind} dense bf16 (MEASURED_PEAKS.json)",
                    "algorithmic_flops_per_launch": flops,
                    "algorithmic_bytes_per_launch": nbytes["decode"]}
    return {"roofline": roofline, "launches_per_step": launches, "flops": flops,
            "bytes": nbytes, "decode_ms_mean": decode_ms}


def config_row(pa, config, dev, steps, warmup, local, graph=True) -> dict:
    """One workload's throughput for the bench line's `configs` object: a short run of
    its step with its own clock sample."""
    if config == "llama13b_swap":
        return swap_row(pa, dev, steps, warmup, local)
    w = make_workload(config, dev)
    sampler = ClockSampler(local)
    t = timed_steps(pa, w, steps, warmup, 0, dev, sampler=sampler, graph=graph)
    a = attention_summary(pa, w, config, 0, t)
    r = a["roofline"]
    dec, stp = percentiles(t["decode_ms"]), percentiles(t["step_ms"])
    row = {"kernel": r["kernel"], "bound": r["bound"], "achieved": r["achieved"],
           "unit": r["unit"], "peak": r["peak"], "frac": r["frac"], "traffic": r["traffic"],
           "decode_us_p50": round(dec["p50"] * 1e3, 2),
           "decode_us_p10": round(dec["p10"] * 1e3, 2),
           "decode_us_p90": round(dec["p90"] * 1e3, 2),
           "step_us_p50": round(stp["p50"] * 1e3, 2),
           "step_us_mean": round(t["total_ms"] / steps * 1e3, 2),
           "eager_step_us_p50": round(percentiles(t["eager_step_ms"])["p50"] * 1e3, 2),
           "steps": steps, "warmup": warmup, "clocks": t["clocks"]}
    if r["bound"] == "hbm":
        row["frac_of_nominal"] = r["frac_of_nominal"]
    del w, t
    torch.cuda.empty_cache()
    return row


def run_ours(args, rank, world, local):
    import paged_kv_cache_119_gb300 as pa
    from paged_kv_cache_119_gb300 import build as pa_build

    if args.config == "llama13b_swap":
        return run_swap(args, rank, world, local)

    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa_build.build()
    w = make_workload(args.config, dev, args.num_seqs)
    part = 0 if args.partition_size is None else args.partition_size
    chunk = w.query_start is not None
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if args.flush_l2 else None
    sampler = ClockSampler(local) if rank == 0 else None
    barrier = torch.distributed.barrier if world > 1 else None
    t = timed_steps(pa, w, args.steps, args.warmup, part, dev, flush=flush, barrier=barrier,
                    sampler=sampler, graph=not args.eager)
    total_ms = t["total_ms"]
    sec = max_over_ranks(total_ms / 1e3, dev) if world > 1 else total_ms / 1e3
    a = attention_summary(pa, w, args.config, part, t)
    nbytes = a["bytes"]
    value, _ = aggregate([sec], [nbytes["kv"] * args.steps * world])
    value /= 1e9

    e2e = None if args.no_e2e else measure_e2e(args, pa, w, t["out"], t["ws"], part, dev)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None
    roofline = a["roofline"]
    if roofline["bound"] == "hbm" and not args.no_read_probe:
        rp = read_probe_gbs(pa, dev)
        roofline["read_probe_gbs"] = round(rp, 1)
        roofline["frac_of_read_probe"] = round(roofline["achieved"] / rp, 4)
    metric, unit = METRIC, "GB/s"
    flops = a["flops"]
    if roofline["bound"] == "tensor":
        value = flops * args.steps * world / sec / 1e12
        metric, unit = CHUNK_METRIC[args.config], "TFLOP/s"
    elif chunk:
        metric = CHUNK_METRIC[args.config]
    decode_ms = a["decode_ms_mean"]
    dec, stp = percentiles(t["decode_ms"]), percentiles(t["step_ms"])
    line = {
        "metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[w.k_cache.dtype],
        "data": "synthetic",
        "config": {"workload": WORKLOADS[args.config], "name": args.config,
                   "num_seqs": w.num_seqs, "kv_bytes_per_step": nbytes["kv"],
                   "partition_size": part,
                   "l2": ("flushed between steps (512 MB write outside the events)"
                          if flush is not None else
                          f"no flush: KV pool {2 * w.k_cache.numel() * w.k_cache.element_size() / 1e9:.2f} GB "
                          "is larger than the 129 MB L2"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_step": round(total_ms / args.steps * 1e3, 2),
        "decode_us": round(decode_ms * 1e3, 2),
        "reshape_us": round(sum(t["reshape_ms"]) / args.steps * 1e3, 2),
        "step_us_p10": round(stp["p10"] * 1e3, 2), "step_us_p50": round(stp["p50"] * 1e3, 2),
        "step_us_p90": round(stp["p90"] * 1e3, 2),
        "timing": ("replays of the step captured in a CUDA graph; per-kernel times from as "
                   "many eager steps" if t["graph"] else "eager steps"),
        "eager_step_us_p50": round(percentiles(t["eager_step_ms"])["p50"] * 1e3, 2),
        "decode_us_p10": round(dec["p10"] * 1e3, 2),
        "decode_us_p50": round(dec["p50"] * 1e3, 2),
        "decode_us_p90": round(dec["p90"] * 1e3, 2),
        "decode_kv_gbs": round(nbytes["kv"] / (decode_ms / 1e3) / 1e9, 1),
        "roofline": roofline,
        "gpu_launches": a["launches_per_step"] * args.steps,
        "clocks": t["clocks"],
    }
    if chunk:
        line["query_rows"] = int(w.q.shape[0])
        line["attention_tflops"] = round(flops / (decode_ms / 1e3) / 1e12, 2)
    if e2e is not None:
        if chunk and unit == "TFLOP/s":
            e2e["value"] = round(flops / (e2e["ms_per_step"] / 1e3) / 1e12, 2)
            e2e["unit"] = "TFLOP/s"
        line["e2e"] = e2e
    if not args.no_configs and args.num_seqs is None and world == 1:
        del t
        torch.cuda.empty_cache()
        line["configs"] = {c: config_row(pa, c, dev, args.config_steps, args.config_warmup, local,
                                         graph=not args.eager)
                           for c in CONFIG_ROWS if c != args.config}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
    return line


def measure_e2e(args, pa, w, out, ws, part, dev):
    """Same step through the public API with per-step inputs in pinned host memory:
    q, new K/V, slots, block tables and context lengths are packed in one pinned
    buffer and copied host->device as one transfer every step (an engine stages its
    step inputs the same way), then the kernels run on views of the device copy, and
    the output is read back device->host; all inside the timed region."""
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    if w.query_start is not None:
        names = names + ("query_start",)
    offsets, total = {}, 0
    for n in names:
        t = getattr(w, n)
        offsets[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, n):
        t = getattr(w, n)
        nbytes = t.numel() * t.element_size()
        return buf[offsets[n]:offsets[n] + nbytes].view(t.dtype).view(t.shape)

    for n in names:
        view(host_buf, n).copy_(getattr(w, n).cpu())
    devb = {n: view(dev_buf, n) for n in names}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total
    d2h = out_host.numel() * out_host.element_size()

    write, decode = step_ops(pa, w)

    def step():
        dev_buf.copy_(host_buf, non_blocking=True)
        write(devb["k_new"], devb["v_new"], devb["slot_mapping"])
        if w.query_start is not None:
            decode(out, devb["q"], devb["block_tables"], devb["context_lens"], part, ws,
                   devb["query_start"])
        else:
            decode(out, devb["q"], devb["block_tables"], devb["context_lens"], part, ws)
        out_host.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(args.warmup):
        step()
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b.record()
    for _ in range(args.steps):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = b.elapsed_time(e) / args.steps
    return {"value": round(w.kv_bytes() / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ------------------------------------------------------------------------------ oracle arms

def _host_inputs(w):
    h = {n: getattr(w, n).cpu() for n in ("q", "k_cache", "v_cache", "k_new", "v_new",
                                          "slot_mapping", "block_tables", "context_lens")}
    if w.query_start is not None:
        h["query_start"] = w.query_start.cpu()
    if w.fp8:
        h["k_scale"], h["v_scale"] = w.meta["k_scale"].cpu(), w.meta["v_scale"].cpu()
    return h


def _oracle_step(h, w, seqs, threads):
    """The oracle's step on sequences [0, seqs): reshape of their new tokens, then decode."""
    import oracle
    nt = sum(1 for (s, _) in w.meta["new_tokens"] if s < seqs)
    if w.fp8:
        oracle.reshape_and_cache_e4m3(h["k_new"][:nt], h["v_new"][:nt], h["k_cache"],
                                      h["v_cache"], h["slot_mapping"][:nt], w.block_size,
                                      h["k_scale"], h["v_scale"])
    else:
        oracle.reshape_and_cache(h["k_new"][:nt], h["v_new"][:nt], h["k_cache"], h["v_cache"],
                                 h["slot_mapping"][:nt], w.block_size)
    _decode_slice(h, w, 0, seqs, threads)


def _sample_bytes(w, seqs):
    esz = w.k_cache.element_size()
    return int(sum(w.context_lens.tolist()[:seqs])) * w.num_kv_heads * 2 * w.head_dim * esz


def _chunk_rows(h, w, s, j0, j1, threads) -> int:
    """The oracle on rows j0 .. j1-1 of sequence s's chunk (all heads), as a
    one-sequence chunk ending at row j1-1's position.  Returns its attention flops."""
    import oracle
    qs = h["query_start"].tolist()
    n, L = qs[s + 1] - qs[s], int(h["context_lens"][s])
    oracle.chunk_attention(h["q"][qs[s] + j0:qs[s] + j1], h["k_cache"], h["v_cache"],
                           h["block_tables"][s:s + 1],
                           torch.tensor([L - n + j1], dtype=torch.int32),
                           torch.tensor([0, j1 - j0], dtype=torch.int32), w.scale,
                           w.num_kv_heads, w.block_size, num_threads=threads,
                           k_scale=h.get("k_scale"), v_scale=h.get("v_scale"))
    return 4 * w.head_dim * w.num_q_heads * sum(L - n + j + 1 for j in range(j0, j1))


def _chunk_sample(w, h, budget_s, threads):
    """(value, unit, description) of the oracle on a bounded leading sample of a
    chunk workload, in the bench line's unit (KV GB/s or attention TFLOP/s)."""
    qs = h["query_start"].tolist()
    if CHUNK_METRIC.get(w.name, "").endswith("TFLOP/s"):
        t = time.perf_counter()
        flops = _chunk_rows(h, w, 0, 0, 1, threads)
        per_row = max(time.perf_counter() - t, 1e-6)
        rows = max(1, min(qs[1], int(budget_s / per_row)))
        t = time.perf_counter()
        flops = _chunk_rows(h, w, 0, 0, rows, threads)
        el = time.perf_counter() - t
        return (flops / el / 1e12, "TFLOP/s",
                f"fp64 C oracle (OpenMP, {threads} threads): the first {rows} query rows of "
                f"sequence 0's {qs[1]}-token chunk, all heads, {el:.1f} s")
    seqs, el = 0, 0.0
    t = time.perf_counter()
    while seqs < w.num_seqs and el < budget_s:
        _chunk_rows(h, w, seqs, 0, qs[seqs + 1] - qs[seqs], threads)
        seqs += 1
        el = time.perf_counter() - t
    return (_sample_bytes(w, seqs) / el / 1e9, "GB/s",
            f"fp64 C oracle (OpenMP, {threads} threads): the chunks of the first {seqs} of "
            f"{w.num_seqs} sequences, all heads, {el:.1f} s")


def cpu_baseline(w, budget_s: float) -> dict:
    """The oracle, as it stands, on the same workload: whole passes over the batch
    (decode of every sequence, all heads) repeated until about budget_s seconds of
    CPU work, or a leading slice of the batch when one pass would take longer."""
    import oracle
    h = _host_inputs(w)
    if w.query_start is not None:
        threads = oracle.max_threads()
        value, unit, sample = _chunk_sample(w, h, budget_s, threads)
        v1, _, sample1 = _chunk_sample(w, h, budget_s / 3, 1)
        return {"value": round(value, 4), "unit": unit, "cores": threads, "kind": "oracle",
                "sample": sample, "one_thread": {"value": round(v1, 5), "unit": unit,
                                                 "cores": 1, "sample": sample1}}
    threads = oracle.max_threads()
    # calibrate on the first 8 sequences, then size the sample to the budget
    t = time.perf_counter()
    _decode_slice(h, w, 0, min(8, w.num_seqs), threads)
    probe = max(time.perf_counter() - t, 1e-6)
    est_pass = probe * w.kv_bytes() / max(_sample_bytes(w, min(8, w.num_seqs)), 1)
    if est_pass <= budget_s:
        passes, seqs = max(1, int(budget_s / est_pass)), w.num_seqs
    else:
        passes, seqs = 1, w.num_seqs
        while seqs > 8 and probe * (_sample_bytes(w, seqs) / _sample_bytes(w, 8)) > budget_s:
            seqs //= 2
    t = time.perf_counter()
    for _ in range(passes):
        _decode_slice(h, w, 0, seqs, threads)
    elapsed = time.perf_counter() - t
    gbs = passes * _sample_bytes(w, seqs) / elapsed / 1e9
    # the same oracle on one thread: leading sequences until about budget_s / 3 seconds
    n1, t = 0, time.perf_counter()
    while n1 < w.num_seqs and (n1 == 0 or time.perf_counter() - t < budget_s / 3):
        _decode_slice(h, w, n1, n1 + 1, 1)
        n1 += 1
    el1 = time.perf_counter() - t
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 C oracle (OpenMP, {threads} threads): {passes} pass(es) over the "
                      f"first {seqs} of {w.num_seqs} sequences, all heads, {elapsed:.1f} s",
            "one_thread": {"value": round(_sample_bytes(w, n1) / el1 / 1e9, 4), "unit": "GB/s",
                           "cores": 1,
                           "sample": f"fp64 C oracle, 1 thread: the first {n1} of {w.num_seqs} "
                                     f"sequences, all heads, {el1:.1f} s"}}


def _decode_slice(h, w, s0, s1, threads):
    import oracle
    oracle.paged_attention(h["q"][s0:s1], h["k_cache"], h["v_cache"], h["block_tables"][s0:s1],
                           h["context_lens"][s0:s1], w.scale, w.num_kv_heads, w.block_size,
                           num_threads=threads, k_scale=h.get("k_scale"),
                           v_scale=h.get("v_scale"))


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    if args.config == "llama13b_swap":
        w = make_workload("llama13b", "cpu", args.num_seqs)
        blocks, bb = swap_plan(w, min(64, w.num_seqs))
        for _ in range(args.warmup):
            swap_cpu_baseline(w, blocks, bb, 0.0)
        t = time.perf_counter()
        vals = [swap_cpu_baseline(w, blocks, bb, 0.0) for _ in range(args.steps)]
        sec = (time.perf_counter() - t) / args.steps
        value = sum(v["value"] for v in vals) / len(vals)
        return {"impl": "reference", "metric": SWAP_METRIC, "value": round(value, 2),
                "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bytes", "data": "synthetic",
                "config": {"workload": WORKLOADS[args.config], "name": args.config},
                "cpu_baseline": dict(vals[-1], value=round(value, 2)),
                "e2e": {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
    w = make_workload(args.config, "cpu", args.num_seqs)
    h = _host_inputs(w)
    threads = oracle.max_threads()
    if w.query_start is not None:
        # each step: the oracle on a bounded leading sample (about 0.5 s of work)
        for _ in range(args.warmup):
            _chunk_sample(w, h, 0.5, threads)
        vals = []
        t = time.perf_counter()
        for _ in range(args.steps):
            value, unit, sample = _chunk_sample(w, h, 0.5, threads)
            vals.append(value)
        sec = (time.perf_counter() - t) / args.steps
        value = sum(vals) / len(vals)
        return {"impl": "reference", "metric": CHUNK_METRIC[args.config],
                "value": round(value, 4), "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOADS[args.config], "name": args.config,
                           "num_seqs": w.num_seqs},
                "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": threads,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
    # a bounded sample: enough sequences for ~0.5 s of oracle work per step
    seqs = max(1, min(w.num_seqs, 16))
    for _ in range(args.warmup):
        _oracle_step(h, w, seqs, threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(h, w, seqs, threads)
    sec = (time.perf_counter() - t) / args.steps
    value = _sample_bytes(w, seqs) / sec / 1e9
    sample = (f"fp64 C oracle (OpenMP, {threads} threads): reshape + decode of the first {seqs} "
              f"of {w.num_seqs} sequences per step")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.config], "name": args.config,
                       "num_seqs": w.num_seqs, "sampled_seqs": seqs},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.run_probe:
        torch.cuda.set_device(local)
        line = run_probe(torch.device("cuda", local)) if rank == 0 else None
    else:
        line = run_reference(args, rank, world) if args.impl == "reference" else \
            run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
