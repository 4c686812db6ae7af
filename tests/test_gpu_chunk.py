"""Chunk attention (several new query tokens per sequence, attended causally over the
paged cache) on the GPU against the CPU oracle.

Each case runs the step as a caller would: pa_reshape_and_cache writes the chunk's
K/V rows (bit-exact against the oracle's byte copy), then pa_chunk_attention; the
attention output is compared element by element with the oracle's fp64 result
(max abs error <= 2e-3 on fp32 output; native output must be the round-to-nearest-
even of a value within 5e-5 of the oracle on the decode kernels' multi-row mode, whose
probabilities carry fp32-level accuracy, and within 2e-3 on the tcgen05 chunk kernel,
whose probabilities are one f16 term).  Head groupings 1, 4, 5 and 8, head_dim
64 / 128, block_size 16 / 32, fp16 / bf16, ragged chunks (n = L, n = 1, n = 0),
forced and automatic context splits.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ATOL = 2e-3
NATIVE_EPS = 5e-5


def native_eps(w):
    """Half-width of the native-output bracket: the attention tolerance on the tcgen05
    chunk kernel (one f16 rounding of each probability: up to 2^-11 of max |v|), 5e-5
    where the probabilities enter P.V as hi + lo halves."""
    name = P.pa_chunk_kernel_name(w.k_cache.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                  w.max_query_len)
    return ATOL if name.startswith("chunk_attn_kernel") else NATIVE_EPS


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


@pytest.fixture(autouse=True)
def clear_error_word(built):
    P.pa_get_device_error()
    yield


def make_case(seed, S, Hq, Hkv, D, B, dtype, lens, chunks, std=1.0):
    rng = np.random.default_rng(seed)
    return workloads._assemble("chunk_case", rng, "cuda", lens=lens, Hq=Hq, Hkv=Hkv, D=D, B=B,
                               dtype=dtype, std=std, chunk=chunks)


def run_and_compare(w, out_dtype=torch.float32, partition_size=0, check_caches=True):
    snap = {n: getattr(w, n).cpu() for n in ("q", "k_cache", "v_cache", "k_new", "v_new",
                                             "slot_mapping", "block_tables", "context_lens",
                                             "query_start")}
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = torch.empty(w.q.shape, dtype=out_dtype, device="cuda")
    P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                         w.query_start, w.scale, w.num_kv_heads, w.block_size,
                         max_query_len=w.max_query_len, max_context_len=w.max_context_len,
                         partition_size=partition_size)
    torch.cuda.synchronize()
    kc, vc = snap["k_cache"].clone(), snap["v_cache"].clone()
    oracle.reshape_and_cache(snap["k_new"], snap["v_new"], kc, vc, snap["slot_mapping"],
                             w.block_size)
    if check_caches:
        assert torch.equal(w.k_cache.cpu().view(torch.int16), kc.view(torch.int16))
        assert torch.equal(w.v_cache.cpu().view(torch.int16), vc.view(torch.int16))
    ref = oracle.chunk_attention(snap["q"], kc, vc, snap["block_tables"], snap["context_lens"],
                                 snap["query_start"], w.scale, w.num_kv_heads, w.block_size,
                                 num_threads=oracle.max_threads())
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    if out_dtype == torch.float32:
        err = np.abs(got - ref).max() if got.size else 0.0
        assert err <= ATOL, f"max abs error {err:.3e}"
    else:
        eps = native_eps(w)
        lo = torch.from_numpy((ref - eps).astype(np.float32)).to(out_dtype).double().numpy()
        hi = torch.from_numpy((ref + eps).astype(np.float32)).to(out_dtype).double().numpy()
        bad = (got < lo) | (got > hi)
        assert not bad.any(), f"{bad.sum()} outputs outside the rounding bracket"
    assert P.pa_get_device_error() == 0
    return got, ref


def test_verify4_llama13b_shape():
    """Speculative verification of 4 tokens per sequence on the LLaMA-13B batch shape
    (MHA: one chunk token row per CTA row group)."""
    w = workloads.make("llama13b_verify4", device="cuda", num_seqs=12)
    run_and_compare(w)


@pytest.mark.parametrize("part", [0, 512, -1])
def test_chunk512_long_context_shape(part):
    """A chunked-prefill step (GQA 8) on a shortened long-context configuration."""
    w = workloads.make("long16_chunk512", device="cuda", num_seqs=2, context=1500,
                       query_len=300)
    run_and_compare(w, partition_size=part)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4), (40, 8), (64, 8)])
@pytest.mark.parametrize("D,B", [(128, 16), (64, 32), (128, 32), (64, 16)])
def test_head_groupings(Hq, Hkv, D, B):
    rng = np.random.default_rng(Hq * 1000 + D + B)
    lens = [1, 17, 64, 65, 129, 300]
    chunks = [1, 17, 1, 30, 129, 77]         # n = L, n = 1, ragged
    w = make_case(int(rng.integers(1 << 30)), len(lens), Hq, Hkv, D, B, torch.bfloat16, lens,
                  chunks)
    run_and_compare(w)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_native_output(dtype):
    w = make_case(7, 4, 32, 8, 128, 16, dtype, [40, 200, 513, 90], [40, 16, 100, 3])
    run_and_compare(w, out_dtype=dtype)


@pytest.mark.parametrize("part", [64, 128, 192, 0, -1])
def test_forced_splits(part):
    """Partition boundaries inside and at the edges of the causal diagonal."""
    w = make_case(11, 3, 16, 2, 128, 16, torch.float16, [700, 130, 1025], [200, 130, 64])
    run_and_compare(w, partition_size=part)


def test_empty_chunks_and_short_contexts():
    """Sequences with no new token own no rows; n = L = 1 is a single-token prefill."""
    w = make_case(13, 5, 8, 2, 64, 16, torch.bfloat16, [1, 50, 9, 33, 2], [1, 0, 9, 0, 2])
    got, ref = run_and_compare(w)
    assert got.shape[0] == 12


def test_single_token_chunks_match_decode():
    """n = 1 for every sequence is decode: the chunk kernel agrees with pa_decode."""
    w = workloads.make("llama13b_verify4", device="cuda", num_seqs=16, query_len=1)
    # query_len 1 builds a decode workload; give it a query_start of one row each
    qs = torch.arange(w.num_seqs + 1, dtype=torch.int32, device="cuda")
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    a = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    P.pa_chunk_attention(a, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, qs,
                         w.scale, w.num_kv_heads, w.block_size, max_query_len=1,
                         max_context_len=w.max_context_len)
    P.pa_decode(b, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                w.num_kv_heads, w.block_size, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert (a - b).abs().max().item() <= 2 * ATOL
    assert P.pa_get_device_error() == 0


def test_full_size_sampled_rows():
    """The full 8 x 32768-token, 512-token chunk step at the launch configuration the
    benchmark times; sampled rows are checked against the oracle one by one."""
    w = workloads.make("long16_chunk512", device="cuda")
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                         w.query_start, w.scale, w.num_kv_heads, w.block_size,
                         max_query_len=w.max_query_len, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() == 0
    rng = np.random.default_rng(5)
    qs = w.query_start.cpu().tolist()
    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    bt, cl = w.block_tables.cpu(), w.context_lens.cpu()
    for s in rng.choice(w.num_seqs, size=2, replace=False).tolist():
        for j in sorted(rng.choice(qs[s + 1] - qs[s], size=3, replace=False).tolist()) + [0]:
            # one row as a one-sequence chunk of length j + 1 ending at its position
            L = int(cl[s]) - (qs[s + 1] - qs[s]) + j + 1
            ref = oracle.chunk_attention(w.q[qs[s] + j:qs[s] + j + 1].cpu(), kc, vc, bt[s:s + 1],
                                         torch.tensor([L], dtype=torch.int32),
                                         torch.tensor([0, 1], dtype=torch.int32), w.scale,
                                         w.num_kv_heads, w.block_size,
                                         num_threads=oracle.max_threads())
            got = out[qs[s] + j].double().cpu().numpy()
            err = np.abs(got - ref[0]).max()
            assert err <= ATOL, (s, j, err)


def test_chunk_longer_than_context_is_flagged():
    """n > L is malformed: the kernel flags it and that sequence's rows are NaN."""
    w = make_case(17, 3, 8, 8, 128, 16, torch.bfloat16, [30, 40, 50], [5, 6, 7])
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    bad_lens = w.context_lens.clone()
    bad_lens[1] = 3                                   # 6 new tokens, context 3
    out = torch.zeros(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, bad_lens,
                         w.query_start, w.scale, w.num_kv_heads, w.block_size,
                         max_query_len=7, max_context_len=50)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() & 0x2
    assert torch.isnan(out[5:11]).all()
    assert torch.isfinite(out[:5]).all() and torch.isfinite(out[11:]).all()


def test_bad_block_id_is_flagged():
    w = make_case(19, 2, 8, 2, 64, 16, torch.float16, [100, 80], [10, 20])
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    bt = w.block_tables.clone()
    bt[0, 2] = w.num_blocks + 5
    out = torch.zeros(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.query_start,
                         w.scale, w.num_kv_heads, w.block_size, max_query_len=20,
                         max_context_len=100)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() & 0x1
    assert torch.isnan(out[:10]).all()
    assert torch.isfinite(out[10:]).all()


def test_canaries_around_output():
    w = make_case(23, 3, 16, 4, 128, 32, torch.bfloat16, [77, 150, 33], [20, 45, 33])
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    R, Hq, D = w.q.shape
    buf = torch.full((R * Hq * D + 2 * 4096,), 12345.0, dtype=torch.float32, device="cuda")
    out = buf[4096:4096 + R * Hq * D].view(R, Hq, D)
    P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                         w.query_start, w.scale, w.num_kv_heads, w.block_size,
                         max_query_len=45, max_context_len=150, partition_size=64)
    torch.cuda.synchronize()
    assert (buf[:4096] == 12345.0).all() and (buf[-4096:] == 12345.0).all()
    assert torch.isfinite(out).all()
    assert P.pa_get_device_error() == 0


@pytest.mark.parametrize("Hq,Hkv,nmax", [(8, 8, 3), (8, 8, 4), (40, 40, 4), (16, 4, 2),
                                         (16, 4, 8), (40, 8, 6), (64, 8, 4), (64, 8, 1)])
@pytest.mark.parametrize("D,B", [(128, 16), (64, 32), (128, 32)])
def test_short_chunks_few_rows(Hq, Hkv, nmax, D, B):
    """At most 32 (token, head) rows per kv head -- speculative verification, short
    chunks -- run on the mma.sync decode kernel in its chunk-row mode."""
    rng = np.random.default_rng(Hq * 7919 + nmax * 31 + D + B)
    lens = [int(x) for x in rng.integers(1, 600, size=7)] + [nmax, 1]
    chunks = [min(L, int(rng.integers(0, nmax + 1))) for L in lens]
    chunks[0] = min(lens[0], nmax)
    w = make_case(int(rng.integers(1 << 30)), len(lens), Hq, Hkv, D, B, torch.bfloat16, lens,
                  chunks)
    run_and_compare(w)


@pytest.mark.parametrize("part", [0, 64, 256, -1])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_short_chunks_splits_and_native_output(part, out_dtype):
    w = make_case(29, 4, 32, 8, 128, 16, torch.float16, [3000, 700, 64, 1], [4, 4, 2, 1])
    run_and_compare(w, out_dtype=out_dtype, partition_size=part)


def test_verify4_full_batch_sampled_rows():
    """The full 256-sequence verification step at the benchmark's launch configuration;
    sampled rows against the oracle."""
    w = workloads.make("llama13b_verify4", device="cuda")
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                         w.query_start, w.scale, w.num_kv_heads, w.block_size,
                         max_query_len=w.max_query_len, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() == 0
    rng = np.random.default_rng(6)
    seqs = sorted(rng.choice(w.num_seqs, size=12, replace=False).tolist())
    qs = w.query_start.cpu()
    rows = torch.cat([torch.arange(int(qs[s]), int(qs[s + 1])) for s in seqs])
    sub_qs = torch.tensor(np.concatenate([[0], np.cumsum([int(qs[s + 1] - qs[s]) for s in seqs])]),
                          dtype=torch.int32)
    ref = oracle.chunk_attention(w.q[rows.cuda()].cpu(), w.k_cache.cpu(), w.v_cache.cpu(),
                                 w.block_tables.cpu()[seqs], w.context_lens.cpu()[seqs], sub_qs,
                                 w.scale, w.num_kv_heads, w.block_size,
                                 num_threads=oracle.max_threads())
    err = np.abs(out[rows.cuda()].double().cpu().numpy() - ref).max()
    assert err <= ATOL, err


# ------------------------------------------------------------------- E4M3 caches

def run_and_compare_fp8(w, out_dtype=torch.float32, partition_size=0):
    ks, vs = w.meta["k_scale"], w.meta["v_scale"]
    snap = {n: getattr(w, n).cpu() for n in ("q", "k_cache", "v_cache", "k_new", "v_new",
                                             "slot_mapping", "block_tables", "context_lens",
                                             "query_start")}
    P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, ks, vs)
    out = torch.empty(w.q.shape, dtype=out_dtype, device="cuda")
    P.pa_chunk_attention_fp8(out, w.q, w.k_cache, w.v_cache, ks, vs, w.block_tables,
                             w.context_lens, w.query_start, w.scale, w.num_kv_heads, w.block_size,
                             max_query_len=w.max_query_len, max_context_len=w.max_context_len,
                             partition_size=partition_size)
    torch.cuda.synchronize()
    kc, vc = snap["k_cache"].view(torch.uint8).clone(), snap["v_cache"].view(torch.uint8).clone()
    oracle.reshape_and_cache_e4m3(snap["k_new"], snap["v_new"], kc, vc, snap["slot_mapping"],
                                  w.block_size, ks.cpu(), vs.cpu())
    assert torch.equal(w.k_cache.cpu().view(torch.uint8), kc)
    assert torch.equal(w.v_cache.cpu().view(torch.uint8), vc)
    ref = oracle.chunk_attention(snap["q"], kc, vc, snap["block_tables"], snap["context_lens"],
                                 snap["query_start"], w.scale, w.num_kv_heads, w.block_size,
                                 num_threads=oracle.max_threads(), k_scale=ks.cpu(),
                                 v_scale=vs.cpu())
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    if out_dtype == torch.float32:
        err = np.abs(got - ref).max()
        assert err <= ATOL, f"max abs error {err:.3e}"
    else:
        eps = native_eps(w)
        lo = torch.from_numpy((ref - eps).astype(np.float32)).to(out_dtype).double().numpy()
        hi = torch.from_numpy((ref + eps).astype(np.float32)).to(out_dtype).double().numpy()
        assert not ((got < lo) | (got > hi)).any()
    assert P.pa_get_device_error() == 0


def test_fp8_verify4_llama13b_shape():
    w = workloads.to_fp8(workloads.make("llama13b_verify4", device="cuda", num_seqs=12))
    run_and_compare_fp8(w)


@pytest.mark.parametrize("Hq,Hkv,nmax", [(8, 8, 4), (16, 4, 8), (40, 8, 3), (64, 8, 4), (64, 8, 40)])
@pytest.mark.parametrize("D,B", [(128, 16), (64, 32)])
@pytest.mark.parametrize("qdtype", [torch.bfloat16, torch.float16])
def test_fp8_chunks(Hq, Hkv, nmax, D, B, qdtype):
    """Short and long chunks over E4M3 caches (every length runs on the multi-row
    decode kernel), every grouping, both head dims, bf16 and f16 queries."""
    rng = np.random.default_rng(Hq + 13 * nmax + D + B)
    lens = [int(x) for x in rng.integers(1, 500, size=6)] + [nmax]
    chunks = [min(L, int(rng.integers(0, nmax + 1))) for L in lens]
    chunks[-1] = nmax
    w = make_case(int(rng.integers(1 << 30)), len(lens), Hq, Hkv, D, B, qdtype, lens, chunks)
    run_and_compare_fp8(workloads.to_fp8(w))


@pytest.mark.parametrize("part", [0, 64, -1])
def test_fp8_chunk_splits_and_native_output(part):
    w = make_case(41, 3, 32, 8, 128, 16, torch.bfloat16, [2500, 300, 40], [4, 2, 4])
    run_and_compare_fp8(workloads.to_fp8(w), out_dtype=torch.bfloat16, partition_size=part)


# ------------------------------------- long chunks over E4M3 caches (tcgen05, f16 stage)

@pytest.mark.parametrize("Hq,Hkv,nmax", [(32, 4, 100), (64, 8, 70), (40, 40, 40)])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("qdtype", [torch.bfloat16, torch.float16])
def test_fp8_long_chunks_on_tensor_cores(Hq, Hkv, nmax, B, qdtype):
    """More than 32 (token, head) rows per kv head over an E4M3 cache at head_dim 128:
    the tcgen05 chunk kernel with its E4M3 -> f16 conversion stage (ragged chunks,
    several 128-row query tiles, contexts from one tile to many)."""
    rng = np.random.default_rng(Hq + 7 * nmax + B)
    lens = [nmax, 3000, 700, 130, 64, 65]
    chunks = [nmax, nmax, int(rng.integers(33, nmax + 1)), nmax // 2, 40, 1]
    chunks = [min(c, L) for c, L in zip(chunks, lens)]
    w = make_case(int(rng.integers(1 << 30)), len(lens), Hq, Hkv, 128, B, qdtype, lens, chunks)
    run_and_compare_fp8(workloads.to_fp8(w))


@pytest.mark.parametrize("part", [0, 64, 192, -1])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_long_chunk_splits_and_native_output(part, out_dtype):
    w = make_case(43, 3, 64, 8, 128, 16, torch.bfloat16, [4100, 900, 200], [96, 64, 40])
    run_and_compare_fp8(workloads.to_fp8(w), out_dtype=out_dtype, partition_size=part)


def _magnitude_case(fp8):
    w = make_case(47, 2, 32, 4, 128, 16, torch.bfloat16, [600, 300], [80, 50])
    if fp8:
        w = workloads.to_fp8(w)
    q = w.q.float()
    q[:10] *= 3e4
    q[10:20] *= 1e-6
    w.q.copy_(q.to(torch.bfloat16))
    w.scale = w.scale / 3e4 * 10        # keep the large rows' scores moderate
    return w


@pytest.mark.parametrize("fp8", [False, True])
def test_long_chunk_query_magnitudes(fp8):
    """Rows of very different size (over E4M3 caches each bf16 row is scaled into f16 by
    its own power of two).  The huge rows make their softmax warps rescale O on the last
    tile and reach the epilogue late, when P.V of the last two tiles may both be done;
    three runs, since that timing varies."""
    for _ in range(3):
        w = _magnitude_case(fp8)
        if fp8:
            run_and_compare_fp8(w)
        else:
            run_and_compare(w)


def _sampled_rows_fp8(w, picks):
    """Checks rows (s, j) of a chunk step over E4M3 caches one by one against the oracle,
    each as a one-row chunk ending at its position."""
    ks, vs = w.meta["k_scale"], w.meta["v_scale"]
    P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, ks, vs)
    out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_chunk_attention_fp8(out, w.q, w.k_cache, w.v_cache, ks, vs, w.block_tables,
                             w.context_lens, w.query_start, w.scale, w.num_kv_heads, w.block_size,
                             max_query_len=w.max_query_len, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() == 0
    qs = w.query_start.cpu().tolist()
    kc, vc = w.k_cache.view(torch.uint8).cpu(), w.v_cache.view(torch.uint8).cpu()
    bt, cl = w.block_tables.cpu(), w.context_lens.cpu()
    for s, j in picks:
        L = int(cl[s]) - (qs[s + 1] - qs[s]) + j + 1
        ref = oracle.chunk_attention(w.q[qs[s] + j:qs[s] + j + 1].cpu(), kc, vc, bt[s:s + 1],
                                     torch.tensor([L], dtype=torch.int32),
                                     torch.tensor([0, 1], dtype=torch.int32), w.scale,
                                     w.num_kv_heads, w.block_size,
                                     num_threads=oracle.max_threads(), k_scale=ks.cpu(),
                                     v_scale=vs.cpu())
        err = np.abs(out[qs[s] + j].double().cpu().numpy() - ref[0]).max()
        assert err <= ATOL, (s, j, err)


def test_fp8_chunk512_full_size_sampled_rows():
    """The full 8 x 32768-token, 512-token chunk step over E4M3 caches (the tcgen05
    kernel with its f16 conversion stage) at the benchmark's launch configuration."""
    w = workloads.to_fp8(workloads.make("long16_chunk512", device="cuda"))
    rng = np.random.default_rng(8)
    picks = [(s, j) for s in rng.choice(w.num_seqs, size=2, replace=False).tolist()
             for j in sorted(rng.choice(512, size=3, replace=False).tolist()) + [0, 511]]
    _sampled_rows_fp8(w, picks)


def test_fp8_verify4_full_batch_sampled_rows():
    """The full 256-sequence verification step over E4M3 caches (decode_tc8_kernel's
    chunk-row mode) at the benchmark's launch configuration."""
    w = workloads.to_fp8(workloads.make("llama13b_verify4", device="cuda"))
    rng = np.random.default_rng(9)
    qs = w.query_start.cpu().tolist()
    picks = [(s, j) for s in rng.choice(w.num_seqs, size=10, replace=False).tolist()
             for j in range(qs[s + 1] - qs[s])]
    _sampled_rows_fp8(w, picks)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("Hq,Hkv,nmax", [(8, 8, 40), (16, 4, 8), (8, 8, 4)])
def test_rows_beyond_the_last_chunk_are_flagged(fp8, Hq, Hkv, nmax):
    """q with rows after query_start[num_seqs] (owned by no sequence) sets the
    context-length error bit on every path (the tcgen05 chunk kernel, and both decode
    kernels' chunk-row modes); the owned rows are still the oracle's."""
    w = make_case(53 + nmax, 3, Hq, Hkv, 128, 16, torch.bfloat16, [300, 90, 200],
                  [nmax, nmax // 2 + 1, nmax])
    if fp8:
        w = workloads.to_fp8(w)
    ks = w.meta["k_scale"] if fp8 else None
    vs = w.meta["v_scale"] if fp8 else None
    if fp8:
        P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, ks, vs)
    else:
        P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    R = w.q.shape[0]
    q2 = torch.cat([w.q, torch.zeros_like(w.q[:3])])
    out = torch.zeros((R + 3,) + tuple(w.q.shape[1:]), dtype=torch.float32, device="cuda")
    args = (w.block_tables, w.context_lens, w.query_start, w.scale, w.num_kv_heads, w.block_size)
    kw = dict(max_query_len=w.max_query_len, max_context_len=w.max_context_len)
    P.pa_get_device_error()
    if fp8:
        P.pa_chunk_attention_fp8(out, q2, w.k_cache, w.v_cache, ks, vs, *args, **kw)
    else:
        P.pa_chunk_attention(out, q2, w.k_cache, w.v_cache, *args, **kw)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() & 0x2
    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    if fp8:
        kc, vc = kc.view(torch.uint8), vc.view(torch.uint8)
    ref = oracle.chunk_attention(w.q.cpu(), kc, vc, w.block_tables.cpu(), w.context_lens.cpu(),
                                 w.query_start.cpu(), w.scale, w.num_kv_heads, w.block_size,
                                 num_threads=oracle.max_threads(),
                                 k_scale=None if ks is None else ks.cpu(),
                                 v_scale=None if vs is None else vs.cpu())
    err = np.abs(out[:R].double().cpu().numpy() - ref).max()
    assert err <= ATOL, err


# ------------------- the tcgen05 chunk kernel: one f16 rounding of each probability

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_tensor_core_probabilities_within_their_f16_bound(dtype):
    """Values four times larger (peaked rows, |v| up to about 20) on the tcgen05 chunk
    kernel: each probability enters P.V as one f16 rounding (2^-11 relative), so the
    output is within 2^-11 of the largest |v| of the cache, plus fp32 rounding."""
    w = make_case(59, 3, 32, 8, 128, 16, dtype, [900, 2100, 130], [100, 64, 40], std=4.0)
    assert P.pa_chunk_kernel_name(w.k_cache.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                  w.max_query_len).startswith("chunk_attn_kernel")
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                         w.query_start, w.scale, w.num_kv_heads, w.block_size,
                         max_query_len=w.max_query_len, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() == 0
    ref = oracle.chunk_attention(w.q.cpu(), w.k_cache.cpu(), w.v_cache.cpu(),
                                 w.block_tables.cpu(), w.context_lens.cpu(), w.query_start.cpu(),
                                 w.scale, w.num_kv_heads, w.block_size,
                                 num_threads=oracle.max_threads())
    vmax = torch.nan_to_num(w.v_cache.float(), nan=0.0).abs().max().item()   # unused slots: NaN
    err = np.abs(out.double().cpu().numpy() - ref).max()
    assert err <= 2.0 ** -11 * vmax + 1e-4, (err, vmax)


def test_bf16_value_outside_f16_range_is_flagged():
    """The tcgen05 chunk kernel multiplies P with V in f16, so over a bf16 cache a
    context value with |v| >= 65536 has no f16 value: the rows that weigh it are not
    finite and set PA_DEVERR_RANGE; every other row is the oracle's.  The largest bf16
    value below that (65280) converts exactly and sets nothing."""
    from paged_kv_cache_119_gb300 import _native as N
    for value, flagged in ((65280.0, False), (1.0e5, True)):
        w = make_case(61, 2, 32, 8, 128, 16, torch.bfloat16, [300, 200], [100, 50])
        assert P.pa_chunk_kernel_name(w.k_cache.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                      w.max_query_len).startswith("chunk_attn_kernel")
        P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
        kvh = 3
        w.v_cache[int(w.block_tables[0, 0]), kvh, 5, 17] = value    # sequence 0, position 5
        out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
        P.pa_get_device_error()
        P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                             w.query_start, w.scale, w.num_kv_heads, w.block_size,
                             max_query_len=w.max_query_len, max_context_len=w.max_context_len)
        torch.cuda.synchronize()
        flags = P.pa_get_device_error()
        assert flags == (N.PA_DEVERR_RANGE if flagged else 0), hex(flags)
        ref = oracle.chunk_attention(w.q.cpu(), w.k_cache.cpu(), w.v_cache.cpu(),
                                     w.block_tables.cpu(), w.context_lens.cpu(),
                                     w.query_start.cpu(), w.scale, w.num_kv_heads, w.block_size,
                                     num_threads=oracle.max_threads())
        got = out.double().cpu().numpy()
        G = w.num_q_heads // w.num_kv_heads
        heads = slice(kvh * G, (kvh + 1) * G)
        n0 = int(w.query_start[1])                # sequence 0's rows
        hit = np.zeros(got.shape, dtype=bool)
        hit[:n0, heads, :] = True
        if flagged:
            assert not np.isfinite(got[:n0, heads, 17]).any()
        else:
            # the rows that weigh 65280: within 2^-11 of it (one f16 rounding per weight)
            assert np.abs(got[hit] - ref[hit]).max() <= 2.0 ** -11 * value
        assert np.abs(got[~hit] - ref[~hit]).max() <= ATOL
