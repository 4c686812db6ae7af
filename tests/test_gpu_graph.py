"""A step captured in a CUDA graph and replayed gives the eager step's bytes (GPU).

A serving loop captures its decode step once and replays it.  Every call on the step
(block copy, cache write, decode or chunk attention, with a workspace and so with the
on-device longest-first order) takes its sizes and pointers at capture time and
allocates or synchronises nothing, so replays must reproduce the eager output bit for
bit.  The step is idempotent (the same new tokens land in the same slots, the same
blocks are copied), so eager and replayed outputs compare directly; the eager output is
checked against the oracle as well, so a replay that repeats a stale buffer still fails.
"""
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ATOL = 2e-3

CASES = {
    "llama13b": dict(num_seqs=24),
    "prefix": dict(num_groups=2),
    "long16": dict(num_seqs=2, context=3000),
    "llama13b_fp8": dict(num_seqs=24),
    "long16_fp8": dict(num_seqs=2, context=3000),
    "llama13b_verify4": dict(num_seqs=12),
    "long16_chunk512": dict(num_seqs=2, context=1500, query_len=300),
}


def _make(name):
    fp8 = name.endswith("_fp8")
    w = workloads.make(name[:-4] if fp8 else name, device="cuda", **CASES[name])
    return workloads.to_fp8(w) if fp8 else w


def _step_fn(w, out, ws):
    pairs = w.copy_pairs

    def step():
        if pairs is not None:
            P.pa_copy_blocks([w.k_cache], [w.v_cache], pairs)
        if w.fp8:
            ks, vs = w.meta["k_scale"], w.meta["v_scale"]
            P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping,
                                       ks, vs)
        else:
            P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
        if w.query_start is not None:
            kw = dict(max_query_len=w.max_query_len, max_context_len=w.max_context_len,
                      partition_size=0, workspace=ws)
            if w.fp8:
                P.pa_chunk_attention_fp8(out, w.q, w.k_cache, w.v_cache, w.meta["k_scale"],
                                         w.meta["v_scale"], w.block_tables, w.context_lens,
                                         w.query_start, w.scale, w.num_kv_heads, w.block_size,
                                         **kw)
            else:
                P.pa_chunk_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables,
                                     w.context_lens, w.query_start, w.scale, w.num_kv_heads,
                                     w.block_size, **kw)
        elif w.fp8:
            P.pa_decode_fp8(out, w.q, w.k_cache, w.v_cache, w.meta["k_scale"], w.meta["v_scale"],
                            w.block_tables, w.context_lens, w.scale, w.num_kv_heads,
                            w.block_size, max_context_len=w.max_context_len, partition_size=0,
                            workspace=ws)
        else:
            P.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                        w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                        partition_size=0, workspace=ws)
    return step


def _workspace(w):
    if w.query_start is not None:
        n = P.pa_chunk_workspace_bytes(w.q.shape[0], w.num_q_heads, w.head_dim,
                                       w.max_context_len, 0)
    else:
        n = P.pa_decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                        w.max_context_len, w.block_size, 0)
    return torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")


def _bytes(t):
    return t.contiguous().view(torch.uint8)


def _oracle(w):
    sc = dict(k_scale=w.meta["k_scale"].cpu(), v_scale=w.meta["v_scale"].cpu()) if w.fp8 else {}
    args = (w.q.cpu(), w.k_cache.cpu(), w.v_cache.cpu(), w.block_tables.cpu(),
            w.context_lens.cpu())
    if w.query_start is not None:
        return oracle.chunk_attention(*args, w.query_start.cpu(), w.scale, w.num_kv_heads,
                                      w.block_size, num_threads=oracle.max_threads(), **sc)
    return oracle.paged_attention(*args, w.scale, w.num_kv_heads, w.block_size,
                                  num_threads=oracle.max_threads(), **sc)


@pytest.mark.parametrize("name", list(CASES))
def test_replayed_step_matches_eager_step(name):
    P.pa_get_device_error()
    w = _make(name)
    ws = _workspace(w)
    eager = torch.full(w.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    step = _step_fn(w, eager, ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = eager.clone()
    k_want, v_want = _bytes(w.k_cache).clone(), _bytes(w.v_cache).clone()

    replayed = torch.full(w.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step_fn(w, replayed, ws)()
    for _ in range(3):
        replayed.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(replayed.view(torch.int32), want.view(torch.int32))
    # unused cache slots hold NaN, so the caches compare as bytes
    assert torch.equal(_bytes(w.k_cache), k_want) and torch.equal(_bytes(w.v_cache), v_want)
    assert P.pa_get_device_error() == 0

    ref = _oracle(w)
    err = (want.cpu().double() - torch.from_numpy(ref)).abs().max().item()
    assert err <= ATOL, f"{name}: max |eager - oracle| = {err:.3g}"
