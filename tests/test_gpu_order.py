"""Longest-first dispatch of one-pass decodes, on the GPU through the C ABI.

An automatic (partition_size 0) pa_decode call on the CUDA-core decode kernel whose grid
holds more CTAs than fit on the GPU at once first sorts its sequences into length
classes, longest first, in the caller's workspace; CTA row z then serves the z-th
sequence of that order.  Each (sequence, head) is still computed by one CTA, so the
output must be bitwise the output of the same call in index order (a workspace too
small for the order turns it off), and within the usual tolerance of the oracle.
Output buffers start as NaN, so a sequence the order dropped or served twice shows.
The tensor-core decode kernels keep the index order (they were measured slower in the
other).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL = 2e-3

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


@pytest.fixture(autouse=True)
def clear_error_word(built):
    P.pa_get_device_error()
    yield


def lengths(S, seed, max_len=2048):
    """Serving-like mix: lognormal around 400 tokens, with empty, one-token and
    full-length contexts placed late in the batch."""
    rng = np.random.default_rng(seed)
    lens = np.clip(np.exp(rng.normal(np.log(400), 0.8, size=S)), 1, max_len).astype(int).tolist()
    lens[-1], lens[-2], lens[-3], lens[-4] = max_len, 0, 1, max_len - 1
    return lens


def make(S, Hq, Hkv, D, B, dtype, fp8, seed):
    rng = np.random.default_rng(seed)
    w = workloads._assemble("order", rng, "cuda", lens=lengths(S, seed), Hq=Hq, Hkv=Hkv, D=D,
                            B=B, dtype=dtype, std=0.5)
    if fp8:
        w = workloads.to_fp8(w)
        P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping,
                                   w.meta["k_scale"], w.meta["v_scale"])
    else:
        P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    return w


def decode(w, fp8, workspace=None, context_lens=None):
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    cl = w.context_lens if context_lens is None else context_lens
    if fp8:
        P.pa_decode_fp8(out, w.q, w.k_cache, w.v_cache, w.meta["k_scale"], w.meta["v_scale"],
                        w.block_tables, cl, w.scale, w.num_kv_heads, w.block_size,
                        max_context_len=w.max_context_len, partition_size=0,
                        workspace=workspace)
    else:
        P.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, cl, w.scale,
                    w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                    partition_size=0, workspace=workspace)
    torch.cuda.synchronize()
    return out


def reference(w, fp8):
    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    extra = {}
    if fp8:
        kc, vc = kc.view(torch.uint8), vc.view(torch.uint8)
        extra = dict(k_scale=w.meta["k_scale"].cpu(), v_scale=w.meta["v_scale"].cpu())
    return oracle.paged_attention(w.q.cpu(), kc, vc, w.block_tables.cpu(), w.context_lens.cpu(),
                                  w.scale, w.num_kv_heads, w.block_size,
                                  num_threads=oracle.max_threads(), **extra)


CASES = [
    # Hq, Hkv, D, B, dtype, E4M3 cache -- all on the CUDA-core decode kernel
    (32, 32, 128, 16, torch.bfloat16, False),   # one head per CTA
    (40, 40, 128, 32, torch.float16, False),
    (16, 8, 64, 16, torch.bfloat16, False),     # two heads per CTA
    (16, 16, 64, 16, torch.float32, False),
    (32, 32, 64, 16, torch.bfloat16, True),     # E4M3 codes converted on the CUDA cores
    (16, 8, 64, 32, torch.float16, True),
]


@pytest.mark.parametrize("Hq,Hkv,D,B,dtype,fp8", CASES)
def test_longest_first_is_bitwise_index_order(Hq, Hkv, D, B, dtype, fp8):
    S = 192
    w = make(S, Hq, Hkv, D, B, dtype, fp8, seed=Hq + Hkv + D + B + fp8)
    kv = w.k_cache.dtype
    assert P.pa_decode_orders_sequences(dtype, kv, S, Hq, Hkv, D, B, w.max_context_len, 0)
    ordered = decode(w, fp8)                                   # the binding's workspace
    assert P.pa_get_device_error() == 0
    plain = decode(w, fp8, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert P.pa_get_device_error() == 0
    assert torch.equal(ordered.view(torch.int32), plain.view(torch.int32))
    ref = reference(w, fp8)
    got = ordered.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= ATOL


@pytest.mark.parametrize("Hq,Hkv,D,B,dtype,fp8", [
    (32, 8, 128, 16, torch.bfloat16, False),    # mma.sync decode
    (32, 32, 128, 16, torch.bfloat16, True),    # E4M3 tcgen05 decode
    (32, 8, 64, 16, torch.bfloat16, True),      # E4M3 mma.sync decode
])
def test_tensor_core_decodes_keep_index_order(Hq, Hkv, D, B, dtype, fp8):
    kv = torch.float8_e4m3fn if fp8 else dtype
    assert not P.pa_decode_orders_sequences(dtype, kv, 192, Hq, Hkv, D, B, 2048, 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_invalid_length_in_an_ordered_call(fp8):
    """A context length above max_context_len is clamped into the longest class by the
    order and flagged by the decode, which writes NaN rows for that sequence only."""
    S = 160
    w = make(S, 32, 32, 64 if fp8 else 128, 16, torch.bfloat16, fp8, seed=77)
    assert P.pa_decode_orders_sequences(torch.bfloat16, w.k_cache.dtype, S, 32, 32,
                                        w.head_dim, 16, w.max_context_len, 0)
    cl = w.context_lens.clone()
    cl[5] = w.max_context_len + 7
    cl[90] = -3
    out = decode(w, fp8, context_lens=cl)
    assert P.pa_get_device_error() & 0x2
    assert torch.isnan(out[5]).all() and torch.isnan(out[90]).all()
    keep = torch.ones(S, dtype=torch.bool)
    keep[5] = keep[90] = False
    assert torch.isfinite(out[keep.cuda()]).all()
    ref = reference(w, fp8)
    err = np.abs(out.double().cpu().numpy()[keep.numpy()] - ref[keep.numpy()]).max()
    assert err <= ATOL


def test_many_sequences():
    """Several thousand sequences: each of the order kernel's threads owns a range of
    several sequences."""
    S = 5000
    rng = np.random.default_rng(5)
    lens = np.clip(np.exp(rng.normal(np.log(100), 0.9, size=S)), 1, 600).astype(int).tolist()
    w = workloads._assemble("order_many", rng, "cuda", lens=lens, Hq=8, Hkv=8, D=64, B=16,
                            dtype=torch.bfloat16, std=0.5)
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    assert P.pa_decode_orders_sequences(torch.bfloat16, torch.bfloat16, S, 8, 8, 64, 16,
                                        w.max_context_len, 0)
    ordered = decode(w, False)
    plain = decode(w, False, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert P.pa_get_device_error() == 0
    assert torch.equal(ordered.view(torch.int32), plain.view(torch.int32))
    got = ordered.double().cpu().numpy()
    rows = rng.choice(S, size=200, replace=False)
    ref = oracle.paged_attention(w.q.cpu()[rows], w.k_cache.cpu(), w.v_cache.cpu(),
                                 w.block_tables.cpu()[rows], w.context_lens.cpu()[rows], w.scale,
                                 w.num_kv_heads, w.block_size, num_threads=oracle.max_threads())
    assert np.abs(got[rows] - ref).max() <= ATOL
