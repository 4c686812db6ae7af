"""64-bit addressing on every attention kernel (GPU).

Each case builds pools of more than 2^31 elements per cache and puts the blocks the
sequences use at the very top, so every element offset the kernel forms exceeds 2^31;
the result must match the oracle run on just those blocks (tables relabelled to them).
The kernels covered: mma.sync GQA (bf16), tcgen05 E4M3 (multi-head), mma.sync E4M3 with
two blocks per tile (GQA 8, block 16), and the tcgen05 chunk kernel over bf16 and E4M3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ATOL = 2e-3
B, D = 16, 128


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


@pytest.fixture(autouse=True)
def clear_error_word(built):
    P.pa_get_device_error()
    yield
    torch.cuda.empty_cache()


def top_pool(Hkv, lens, fp8, seed):
    """Pools just past 2^31 elements per cache; sequence blocks at the top.  Returns the
    device pools, tables, lengths, and the compacted CPU pools and tables for the oracle."""
    N = 2 ** 31 // (Hkv * B * D) + 64
    assert N * Hkv * B * D > 2 ** 31
    need = [math.ceil(L / B) for L in lens]
    base = N - sum(need)
    g = torch.Generator(device="cuda").manual_seed(seed)
    dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
    kc = torch.empty(N, Hkv, B, D, dtype=dt, device="cuda")
    vc = torch.empty_like(kc)
    for c in (kc, vc):
        c[base:] = torch.randn(sum(need), Hkv, B, D, generator=g, device="cuda").to(dt)
    bt = torch.full((len(lens), max(need)), -1, dtype=torch.int32)
    nxt = base
    for s, n in enumerate(need):
        bt[s, :n] = torch.arange(nxt, nxt + n, dtype=torch.int32)
        nxt += n
    cl = torch.tensor(lens, dtype=torch.int32)
    small_k, small_v = kc[base:].cpu(), vc[base:].cpu()
    bt_local = torch.where(bt >= 0, bt - base, bt)
    return kc, vc, bt.cuda(), cl.cuda(), small_k, small_v, bt_local, cl


@pytest.mark.parametrize("Hq,Hkv,fp8,kernel", [
    (64, 8, False, "decode_mma_kernel"),
    (40, 40, True, "decode_tc8_kernel"),
    (64, 8, True, "decode_mma_kernel"),
])
def test_decode_beyond_2_pow_31_elements(Hq, Hkv, fp8, kernel):
    lens = [70, 33, 200]
    kc, vc, bt, cl, sk, sv, btl, clh = top_pool(Hkv, lens, fp8, Hq + Hkv)
    dt = kc.dtype
    assert P.pa_decode_kernel_name(dt, Hq, Hkv, D) == kernel
    q = torch.randn(len(lens), Hq, D, device="cuda").bfloat16()
    out = torch.empty(len(lens), Hq, D, device="cuda")
    scale = 1 / math.sqrt(D)
    if fp8:
        ks = torch.ones(Hkv, device="cuda")
        vs = torch.full((Hkv,), 0.5, device="cuda")
        P.pa_decode_fp8(out, q, kc, vc, ks, vs, bt, cl, scale, Hkv, B, max_context_len=max(lens))
        ref = oracle.paged_attention(q.cpu(), sk.view(torch.uint8), sv.view(torch.uint8), btl, clh,
                                     scale, Hkv, B, k_scale=ks.cpu(), v_scale=vs.cpu())
    else:
        P.pa_decode(out, q, kc, vc, bt, cl, scale, Hkv, B, max_context_len=max(lens))
        ref = oracle.paged_attention(q.cpu(), sk, sv, btl, clh, scale, Hkv, B)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() == 0
    assert np.abs(out.double().cpu().numpy() - ref).max() <= ATOL


@pytest.mark.parametrize("fp8", [False, True])
def test_chunk_beyond_2_pow_31_elements(fp8):
    Hq, Hkv = 64, 8
    lens, chunks = [300, 120], [40, 33]
    kc, vc, bt, cl, sk, sv, btl, clh = top_pool(Hkv, lens, fp8, 77 + fp8)
    qs = torch.tensor([0, chunks[0], chunks[0] + chunks[1]], dtype=torch.int32)
    assert P.pa_chunk_kernel_name(kc.dtype, Hq, Hkv, D, max(chunks)).startswith("chunk_attn_kernel")
    q = torch.randn(sum(chunks), Hq, D, device="cuda").bfloat16()
    out = torch.empty(sum(chunks), Hq, D, device="cuda")
    scale = 1 / math.sqrt(D)
    kw = dict(max_query_len=max(chunks), max_context_len=max(lens))
    if fp8:
        ks = torch.ones(Hkv, device="cuda")
        vs = torch.full((Hkv,), 0.5, device="cuda")
        P.pa_chunk_attention_fp8(out, q, kc, vc, ks, vs, bt, cl, qs.cuda(), scale, Hkv, B, **kw)
        ref = oracle.chunk_attention(q.cpu(), sk.view(torch.uint8), sv.view(torch.uint8), btl, clh,
                                     qs, scale, Hkv, B, k_scale=ks.cpu(), v_scale=vs.cpu())
    else:
        P.pa_chunk_attention(out, q, kc, vc, bt, cl, qs.cuda(), scale, Hkv, B, **kw)
        ref = oracle.chunk_attention(q.cpu(), sk, sv, btl, clh, qs, scale, Hkv, B)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() == 0
    assert np.abs(out.double().cpu().numpy() - ref).max() <= ATOL
