"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Cache writes and block copies must match bit for bit (whole pools compared as
raw bytes, NaN fill included).  Attention written as fp32 must be within
2e-3 max abs error of the fp64 oracle; written in the cache dtype it must be
the round-to-nearest-even of a value within 5e-5 of the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL = 2e-3          # max abs error on fp32 output (fp16/bf16 inputs, fp32 accumulation)

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


@pytest.fixture(autouse=True)
def clear_error_word(built):
    P.pa_get_device_error()          # every test starts from a clear error word
    yield


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.view({4: torch.int32, 2: torch.int16}[t.element_size()])


def snapshot(w):
    """Host copies of the step's inputs, taken before the GPU mutates the caches."""
    return dict(k_cache=w.k_cache.cpu(), v_cache=w.v_cache.cpu(), q=w.q.cpu(),
                k_new=w.k_new.cpu(), v_new=w.v_new.cpu(), slot_mapping=w.slot_mapping.cpu(),
                block_tables=w.block_tables.cpu(), context_lens=w.context_lens.cpu())


def gpu_step(w, out_dtype=torch.float32, partition_size=None):
    if w.copy_pairs is not None:
        P.pa_copy_blocks([w.k_cache], [w.v_cache], w.copy_pairs)
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = torch.empty(w.num_seqs, w.num_q_heads, w.head_dim, dtype=out_dtype, device="cuda")
    P.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                partition_size=w.partition_size if partition_size is None else partition_size)
    torch.cuda.synchronize()
    return out


def oracle_step(w, snap):
    kc, vc = snap["k_cache"].clone(), snap["v_cache"].clone()
    if w.copy_pairs is not None:
        oracle.copy_blocks([kc, vc], w.copy_pairs)
    oracle.reshape_and_cache(snap["k_new"], snap["v_new"], kc, vc, snap["slot_mapping"],
                             w.block_size)
    out = oracle.paged_attention(snap["q"], kc, vc, snap["block_tables"], snap["context_lens"],
                                 w.scale, w.num_kv_heads, w.block_size,
                                 num_threads=oracle.max_threads())
    return out, kc, vc


NATIVE_EPS = 5e-5    # native-dtype output: the rounding of a value within this of the oracle


def check_attention(out_gpu, ref, dtype):
    """fp32 output: max abs error <= ATOL.  Native fp16/bf16 output: each value is the
    round-to-nearest-even of some y with |y - ref| <= NATIVE_EPS; rounding is monotone,
    so that is RNE(ref - eps) <= out <= RNE(ref + eps) elementwise."""
    got = out_gpu.double().cpu().numpy()
    assert np.isfinite(got).all(), "non-finite output"
    if out_gpu.dtype == torch.float32:
        err = np.abs(got - ref).max()
        assert err <= ATOL, f"max abs error {err:.3e} > {ATOL}"
        return err
    lo = torch.from_numpy((ref - NATIVE_EPS).astype(np.float32)).to(out_gpu.dtype).double().numpy()
    hi = torch.from_numpy((ref + NATIVE_EPS).astype(np.float32)).to(out_gpu.dtype).double().numpy()
    bad = (got < lo) | (got > hi)
    assert not bad.any(), (f"{int(bad.sum())} values are not a rounding of the oracle "
                           f"within {NATIVE_EPS}: e.g. got {got[bad][:4]}, ref {ref[bad][:4]}")
    return np.abs(got - ref).max()


def run_and_compare(w, out_dtype=torch.float32, partition_size=None):
    snap = snapshot(w)
    out = gpu_step(w, out_dtype, partition_size)
    ref, kc, vc = oracle_step(w, snap)
    assert torch.equal(bits(w.k_cache.cpu()), bits(kc)), "k_cache differs from the oracle"
    assert torch.equal(bits(w.v_cache.cpu()), bits(vc)), "v_cache differs from the oracle"
    err = check_attention(out, ref, w.dtype)
    assert P.pa_get_device_error() == 0
    return out, ref, err


# ------------------------------------------------------------------ the five configs, scaled

SMALL = {
    "tiny": dict(),
    "opt13b": dict(num_seqs=6, max_len=700),
    "llama13b": dict(num_seqs=12),
    "prefix": dict(num_groups=2, group_size=4, prefix_blocks=8, max_suffix=60),
    "long16": dict(num_seqs=2, context=3000),
    "long32": dict(num_seqs=2, context=3000),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("out_kind", ["f32", "native"])
def test_config_small(name, out_kind):
    w = workloads.make(name, device="cuda", **SMALL[name])
    run_and_compare(w, torch.float32 if out_kind == "f32" else w.dtype)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_tiny_half_types(dtype):
    w = workloads.make("tiny", device="cuda", dtype=dtype)
    run_and_compare(w)


@pytest.mark.parametrize("part", [-1, 0, 16, 32, 512])
def test_split_and_unsplit_agree(part):
    """Every partitioning gives the oracle's result (ragged last partition included)."""
    w = workloads.make("llama13b", device="cuda", num_seqs=10)
    run_and_compare(w, partition_size=part)


# ------------------------------------------------------------------ full sizes

FULL = ["opt13b", "llama13b", "prefix", "long16", "long32"]


@pytest.mark.parametrize("name", FULL)
@pytest.mark.parametrize("part", ["config", "auto"])
def test_config_full_size(name, part):
    """The full workload: with the config's partition size (512 tokens for the long
    contexts) and with the automatic split the benchmark times."""
    w = workloads.make(name, device="cuda")
    run_and_compare(w, partition_size=None if part == "config" else 0)


# ------------------------------------------------------------------ invariants

def test_block_relabelling_is_bitwise_invariant():
    w = workloads.make("llama13b", device="cuda", num_seqs=8)
    out1 = gpu_step(w)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(3)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_blocks, device="cuda")
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache                 # block b moves to perm[b]
    v2[perm] = w.v_cache
    bt2 = torch.where(w.block_tables >= 0, perm[w.block_tables.long().clamp(min=0)].int(),
                      w.block_tables)
    out2 = torch.empty_like(out1)
    P.pa_decode(out2, w.q, k2, v2, bt2, w.context_lens, w.scale, w.num_kv_heads, w.block_size,
                max_context_len=w.max_context_len)
    assert torch.equal(bits(out1), bits(out2))


def test_shared_prefix_equals_private_copies_bitwise():
    w = workloads.make("prefix", device="cuda", num_groups=2, group_size=4, prefix_blocks=6,
                       max_suffix=40)
    out_shared = gpu_step(w)
    # give every sequence private copies of all its blocks and decode again
    S, W = w.block_tables.shape
    n_used = int((w.block_tables >= 0).sum())
    k2 = torch.full((n_used + 1,) + tuple(w.k_cache.shape[1:]), float("nan"), dtype=w.dtype,
                    device="cuda")
    v2 = k2.clone()
    bt2 = torch.full_like(w.block_tables, -1)
    nxt = 0
    for s in range(S):
        for j in range(W):
            b = int(w.block_tables[s, j])
            if b < 0:
                continue
            k2[nxt] = w.k_cache[b]
            v2[nxt] = w.v_cache[b]
            bt2[s, j] = nxt
            nxt += 1
    out_priv = torch.empty_like(out_shared)
    P.pa_decode(out_priv, w.q, k2, v2, bt2, w.context_lens, w.scale, w.num_kv_heads,
                w.block_size, max_context_len=w.max_context_len)
    assert torch.equal(bits(out_shared), bits(out_priv))


def test_single_token_context_returns_v0_exactly():
    w = workloads.make("tiny", device="cuda", lens=[1, 1, 1, 1], dtype=torch.bfloat16)
    out = gpu_step(w)
    hk = torch.arange(w.num_q_heads, device="cuda") // (w.num_q_heads // w.num_kv_heads)
    assert torch.equal(out, w.v_new[:, hk, :].float())


def test_empty_context_gives_zeros():
    w = workloads.make("tiny", device="cuda", lens=[0, 5, 0, 17], dtype=torch.float16)
    out = gpu_step(w)
    assert torch.equal(out[0], torch.zeros_like(out[0])) and torch.equal(out[2], out[0])
    snap_ok = torch.isfinite(out[[1, 3]]).all()
    assert snap_ok


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (12, 4), (24, 4), (64, 8)])
@pytest.mark.parametrize("D,B", [(64, 16), (128, 32)])
def test_head_groupings(Hq, Hkv, D, B):
    """MHA and GQA with groups 1..8, a non-power-of-two group, head_dim 64/128, B 16/32."""
    rng = np.random.default_rng(Hq * 100 + Hkv + D + B)
    lens = [int(x) for x in rng.integers(1, 300, size=5)]
    w = workloads._assemble("groups", rng, "cuda", lens=lens, Hq=Hq, Hkv=Hkv, D=D, B=B,
                            dtype=torch.bfloat16, std=1.0)
    run_and_compare(w)


def test_many_layers_and_pairs_copy_in_chunks():
    """copy_blocks over more layers and pairs than one launch carries."""
    torch.manual_seed(0)
    layers, n, pairs = 11, 1600, 700
    kc = [torch.randn(n, 2, 16, 64, device="cuda", dtype=torch.float16) for _ in range(layers)]
    vc = [torch.randn(n, 2, 16, 64, device="cuda", dtype=torch.float16) for _ in range(layers)]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(1))
    pr = torch.stack([perm[:pairs], perm[pairs:2 * pairs]], 1)
    host = [t.cpu() for t in kc + vc]
    P.pa_copy_blocks(kc, vc, pr)
    oracle.copy_blocks(host, pr.numpy())
    for a, b in zip(kc + vc, host):
        assert torch.equal(bits(a.cpu()), bits(b))


def test_reshape_skips_negative_slots_and_keeps_bytes():
    w = workloads.make("tiny", device="cuda", dtype=torch.bfloat16)
    w.slot_mapping[1] = -1
    k_before = w.k_cache.cpu()
    snap = snapshot(w)
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    kc, vc = snap["k_cache"].clone(), snap["v_cache"].clone()
    oracle.reshape_and_cache(snap["k_new"], snap["v_new"], kc, vc, snap["slot_mapping"], 16)
    assert torch.equal(bits(w.k_cache.cpu()), bits(kc))
    assert torch.equal(bits(w.v_cache.cpu()), bits(vc))
    assert not torch.equal(bits(k_before), bits(kc))


# ------------------------------------------------------------------ guards and device checks

def test_canaries_around_output_and_pool_survive():
    w = workloads.make("llama13b", device="cuda", num_seqs=6)
    S, Hq, D = w.q.shape
    pad = 4096
    big = torch.full((pad + S * Hq * D + pad,), 12345.0, device="cuda")
    out = big[pad:pad + S * Hq * D].view(S, Hq, D)
    kbig = torch.full((w.k_cache.numel() + 2 * pad,), 3.0, device="cuda",
                      dtype=w.dtype)
    kbig[pad:pad + w.k_cache.numel()] = w.k_cache.flatten()
    k_in = kbig[pad:pad + w.k_cache.numel()].view_as(w.k_cache)
    P.pa_reshape_and_cache(w.k_new, w.v_new, k_in, w.v_cache, w.slot_mapping)
    P.pa_decode(out, w.q, k_in, w.v_cache, w.block_tables, w.context_lens, w.scale,
                w.num_kv_heads, w.block_size, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert (big[:pad] == 12345.0).all() and (big[-pad:] == 12345.0).all()
    assert (kbig[:pad] == 3.0).all() and (kbig[-pad:] == 3.0).all()
    assert torch.isfinite(out).all()


def test_bad_block_id_is_flagged_not_faulted():
    w = workloads.make("tiny", device="cuda")
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    w.block_tables[3, 1] = w.num_blocks + 5          # outside the pool
    out = torch.empty(4, 2, 64, device="cuda")
    P.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, 2, 16,
                max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() & 1
    assert torch.isnan(out[3]).all() and torch.isfinite(out[:3]).all()
    assert P.pa_get_device_error() == 0             # reading clears the word


def test_context_longer_than_max_is_flagged():
    w = workloads.make("tiny", device="cuda")
    out = torch.empty(4, 2, 64, device="cuda")
    P.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, 2, 16,
                max_context_len=20)                  # sequence 3 has 37 tokens
    torch.cuda.synchronize()
    assert P.pa_get_device_error() & 2
    assert torch.isnan(out[3]).all()


def test_slot_outside_pool_is_flagged_and_skipped():
    w = workloads.make("tiny", device="cuda")
    before = w.k_cache.cpu()
    w.slot_mapping[:] = w.num_blocks * 16 + 3
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() & 4
    assert torch.equal(bits(w.k_cache.cpu()), bits(before))


def test_int64_addressing_beyond_2_pow_31_elements():
    """A pool with more than 2^31 elements per cache; the used blocks sit at the top."""
    Hkv, B, D, S = 40, 16, 128, 2
    N = 26400                                       # 26400 * 40 * 16 * 128 > 2^31
    assert N * Hkv * B * D > 2 ** 31
    lens = [70, 33]
    need = [math.ceil(L / B) for L in lens]
    ids = list(range(N - sum(need), N))
    tables = [ids[:need[0]], ids[need[0]:]]
    g = torch.Generator(device="cuda").manual_seed(5)
    kc = torch.empty(N, Hkv, B, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    top = slice(N - sum(need), N)
    kc[top] = torch.randn(sum(need), Hkv, B, D, generator=g, device="cuda").bfloat16()
    vc[top] = torch.randn(sum(need), Hkv, B, D, generator=g, device="cuda").bfloat16()
    q = torch.randn(S, Hkv, D, generator=g, device="cuda").bfloat16()
    bt = torch.full((S, 8), -1, dtype=torch.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = torch.tensor(t, dtype=torch.int32)
    cl = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty(S, Hkv, D, device="cuda")
    P.pa_decode(out, q, kc, vc, bt.cuda(), cl.cuda(), 1 / math.sqrt(D), Hkv, B,
                max_context_len=max(lens))
    kt, vt = kc[top].cpu(), vc[top].cpu()
    base = N - sum(need)
    small_k = torch.zeros(sum(need), Hkv, B, D, dtype=torch.bfloat16)
    small_k[:] = kt
    bt_local = torch.where(bt >= 0, bt - base, bt)
    ref = oracle.paged_attention(q.cpu(), small_k, vt, bt_local, cl, 1 / math.sqrt(D), Hkv, B)
    assert np.abs(out.double().cpu().numpy() - ref).max() <= ATOL
    del kc, vc
    torch.cuda.empty_cache()
