"""Swapping KV blocks between the GPU pool and a pinned CPU pool (pa_swap_blocks) on
the GPU: bit-exact against the oracle's byte moves, and a swapped-out, swapped-in
sequence decodes exactly as before under its new block table."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


def raw(t):
    return t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16)


def test_swap_out_and_in_bit_exact_and_decode_unchanged():
    w = workloads.make("llama13b", device="cuda", num_seqs=24)
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out0 = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_decode(out0, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                w.num_kv_heads, w.block_size, max_context_len=w.max_context_len)
    victims = [3, 10, 17]
    bt = w.block_tables.cpu()
    nblk = [(int(w.context_lens[s]) + w.block_size - 1) // w.block_size for s in victims]
    gpu_blocks = [int(b) for s, n in zip(victims, nblk) for b in bt[s, :n]]
    # swap out: GPU blocks -> CPU pool slots 0 .. n-1 (all-or-nothing per sequence)
    shape = (len(gpu_blocks) + 5,) + tuple(w.k_cache.shape[1:])
    cpu_k = torch.zeros(shape, dtype=w.dtype).pin_memory()
    cpu_v = torch.zeros(shape, dtype=w.dtype).pin_memory()
    out_pairs = [(b, i) for i, b in enumerate(gpu_blocks)]
    ref_k, ref_v = cpu_k.clone(), cpu_v.clone()
    oracle.swap_blocks([w.k_cache.cpu(), w.v_cache.cpu()], [ref_k, ref_v], out_pairs)
    P.pa_swap_blocks([w.k_cache, w.v_cache], [cpu_k, cpu_v], out_pairs)
    torch.cuda.synchronize()
    assert torch.equal(raw(cpu_k), raw(ref_k)) and torch.equal(raw(cpu_v), raw(ref_v))
    # the freed GPU blocks are reused by someone else
    w.k_cache[gpu_blocks] = float("nan")
    w.v_cache[gpu_blocks] = float("nan")
    # swap in: into other GPU blocks -- a shuffle of the pool's free blocks and the
    # victims' own freed ones, so most land somewhere new
    used = set(int(b) for b in bt[bt >= 0]) - set(gpu_blocks)
    candidates = [b for b in range(w.num_blocks) if b not in used]
    free = [int(x) for x in np.random.default_rng(4).permutation(candidates)[:len(gpu_blocks)]]
    assert len(free) == len(gpu_blocks)
    assert sum(a != b for a, b in zip(free, gpu_blocks)) > len(gpu_blocks) // 2
    in_pairs = [(i, b) for i, b in enumerate(free)]
    want_k, want_v = w.k_cache.cpu(), w.v_cache.cpu()
    oracle.swap_blocks([cpu_k, cpu_v], [want_k, want_v], in_pairs)
    P.pa_swap_blocks([cpu_k, cpu_v], [w.k_cache, w.v_cache], in_pairs)
    torch.cuda.synchronize()
    assert torch.equal(raw(w.k_cache.cpu()), raw(want_k))
    assert torch.equal(raw(w.v_cache.cpu()), raw(want_v))
    # the sequences' tables now name the new blocks; attention is bit-identical
    bt2 = bt.clone()
    it = iter(free)
    for s, n in zip(victims, nblk):
        for j in range(n):
            bt2[s, j] = next(it)
    out1 = torch.empty_like(out0)
    P.pa_decode(out1, w.q, w.k_cache, w.v_cache, bt2.cuda(), w.context_lens, w.scale,
                w.num_kv_heads, w.block_size, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out0, out1)
    assert P.pa_get_device_error() == 0


def test_swap_many_layers_and_pairs_chunked_launches():
    """80 caches (40 layers x K, V) and 1500 pairs: more than one launch's worth of
    both; every byte matches the oracle."""
    g = torch.Generator(device="cuda").manual_seed(5)
    L, N, M, shape = 80, 1600, 1700, (2, 16, 64)
    gpu = [torch.randn((N,) + shape, generator=g, device="cuda").to(torch.float16)
           for _ in range(L)]
    cpu = [torch.zeros((M,) + shape, dtype=torch.float16).pin_memory() for _ in range(L)]
    rng = np.random.default_rng(3)
    src = rng.choice(N, size=1500, replace=False)
    dst = rng.choice(M, size=1500, replace=False)
    pairs = np.stack([src, dst], 1)
    want = [c.clone() for c in cpu]
    oracle.swap_blocks([t.cpu() for t in gpu], want, pairs)
    P.pa_swap_blocks(gpu, cpu, pairs)
    torch.cuda.synchronize()
    for a, b in zip(cpu, want):
        assert torch.equal(raw(a), raw(b))


def test_swap_fp8_pools_and_device_to_device():
    """Byte pools of any element type; both pools on the device also works."""
    g = torch.Generator(device="cuda").manual_seed(9)
    a = torch.randint(0, 256, (40, 8, 16, 128), generator=g, device="cuda",
                      dtype=torch.uint8).view(torch.float8_e4m3fn)
    b = torch.zeros((30, 8, 16, 128), dtype=torch.uint8).pin_memory().view(torch.float8_e4m3fn)
    c = torch.zeros((25, 8, 16, 128), device="cuda", dtype=torch.uint8)
    pairs = [(39, 0), (0, 29), (17, 3)]
    P.pa_swap_blocks(a, b, pairs)
    P.pa_swap_blocks(b, c, [(0, 24), (29, 0), (3, 1)])
    torch.cuda.synchronize()
    av = a.view(torch.uint8).cpu()
    assert torch.equal(b.view(torch.uint8)[0], av[39])
    assert torch.equal(b.view(torch.uint8)[29], av[0])
    assert torch.equal(c.cpu()[24], av[39]) and torch.equal(c.cpu()[0], av[0])
    assert torch.equal(c.cpu()[1], av[17])
    assert int(c.cpu()[2:24].sum()) == 0


def test_swap_refuses_pageable_host_memory():
    gpu = torch.zeros((4, 64), device="cuda", dtype=torch.float16)
    host = torch.zeros((4, 64), dtype=torch.float16)          # not pinned
    with pytest.raises(ValueError):
        P.pa_swap_blocks(gpu, host, [(0, 1)])


def test_block_manager_drives_swap_out_and_in():
    """The host manager preempts a forked group (its pairs drive pa_swap_blocks into
    pinned CPU pools), another sequence reuses the freed GPU blocks, the group returns
    into new GPU blocks and decodes bit-identically."""
    from paged_kv_cache_119_gb300.block_manager import BlockManager
    Hq, Hkv, D, B, N = 16, 4, 128, 16, 64
    g = torch.Generator(device="cuda").manual_seed(11)
    m = BlockManager(N, B)
    m.set_cpu_pool(N)
    kc = torch.full((N, Hkv, B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))

    def write(slots):
        k = torch.randn(len(slots), Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn(len(slots), Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
        P.pa_reshape_and_cache(k, v, kc, vc, torch.as_tensor(slots, device="cuda"))

    write(m.add_sequence(0, 70))
    for c in (1, 2):
        m.fork(0, c)
    for _ in range(20):
        slots, pairs = m.append([0, 1, 2])
        if len(pairs):
            P.pa_copy_blocks([kc], [vc], pairs)
        write(slots)
    group = [0, 1, 2]
    q = torch.randn(3, Hq, D, generator=g, device="cuda").to(torch.bfloat16)

    def decode(tables, lens):
        out = torch.empty(3, Hq, D, dtype=torch.float32, device="cuda")
        P.pa_decode(out, q, kc, vc, torch.as_tensor(tables, device="cuda"),
                    torch.as_tensor(lens, device="cuda"), 0.1, Hkv, B)
        return out

    t0, l0 = m.block_tables(group, 16)
    out0 = decode(t0, l0)
    cpu_k = torch.zeros((N,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    cpu_v = torch.zeros_like(cpu_k).pin_memory()
    P.pa_swap_blocks([kc, vc], [cpu_k, cpu_v], m.swap_out(group))
    # another sequence takes every free GPU block and overwrites it
    other = m.num_free_blocks() * B
    write(m.add_sequence(50, other))
    m.free(50)
    P.pa_swap_blocks([cpu_k, cpu_v], [kc, vc], m.swap_in(group))
    t1, l1 = m.block_tables(group, 16)
    assert (l1 == l0).all() and not (t1 == t0).all()
    out1 = decode(t1, l1)
    torch.cuda.synchronize()
    assert torch.equal(out0, out1)
    ref = oracle.paged_attention(q.cpu(), kc.cpu(), vc.cpu(), torch.as_tensor(t1),
                                 torch.as_tensor(l1), 0.1, Hkv, B)
    assert np.abs(out1.double().cpu().numpy() - ref).max() <= 2e-3
    assert P.pa_get_device_error() == 0


def test_swap_full_size_benchmark_step():
    """The benchmark's swap step at full size: every block of the last 64 of 256
    LLaMA-13B-shaped sequences, K and V, out to a pinned CPU pool in one launch and back
    in one launch; every byte against the oracle's moves, and the pool unchanged after
    the round trip."""
    import bench
    w = workloads.make("llama13b", device="cuda")
    blocks, bb = bench.swap_plan(w, 64)
    n = len(blocks)
    cpu_k = torch.full((n,) + tuple(w.k_cache.shape[1:]), 7.0, dtype=w.dtype).pin_memory()
    cpu_v = torch.full_like(cpu_k, 7.0).pin_memory()
    out_pairs = torch.tensor([(b, i) for i, b in enumerate(blocks)], dtype=torch.int64)
    before_k, before_v = w.k_cache.cpu(), w.v_cache.cpu()
    want_k, want_v = cpu_k.clone(), cpu_v.clone()
    oracle.swap_blocks([before_k, before_v], [want_k, want_v], out_pairs.numpy())
    P.pa_swap_blocks([w.k_cache, w.v_cache], [cpu_k, cpu_v], out_pairs)
    torch.cuda.synchronize()
    assert torch.equal(raw(cpu_k), raw(want_k)) and torch.equal(raw(cpu_v), raw(want_v))
    w.k_cache[blocks] = float("nan")              # the GPU blocks are reused meanwhile
    w.v_cache[blocks] = float("nan")
    P.pa_swap_blocks([cpu_k, cpu_v], [w.k_cache, w.v_cache], out_pairs.flip(1).contiguous())
    torch.cuda.synchronize()
    assert torch.equal(raw(w.k_cache.cpu()), raw(before_k))
    assert torch.equal(raw(w.v_cache.cpu()), raw(before_v))
    assert P.pa_get_device_error() == 0
