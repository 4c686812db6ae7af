"""End to end on the GPU: the C++ block manager drives copy_blocks, reshape_and_cache and
decode through prefill, fork (parallel sampling), decode steps with copy-on-write, and
frees.  Each step is checked against the reference model + CPU oracle (same slots, same
copy pairs, bit-identical caches, attention within tolerance); at the end every live
sequence's attention is checked against dense attention over its own token history."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_119_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


def bits(t):
    return t.view({4: torch.int32, 2: torch.int16}[t.element_size()])


@pytest.mark.parametrize("Hq,Hkv,B", [(8, 8, 16), (16, 4, 16), (16, 2, 32)])
def test_parallel_sampling_with_copy_on_write(Hq, Hkv, B):
    D, dtype, N = 128, torch.bfloat16, 160
    gen = torch.Generator().manual_seed(Hq * 10 + Hkv + B)
    rng = np.random.default_rng(Hq + Hkv + B)
    order = rng.permutation(N)
    mgr, ref = BlockManager(N, B, order), BlockManagerModel(N, B, order)
    kc = torch.full((N, Hkv, B, D), float("nan"), dtype=dtype, device="cuda")
    vc = kc.clone()
    kc_h, vc_h = kc.cpu(), vc.cpu()
    history = {}                                    # seq -> (K rows, V rows) as [L, Hkv, D]

    def write(seqs_slots, k, v):
        slots = torch.tensor(seqs_slots, dtype=torch.int64)
        P.pa_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, slots.cuda())
        oracle.reshape_and_cache(k, v, kc_h, vc_h, slots, B)

    # prefill three prompts of ragged lengths, then fork each into 4 samples
    live = []
    for p, L in enumerate((37, 50, 16)):
        s = 100 * p
        slots = mgr.add_sequence(s, L)
        assert list(slots) == ref.add_sequence(s, L)
        k = torch.randn(L, Hkv, D, generator=gen).to(dtype)
        v = torch.randn(L, Hkv, D, generator=gen).to(dtype)
        write(list(slots), k, v)
        history[s] = (k, v)
        live.append(s)
        for j in range(1, 4):
            mgr.fork(s, s + j)
            ref.fork(s, s + j)
            history[s + j] = (k.clone(), v.clone())
            live.append(s + j)

    saw_copy = False
    for step in range(24):
        if step == 11:                               # drop one sample of each prompt
            for s in (3, 103, 203):
                mgr.free(s)
                ref.free_sequence(s)
                live.remove(s)
        slots, pairs = mgr.append(live)
        rslots, rpairs = ref.append(live)
        assert list(slots) == rslots and [tuple(x) for x in pairs] == rpairs
        if len(pairs):
            saw_copy = True
            P.pa_copy_blocks([kc], [vc], pairs)
            oracle.copy_blocks([kc_h, vc_h], pairs)
        k = torch.randn(len(live), Hkv, D, generator=gen).to(dtype)
        v = torch.randn(len(live), Hkv, D, generator=gen).to(dtype)
        write(list(slots), k, v)
        for i, s in enumerate(live):
            hk, hv = history[s]
            history[s] = (torch.cat([hk, k[i:i + 1]]), torch.cat([hv, v[i:i + 1]]))
        # decode the whole batch
        W = 8
        table, lens = mgr.block_tables(live, W)
        rtable = np.full((len(live), W), -1, dtype=np.int32)
        for i, s in enumerate(live):
            rtable[i, :len(ref.tables[s])] = ref.tables[s]
        assert np.array_equal(table, rtable)
        q = torch.randn(len(live), Hq, D, generator=gen).to(dtype)
        out = torch.empty(len(live), Hq, D, device="cuda")
        P.pa_decode(out, q.cuda(), kc, vc, torch.from_numpy(table).cuda(),
                    torch.from_numpy(lens).cuda(), D ** -0.5, Hkv, B)
        torch.cuda.synchronize()
        want = oracle.paged_attention(q, kc_h, vc_h, torch.from_numpy(table),
                                      torch.from_numpy(lens), D ** -0.5, Hkv, B)
        assert np.abs(out.double().cpu().numpy() - want).max() <= ATOL
        assert torch.equal(bits(kc.cpu()), bits(kc_h)) and torch.equal(bits(vc.cpu()), bits(vc_h))
    assert saw_copy, "the scenario never exercised copy-on-write"
    assert P.pa_get_device_error() == 0

    # every sequence still sees exactly its own history
    table, lens = mgr.block_tables(live, 8)
    q = torch.randn(len(live), Hq, D, generator=gen).to(dtype)
    out = torch.empty(len(live), Hq, D, device="cuda")
    P.pa_decode(out, q.cuda(), kc, vc, torch.from_numpy(table).cuda(),
                torch.from_numpy(lens).cuda(), D ** -0.5, Hkv, B)
    torch.cuda.synchronize()
    for i, s in enumerate(live):
        hk, hv = history[s]
        assert lens[i] == hk.shape[0]
        dense = oracle.paged_attention(q[i:i + 1], hk.view(-1, 1, Hkv, D).transpose(1, 2).contiguous(),
                                       hv.view(-1, 1, Hkv, D).transpose(1, 2).contiguous(),
                                       torch.arange(hk.shape[0], dtype=torch.int32).view(1, -1),
                                       torch.tensor([hk.shape[0]], dtype=torch.int32),
                                       D ** -0.5, Hkv, 1)
        assert np.abs(out[i].double().cpu().numpy() - dense[0]).max() <= ATOL
