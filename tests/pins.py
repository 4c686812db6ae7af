"""Pins for the CPU oracle: facts that hold independently of the oracle's code.

Every ``pin_*`` function takes the loaded oracle library and raises
AssertionError when the oracle disagrees with:
  * a worked example printed by the pages (tests/golden/*.json, each citing
    its page and figure / section),
  * a hand-computed closed form,
  * PyTorch's float64 ``scaled_dot_product_attention`` on the unpaged arrays
    (a library routine, independent of the oracle's gather),
  * IEEE decoding of every fp16 / bf16 bit pattern by PyTorch,
  * invariants the pages state (paging changes storage, not the result).

``tests/test_oracle_pins.py`` runs them against the real oracle and
``tests/test_oracle_mutants.py`` runs them against copies of the oracle with
one planted mistake each, checking that some pin fails for every mistake.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# ----------------------------------------------------------------------------- helpers

def dense_reference(q, K, V, scale):
    """Unpaged attention by PyTorch (float64).  q [Hq, D]; K, V [L, Hkv, D]."""
    q64 = q.double()[None, :, None, :]                       # [1, Hq, 1, D]
    k64 = K.double().permute(1, 0, 2)[None]                  # [1, Hkv, L, D]
    v64 = V.double().permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(q64, k64, v64, scale=scale,
                                       enable_gqa=q.shape[0] != K.shape[1])
    return o[0, :, 0, :].numpy()                             # [Hq, D]


def scatter_dense(K_list, V_list, tables, num_blocks, B, dtype, fill=float("nan")):
    """Write each sequence's dense [L, Hkv, D] rows into a pool through its table."""
    Hkv, D = K_list[0].shape[1], K_list[0].shape[2]
    kc = torch.full((num_blocks, Hkv, B, D), fill, dtype=dtype)
    vc = torch.full((num_blocks, Hkv, B, D), fill, dtype=dtype)
    for K, V, tab in zip(K_list, V_list, tables):
        for t in range(K.shape[0]):
            kc[tab[t // B], :, t % B, :] = K[t]
            vc[tab[t // B], :, t % B, :] = V[t]
    return kc, vc


def table_tensor(tables, width=None):
    W = width or max(1, max(len(t) for t in tables))
    bt = torch.full((len(tables), W), -1, dtype=torch.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = torch.tensor(t, dtype=torch.int32)
    return bt


def random_case(rng, S, Hq, Hkv, D, B, dtype, max_len, extra_blocks=3):
    """Dense K/V per sequence plus a randomly permuted pool holding them."""
    lens = [int(x) for x in rng.integers(1, max_len + 1, size=S)]
    need = [math.ceil(L / B) for L in lens]
    N = sum(need) + extra_blocks
    perm = rng.permutation(N)
    tables, pos = [], 0
    for n in need:
        tables.append([int(x) for x in perm[pos:pos + n]])
        pos += n
    g = torch.Generator().manual_seed(int(rng.integers(0, 2**31)))
    K = [torch.randn(L, Hkv, D, generator=g).to(dtype) for L in lens]
    V = [torch.randn(L, Hkv, D, generator=g).to(dtype) for L in lens]
    q = torch.randn(S, Hq, D, generator=g).to(dtype)
    kc, vc = scatter_dense(K, V, tables, N, B, dtype)
    return dict(lens=lens, tables=tables, N=N, K=K, V=V, q=q, kc=kc, vc=vc)


def run_oracle(lib, q, kc, vc, tables, lens, scale, Hkv, B, width=None):
    return oracle.paged_attention(q, kc, vc, table_tensor(tables, width),
                                  torch.tensor(lens, dtype=torch.int32), scale, Hkv, B, lib=lib)


def selector_case(B, n_blocks, table, D=4, H=1):
    """A pool whose V rows name their own (block, offset), for exact mapping checks."""
    kc = torch.zeros(n_blocks, H, B, D, dtype=torch.float64).float()
    vc = torch.zeros(n_blocks, H, B, D).float()
    for b in range(n_blocks):
        for o in range(B):
            vc[b, :, o, 0] = b
            vc[b, :, o, 1] = o
            vc[b, :, o, 2] = 1.0
    return kc, vc


# ----------------------------------------------------------------------------- pins

def pin_f16_decoder(lib):
    """Every binary16 bit pattern decodes as PyTorch decodes it."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.float16).double().numpy()
    got = np.array([lib.orc_f16_to_f64(i) for i in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def pin_bf16_decoder(lib):
    """Every bfloat16 bit pattern decodes as PyTorch decodes it."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()
    got = np.array([lib.orc_bf16_to_f64(i) for i in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def pin_hand_3token(lib):
    """The hand-computed 1-head, 3-token case (tests/golden/hand_3token.json)."""
    g = golden("hand_3token.json")
    B, D, N = g["block_size"], g["head_dim"], g["num_blocks"]
    kc = torch.full((N, 1, B, D), float("nan"), dtype=torch.float64).float()
    vc = kc.clone()
    for (blk, off), k, v in zip(g["placement"], g["k"], g["v"]):
        kc[blk, 0, off] = torch.tensor(k)
        vc[blk, 0, off] = torch.tensor(v)
    q = torch.tensor([[g["q"]]], dtype=torch.float32)
    out = run_oracle(lib, q, kc, vc, [g["block_table"]], [len(g["k"])], g["scale"], 1, B)
    np.testing.assert_allclose(out[0, 0], g["expected"], rtol=1e-15, atol=0)


def pin_single_token_is_v0(lib):
    """L = 1: the only weight is 1, so o equals v_0 exactly (any q, any scale)."""
    rng = np.random.default_rng(7)
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        c = random_case(rng, 1, 4, 2, 32, 16, dtype, max_len=1)
        out = run_oracle(lib, c["q"], c["kc"], c["vc"], c["tables"], c["lens"], 0.3, 2, 16)
        ref = c["V"][0][0].double().numpy()               # [Hkv, D]
        assert np.array_equal(out[0], ref[[0, 0, 1, 1]])


def pin_equal_keys_give_mean(lib):
    """All keys equal (or q = 0): uniform weights, o = mean of the values."""
    rng = np.random.default_rng(8)
    c = random_case(rng, 2, 2, 2, 16, 4, torch.float32, max_len=11)
    for s, L in enumerate(c["lens"]):
        c["K"][s][:] = c["K"][s][0:1]                     # identical keys
    kc, vc = scatter_dense(c["K"], c["V"], c["tables"], c["N"], 4, torch.float32)
    out = run_oracle(lib, c["q"], kc, vc, c["tables"], c["lens"], 0.7, 2, 4)
    for s in range(2):
        np.testing.assert_allclose(out[s], c["V"][s].double().mean(0).numpy(), rtol=1e-13,
                                   atol=1e-15)
    q0 = torch.zeros_like(c["q"])
    out0 = run_oracle(lib, q0, c["kc"], c["vc"], c["tables"], c["lens"], 0.7, 2, 4)
    for s in range(2):
        np.testing.assert_allclose(out0[s], c["V"][s].double().mean(0).numpy(), rtol=1e-13,
                                   atol=1e-15)


def pin_dense_equality(lib):
    """Paging changes only where K/V live: the oracle equals PyTorch's float64 SDPA on
    the unpaged arrays, for MHA and GQA, every dtype, several block sizes."""
    rng = np.random.default_rng(9)
    cases = [(3, 4, 4, 8, 1, torch.float32, 7), (3, 4, 2, 16, 2, torch.float16, 13),
             (4, 8, 2, 32, 4, torch.bfloat16, 29), (3, 6, 3, 64, 16, torch.float32, 70),
             (2, 8, 1, 128, 32, torch.bfloat16, 100)]
    for S, Hq, Hkv, D, B, dtype, max_len in cases:
        c = random_case(rng, S, Hq, Hkv, D, B, dtype, max_len)
        scale = 1.0 / math.sqrt(D)
        out = run_oracle(lib, c["q"], c["kc"], c["vc"], c["tables"], c["lens"], scale, Hkv, B)
        for s in range(S):
            ref = dense_reference(c["q"][s], c["K"][s], c["V"][s], scale)
            np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-13)


def pin_scale_is_applied(lib):
    """The scale multiplies q.k (checked against SDPA at a scale far from 1/sqrt(d))."""
    rng = np.random.default_rng(10)
    c = random_case(rng, 2, 2, 2, 8, 4, torch.float32, 9)
    for scale in (0.05, 2.5):
        out = run_oracle(lib, c["q"], c["kc"], c["vc"], c["tables"], c["lens"], scale, 2, 4)
        for s in range(2):
            ref = dense_reference(c["q"][s], c["K"][s], c["V"][s], scale)
            np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-13)


def pin_permutation_invariance(lib):
    """Any relabelling of physical blocks leaves the output bit-identical."""
    rng = np.random.default_rng(11)
    c = random_case(rng, 3, 4, 2, 32, 8, torch.bfloat16, 60, extra_blocks=5)
    base = run_oracle(lib, c["q"], c["kc"], c["vc"], c["tables"], c["lens"], 0.2, 2, 8)
    relabel = rng.permutation(c["N"])
    tables2 = [[int(relabel[b]) for b in t] for t in c["tables"]]
    kc2, vc2 = scatter_dense(c["K"], c["V"], tables2, c["N"], 8, torch.bfloat16)
    out2 = run_oracle(lib, c["q"], kc2, vc2, tables2, c["lens"], 0.2, 2, 8)
    assert np.array_equal(base, out2)


def pin_shared_vs_copied_prefix(lib):
    """Two sequences reading one shared prefix block set, or private copies of it,
    give bit-identical outputs (block sharing, Figures 8 and 9)."""
    rng = np.random.default_rng(12)
    B, Hkv, D = 4, 2, 16
    g = torch.Generator().manual_seed(5)
    P, L = 10, 14                                      # prefix tokens, total tokens
    prefix_k, prefix_v = torch.randn(P, Hkv, D, generator=g), torch.randn(P, Hkv, D, generator=g)
    tails = [(torch.randn(L - P, Hkv, D, generator=g), torch.randn(L - P, Hkv, D, generator=g))
             for _ in range(2)]
    K = [torch.cat([prefix_k, t[0]]) for t in tails]
    V = [torch.cat([prefix_v, t[1]]) for t in tails]
    q = torch.randn(2, 2, D, generator=g)
    # private copies: 4 blocks per sequence
    priv = [[0, 1, 2, 3], [4, 5, 6, 7]]
    kc1, vc1 = scatter_dense(K, V, priv, 12, B, torch.float32)
    out1 = run_oracle(lib, q, kc1, vc1, priv, [L, L], 0.25, Hkv, B)
    # shared: the first two (full) prefix blocks are shared; block 2 holds prefix
    # tokens 8-9 plus private tokens, so it is per sequence.
    shared = [[9, 10, 2, 3], [9, 10, 6, 7]]
    kc2, vc2 = scatter_dense(K, V, shared, 12, B, torch.float32)
    out2 = run_oracle(lib, q, kc2, vc2, shared, [L, L], 0.25, Hkv, B)
    assert np.array_equal(out1, out2)
    del rng


def pin_brute_force_small(lib):
    """Exhaustive small sweep, L in [1, 3B+1], B in {1, 2, 4}, against a direct loop that
    reads the pool slot by slot (no gather into contiguous arrays)."""
    rng = np.random.default_rng(13)
    D, Hq, Hkv = 3, 2, 1
    for B in (1, 2, 4):
        for L in range(1, 3 * B + 2):
            n = math.ceil(L / B)
            N = n + 2
            tab = [int(x) for x in rng.permutation(N)[:n]]
            kc = torch.from_numpy(rng.standard_normal((N, Hkv, B, D))).float()
            vc = torch.from_numpy(rng.standard_normal((N, Hkv, B, D))).float()
            q = torch.from_numpy(rng.standard_normal((1, Hq, D))).float()
            out = run_oracle(lib, q, kc, vc, [tab], [L], 0.9, Hkv, B)
            kk, vv, qq = kc.double().numpy(), vc.double().numpy(), q.double().numpy()
            for h in range(Hq):
                w = []
                for t in range(L):
                    blk, off = tab[t // B], t % B
                    w.append(math.exp(0.9 * sum(qq[0, h, d] * kk[blk, 0, off, d]
                                                for d in range(D))))
                tot = sum(w)
                for d in range(D):
                    ref = sum(w[t] * vv[tab[t // B], 0, t % B, d] for t in range(L)) / tot
                    assert abs(out[0, h, d] - ref) <= 1e-12 * max(1.0, abs(ref))


def pin_p3_mapping_table(lib):
    """Zero-based table (iaim.asia, section KV Cache 如何按块分配): token t of logical
    block j is read from block_table[j].  A one-hot key selects token t; the output
    must be the V row that the golden table places it in."""
    g = golden("p3_mapping.json")
    B = g["block_size"]
    table = [5, 0, 3]
    N = 6
    D = 4
    kc, vc = selector_case(B, N, table, D=D)
    for row in g["rows"]:
        for t in (row["first_token"], (row["first_token"] + row["last_token"]) // 2,
                  row["last_token"]):
            kc2 = torch.zeros_like(kc)
            blk = table[row["table_entry"]]
            off = t - row["first_token"]
            kc2[blk, 0, off, 3] = 1.0                      # only token t matches q
            q = torch.tensor([[[0.0, 0.0, 0.0, 2000.0]]])
            out = run_oracle(lib, q, kc2, vc, [table], [48], 1.0, 1, B)
            assert out[0, 0, 0] == blk and out[0, 0, 1] == off, (t, out[0, 0])


def pin_fig6_decode_walkthrough(lib):
    """Figure 6: prefill into blocks [7, 1], decode 1 fills block 1 slot 3, decode 2
    writes block 3 slot 0; attention over the grown table equals dense attention."""
    g = golden("fig6_block_table.json")
    B, D, Hkv = g["block_size"], 8, 2
    N = 8
    gen = torch.Generator().manual_seed(21)
    toks_k = torch.randn(9, Hkv, D, generator=gen)
    toks_v = torch.randn(9, Hkv, D, generator=gen)
    kc = torch.full((N, Hkv, B, D), float("nan"))
    vc = kc.clone()
    pre = g["prefill"]["placement"]
    slots = torch.tensor([b * B + o for b, o in pre], dtype=torch.int64)
    oracle.reshape_and_cache(toks_k[:7], toks_v[:7], kc, vc, slots, B, lib=lib)
    for i, (b, o) in enumerate(pre):
        assert torch.equal(kc[b, :, o], toks_k[i]) and torch.equal(vc[b, :, o], toks_v[i])
    filled = [int((~torch.isnan(kc[b, 0, :, 0])).sum()) for b in g["prefill"]["block_table"]]
    assert filled == g["prefill"]["filled"]
    q = torch.randn(1, 4, D, generator=gen)
    for step in ("decode1", "decode2"):
        st = g[step]
        t = st["token"]
        oracle.reshape_and_cache(toks_k[t:t + 1], toks_v[t:t + 1], kc, vc,
                                 torch.tensor([st["block"] * B + st["offset"]]), B, lib=lib)
        assert torch.equal(kc[st["block"], :, st["offset"]], toks_k[t])
        filled = [int((~torch.isnan(kc[b, 0, :, 0])).sum()) for b in st["block_table"]]
        assert filled == st["filled"]
        out = run_oracle(lib, q, kc, vc, [st["block_table"]], [t + 1], 0.3, Hkv, B)
        ref = dense_reference(q[0], toks_k[:t + 1], toks_v[:t + 1], 0.3)
        np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-13)


def pin_p5_block_table(lib):
    """p5 section 2.3: 7 tokens, block_size 4, table [3, 7] (one slot left)."""
    g = golden("p5_block_table.json")
    B, D = g["block_size"], 4
    gen = torch.Generator().manual_seed(22)
    k = torch.randn(g["tokens"], 1, D, generator=gen)
    v = torch.randn(g["tokens"], 1, D, generator=gen)
    kc = torch.full((8, 1, B, D), float("nan"))
    vc = kc.clone()
    slots = torch.tensor([b * B + o for b, o in g["placement"]], dtype=torch.int64)
    oracle.reshape_and_cache(k, v, kc, vc, slots, B, lib=lib)
    last = g["block_table"][-1]
    assert int(torch.isnan(kc[last, 0, :, 0]).sum()) == g["free_slots_in_last_block"]
    q = torch.randn(1, 1, D, generator=gen)
    out = run_oracle(lib, q, kc, vc, [g["block_table"]], [g["tokens"]], 0.5, 1, B)
    np.testing.assert_allclose(out[0], dense_reference(q[0], k, v, 0.5), rtol=1e-12, atol=1e-13)


def pin_fig8_copy_on_write(lib):
    """Figure 8: copy block 1 -> 3, A1 writes into 3, A2 into 1; the prompt part of
    both is unchanged and each sample's attention equals its own dense attention."""
    g = golden("fig8_cow.json")
    B, D, Hkv, N = g["block_size"], 8, 2, 8
    gen = torch.Generator().manual_seed(23)
    pk, pv = torch.randn(7, Hkv, D, generator=gen), torch.randn(7, Hkv, D, generator=gen)
    kc = torch.full((N, Hkv, B, D), float("nan"))
    vc = kc.clone()
    shared = g["shared_table"]
    slots = torch.tensor([shared[t // B] * B + t % B for t in range(7)])
    oracle.reshape_and_cache(pk, pv, kc, vc, slots, B, lib=lib)
    before7 = kc[7].clone()
    oracle.copy_blocks([kc, vc], [[g["copy"]["src"], g["copy"]["dst"]]], lib=lib)
    src, dst = g["copy"]["src"], g["copy"]["dst"]
    assert torch.equal(kc[dst].view(torch.int32), kc[src].view(torch.int32))
    assert torch.equal(vc[dst].view(torch.int32), vc[src].view(torch.int32))
    assert torch.equal(kc[7].view(torch.int32), before7.view(torch.int32))
    pos = g["write_position"]
    a1k, a1v = torch.randn(1, Hkv, D, generator=gen), torch.randn(1, Hkv, D, generator=gen)
    a2k, a2v = torch.randn(1, Hkv, D, generator=gen), torch.randn(1, Hkv, D, generator=gen)
    t1, t2 = g["a1_table_after"], g["a2_table_after"]
    oracle.reshape_and_cache(a1k, a1v, kc, vc, torch.tensor([t1[pos // B] * B + pos % B]), B,
                             lib=lib)
    oracle.reshape_and_cache(a2k, a2v, kc, vc, torch.tensor([t2[pos // B] * B + pos % B]), B,
                             lib=lib)
    q = torch.randn(2, 2, D, generator=gen)
    out = run_oracle(lib, q, kc, vc, [t1, t2], [pos + 1, pos + 1], 0.35, Hkv, B)
    np.testing.assert_allclose(out[0], dense_reference(q[0], torch.cat([pk, a1k]),
                                                       torch.cat([pv, a1v]), 0.35),
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out[1], dense_reference(q[1], torch.cat([pk, a2k]),
                                                       torch.cat([pv, a2v]), 0.35),
                               rtol=1e-12, atol=1e-13)


def pin_copy_blocks_reads_pre_copy_state(lib):
    """Copies read the state before the call: with pairs (a->b, b->c), c receives the
    old content of b, not a's."""
    pool = torch.arange(5 * 6, dtype=torch.float32).reshape(5, 6)
    old = pool.clone()
    oracle.copy_blocks([pool], [[0, 1], [1, 2]], lib=lib)
    assert torch.equal(pool[1], old[0]) and torch.equal(pool[2], old[1])
    assert torch.equal(pool[[0, 3, 4]], old[[0, 3, 4]])


def pin_reshape_bytes(lib):
    """reshape_and_cache is a byte copy: NaN payloads, -0.0 and untouched bytes survive,
    negative slots are skipped, each head's row lands at [slot/B][h][slot%B]."""
    B, Hkv, D, N = 4, 3, 8, 5
    gen = torch.Generator().manual_seed(24)
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        kc = torch.randn(N, Hkv, B, D, generator=gen).to(dtype)
        vc = torch.randn(N, Hkv, B, D, generator=gen).to(dtype)
        k = torch.randn(3, Hkv, D, generator=gen).to(dtype)
        v = torch.randn(3, Hkv, D, generator=gen).to(dtype)
        ib = torch.int32 if dtype == torch.float32 else torch.int16
        k.view(ib)[0, 0, 0] = -1              # a NaN with a payload
        k[0, 0, 1] = -0.0
        k0, v0 = kc.clone(), vc.clone()
        slots = torch.tensor([13, -1, 6])
        oracle.reshape_and_cache(k, v, kc, vc, slots, B, lib=lib)
        exp_k, exp_v = k0.clone(), v0.clone()
        exp_k[3, :, 1] = k[0]
        exp_v[3, :, 1] = v[0]
        exp_k[1, :, 2] = k[2]
        exp_v[1, :, 2] = v[2]
        assert torch.equal(kc.view(ib), exp_k.view(ib))
        assert torch.equal(vc.view(ib), exp_v.view(ib))


def pin_e4m3_decoder(lib):
    """Every OCP E4M3 code decodes as PyTorch's float8_e4m3fn decodes it."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([lib.orc_e4m3_to_f64(i) for i in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def _e4m3_probe_values():
    """fp32 values spanning E4M3's range: every code value, every midpoint between
    neighbours (ties), the midpoints nudged up and down, subnormals, both signs."""
    pos = torch.arange(0, 127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = pos.double()
    mids = (vals[1:] + vals[:-1]) / 2
    pts = torch.cat([vals, mids, mids * (1 + 2 ** -20), mids * (1 - 2 ** -20),
                     torch.linspace(0, 448, 2001, dtype=torch.float64)])
    pts = torch.cat([pts, -pts]).float()
    return pts[pts.abs() <= 448]


def pin_e4m3_encoder_rounds_to_nearest_even(lib):
    """In range, the encoder equals PyTorch's round-to-nearest-even cast, ties included."""
    x = _e4m3_probe_values()
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([lib.orc_f32_to_e4m3(float(v)) for v in x.tolist()], dtype=np.uint8)
    assert np.array_equal(ref, got)


def pin_e4m3_encoder_saturates(lib):
    """Beyond the largest finite magnitude (448) the encoder saturates (the reading for
    quantised caches); NaN stays NaN."""
    for x, code in [(449.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (float("inf"), 0x7E),
                    (-449.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE)]:
        assert lib.orc_f32_to_e4m3(x) == code, x
    assert lib.orc_f32_to_e4m3(float("nan")) & 0x7F == 0x7F


def _fp8_case(seed, S, Hq, Hkv, D, B, max_len):
    rng = np.random.default_rng(seed)
    c = random_case(rng, S, Hq, Hkv, D, B, torch.float32, max_len)
    g = torch.Generator().manual_seed(seed)
    ks = (torch.rand(Hkv, generator=g) * 0.02 + 0.005).float()      # per-head scales
    vs = (torch.rand(Hkv, generator=g) * 0.02 + 0.005).float()
    kq = torch.randint(0, 256, c["kc"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
    vq = torch.randint(0, 256, c["vc"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
    kq[(kq & 0x7F) == 0x7F] = 0x3F                                   # no NaN codes
    vq[(vq & 0x7F) == 0x7F] = 0x38
    return c, kq, vq, ks, vs


def pin_e4m3_attention_equals_dequantized_sdpa(lib):
    """Attention over an E4M3 cache equals PyTorch float64 SDPA over the dequantised
    (code value x the kv head's own scale) unpaged K and V."""
    for seed, (S, Hq, Hkv, D, B, max_len) in enumerate([(3, 4, 2, 16, 4, 23), (2, 8, 4, 32, 16, 60)]):
        c, kq, vq, ks, vs = _fp8_case(seed + 31, S, Hq, Hkv, D, B, max_len)
        out = oracle.paged_attention(c["q"], kq, vq, table_tensor(c["tables"]),
                                     torch.tensor(c["lens"], dtype=torch.int32), 0.3, Hkv, B,
                                     lib=lib, k_scale=ks, v_scale=vs)
        kd = kq.view(torch.float8_e4m3fn).double() * ks.double()[None, :, None, None]
        vd = vq.view(torch.float8_e4m3fn).double() * vs.double()[None, :, None, None]
        for s, L in enumerate(c["lens"]):
            tab = c["tables"][s]
            K = torch.stack([kd[tab[t // B], :, t % B] for t in range(L)])
            V = torch.stack([vd[tab[t // B], :, t % B] for t in range(L)])
            np.testing.assert_allclose(out[s], dense_reference(c["q"][s], K, V, 0.3),
                                       rtol=1e-12, atol=1e-12)


def pin_e4m3_cache_write(lib):
    """The quantising cache write stores PyTorch's nearest-even code of fp32(x) / scale[h]
    (IEEE fp32 division) at each token's slot, per head; other bytes are untouched."""
    Hkv, D, B, N = 3, 16, 4, 6
    g = torch.Generator().manual_seed(77)
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        k = (torch.randn(5, Hkv, D, generator=g) * 3).to(dtype)
        v = (torch.randn(5, Hkv, D, generator=g) * 3).to(dtype)
        ks = torch.tensor([0.01, 0.02, 0.05])
        vs = torch.tensor([0.03, 0.015, 0.04])
        kc = torch.full((N, Hkv, B, D), 0xAB, dtype=torch.uint8)
        vc = kc.clone()
        slots = torch.tensor([21, -1, 2, 9, 15])
        oracle.reshape_and_cache_e4m3(k, v, kc, vc, slots, B, ks, vs, lib=lib)
        want_k = torch.full_like(kc, 0xAB)
        want_v = torch.full_like(vc, 0xAB)
        for i, sl in enumerate(slots.tolist()):
            if sl < 0:
                continue
            qk = (k[i].float() / ks[:, None]).clamp(-448, 448)
            qv = (v[i].float() / vs[:, None]).clamp(-448, 448)
            want_k[sl // B, :, sl % B] = qk.to(torch.float8_e4m3fn).view(torch.uint8)
            want_v[sl // B, :, sl % B] = qv.to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(kc, want_k) and torch.equal(vc, want_v)


# ----------------------------------------------------------------------------- chunks

def chunk_case(rng, S, Hq, Hkv, D, B, dtype, max_len, full_prefill=False):
    """A paged case plus a chunk of n_s <= L_s query rows per sequence."""
    c = random_case(rng, S, Hq, Hkv, D, B, dtype, max_len)
    ns = [L if full_prefill else int(rng.integers(1, L + 1)) for L in c["lens"]]
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    g = torch.Generator().manual_seed(int(rng.integers(0, 2**31)))
    c["ns"] = ns
    c["query_start"] = torch.from_numpy(qs)
    c["qc"] = torch.randn(int(qs[-1]), Hq, D, generator=g).to(dtype)
    return c


def run_chunk(lib, c, scale, Hkv, B, query_start=None, lens=None, q=None):
    lens = c["lens"] if lens is None else lens
    return oracle.chunk_attention(c["qc"] if q is None else q, c["kc"], c["vc"],
                                  table_tensor(c["tables"]), torch.tensor(lens, dtype=torch.int32),
                                  c["query_start"] if query_start is None else query_start,
                                  scale, Hkv, B, lib=lib)


def pin_chunk_hand_case(lib):
    """Two sequences with chunks of 2 and 1 tokens, evaluated by hand
    (tests/golden/chunk_causal_hand.json)."""
    g = golden("chunk_causal_hand.json")
    B, D, N = g["block_size"], g["head_dim"], g["num_blocks"]
    kc = torch.full((N, 1, B, D), float("nan"))
    vc = kc.clone()
    q, tables, lens = [], [], []
    for sq in g["sequences"]:
        for t, (k, v) in enumerate(zip(sq["k"], sq["v"])):
            kc[sq["block_table"][t // B], 0, t % B] = torch.tensor(k)
            vc[sq["block_table"][t // B], 0, t % B] = torch.tensor(v)
        q += sq["q"]
        tables.append(sq["block_table"])
        lens.append(sq["context_len"])
    out = oracle.chunk_attention(torch.tensor(q)[:, None, :], kc, vc, table_tensor(tables),
                                 torch.tensor(lens, dtype=torch.int32),
                                 torch.tensor(g["query_start"], dtype=torch.int32), g["scale"],
                                 1, B, lib=lib)
    np.testing.assert_allclose(out[:, 0], g["expected"], rtol=1e-14, atol=0)


def pin_chunk_full_prefill_is_causal_sdpa(lib):
    """A chunk that is the whole context (n = L) is ordinary causal self-attention:
    PyTorch's float64 SDPA with is_causal=True on the unpaged arrays, MHA and GQA."""
    rng = np.random.default_rng(21)
    for S, Hq, Hkv, D, B, dtype, max_len in [(3, 4, 4, 16, 4, torch.float32, 23),
                                             (2, 8, 2, 32, 16, torch.bfloat16, 40),
                                             (2, 6, 3, 64, 8, torch.float16, 19)]:
        c = chunk_case(rng, S, Hq, Hkv, D, B, dtype, max_len, full_prefill=True)
        scale = 1.0 / math.sqrt(D)
        out = run_chunk(lib, c, scale, Hkv, B)
        qs = c["query_start"].tolist()
        for s in range(S):
            q64 = c["qc"][qs[s]:qs[s + 1]].double().permute(1, 0, 2)[None]
            k64 = c["K"][s].double().permute(1, 0, 2)[None]
            v64 = c["V"][s].double().permute(1, 0, 2)[None]
            ref = F.scaled_dot_product_attention(q64, k64, v64, scale=scale, is_causal=True,
                                                 enable_gqa=Hq != Hkv)[0].permute(1, 0, 2)
            np.testing.assert_allclose(out[qs[s]:qs[s + 1]], ref.numpy(), rtol=1e-12, atol=1e-13)


def pin_chunk_rows_see_their_prefix(lib):
    """Chunk row j of a sequence (n < L) equals unmasked SDPA over the first
    L - n + j + 1 cached tokens; the last row sees the whole context."""
    rng = np.random.default_rng(22)
    c = chunk_case(rng, 4, 4, 2, 32, 8, torch.bfloat16, 45)
    scale = 1.0 / math.sqrt(32)
    out = run_chunk(lib, c, scale, 2, 8)
    qs = c["query_start"].tolist()
    for s, (L, n) in enumerate(zip(c["lens"], c["ns"])):
        for j in range(n):
            vis = L - n + j + 1
            ref = dense_reference(c["qc"][qs[s] + j], c["K"][s][:vis], c["V"][s][:vis], scale)
            np.testing.assert_allclose(out[qs[s] + j], ref, rtol=1e-12, atol=1e-13)


def pin_chunking_invariance(lib):
    """Chunked prefill: attending a chunk at once equals attending it as two
    consecutive chunks, the first over the shorter context it had then."""
    rng = np.random.default_rng(23)
    c = chunk_case(rng, 3, 4, 4, 16, 4, torch.float32, 40, full_prefill=True)
    whole = run_chunk(lib, c, 0.25, 4, 4)
    qs = c["query_start"].tolist()
    for s, L in enumerate(c["lens"]):
        n1 = L // 2
        rows = c["qc"][qs[s]:qs[s + 1]]
        one = dict(c, tables=[c["tables"][s]])
        first = run_chunk(lib, one, 0.25, 4, 4, torch.tensor([0, n1], dtype=torch.int32),
                          [n1], rows[:n1]) if n1 > 0 else np.zeros((0,) + whole.shape[1:])
        second = run_chunk(lib, one, 0.25, 4, 4, torch.tensor([0, L - n1], dtype=torch.int32),
                           [L], rows[n1:])
        assert np.array_equal(np.concatenate([first, second]), whole[qs[s]:qs[s + 1]])


def pin_chunk_of_one_is_decode_sdpa(lib):
    """One new token per sequence (n = 1) is plain decode attention over the whole
    context (SDPA on the unpaged arrays), as in the single-query kernel."""
    rng = np.random.default_rng(24)
    c = random_case(rng, 5, 8, 2, 64, 16, torch.bfloat16, 70)
    c["query_start"] = torch.arange(6, dtype=torch.int32)
    c["qc"] = c["q"]
    out = run_chunk(lib, c, 0.125, 2, 16)
    for s in range(5):
        np.testing.assert_allclose(out[s], dense_reference(c["q"][s], c["K"][s], c["V"][s], 0.125),
                                   rtol=1e-12, atol=1e-13)


def pin_chunk_e4m3_equals_dequantized_causal_sdpa(lib):
    """Whole-context chunks over E4M3 pools equal PyTorch's float64 causal SDPA on the
    dequantised (code x per-kv-head scale) keys and values."""
    rng = np.random.default_rng(26)
    c = chunk_case(rng, 2, 8, 2, 32, 8, torch.float32, 30, full_prefill=True)
    ks = torch.tensor([0.05, 0.11])
    vs = torch.tensor([0.07, 0.03])
    kq = (c["kc"] / ks[None, :, None, None]).to(torch.float8_e4m3fn)
    vq = (c["vc"] / vs[None, :, None, None]).to(torch.float8_e4m3fn)
    out = oracle.chunk_attention(c["qc"], kq, vq, table_tensor(c["tables"]),
                                 torch.tensor(c["lens"], dtype=torch.int32), c["query_start"],
                                 0.25, 2, 8, lib=lib, k_scale=ks, v_scale=vs)
    kd = kq.double() * ks.double()[None, :, None, None]
    vd = vq.double() * vs.double()[None, :, None, None]
    qs = c["query_start"].tolist()
    for s, (L, tab) in enumerate(zip(c["lens"], c["tables"])):
        K = torch.stack([kd[tab[t // 8], :, t % 8] for t in range(L)])      # [L, Hkv, D]
        V = torch.stack([vd[tab[t // 8], :, t % 8] for t in range(L)])
        q64 = c["qc"][qs[s]:qs[s + 1]].double().permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(q64, K.permute(1, 0, 2)[None], V.permute(1, 0, 2)[None],
                                             scale=0.25, is_causal=True, enable_gqa=True)
        np.testing.assert_allclose(out[qs[s]:qs[s + 1]], ref[0].permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-13)


def pin_chunk_longer_than_context_is_nan(lib):
    """A chunk longer than its context is malformed: its rows come back NaN and the
    other sequences are unaffected."""
    rng = np.random.default_rng(25)
    c = random_case(rng, 2, 2, 2, 8, 4, torch.float32, 9)
    lens = [c["lens"][0], c["lens"][1]]
    n0 = lens[0] + 1
    c["query_start"] = torch.tensor([0, n0, n0 + 1], dtype=torch.int32)
    c["qc"] = torch.randn(n0 + 1, 2, 8)
    out = run_chunk(lib, c, 0.5, 2, 4)
    assert np.isnan(out[:n0]).all()
    ref = dense_reference(c["qc"][n0], c["K"][1], c["V"][1], 0.5)
    np.testing.assert_allclose(out[n0], ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- swapping

def pin_swap_moves_blocks_by_index(lib):
    """swap_blocks writes dst[d] = src[s] for each pair (numpy fancy indexing as the
    reference), leaves every other destination block and the source untouched."""
    g = torch.Generator().manual_seed(31)
    src = [torch.randn(9, 2, 4, 8, generator=g).to(torch.bfloat16) for _ in range(3)]
    dst = [torch.randn(6, 2, 4, 8, generator=g).to(torch.bfloat16) for _ in range(3)]
    before_src = [t.clone() for t in src]
    want = [t.clone() for t in dst]
    pairs = [(7, 0), (2, 5), (4, 3)]
    for w, sr in zip(want, src):
        w[[d for _, d in pairs]] = sr[[s for s, _ in pairs]]
    oracle.swap_blocks(src, dst, pairs, lib=lib)
    for a, b in zip(dst, want):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(src, before_src):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def pin_swap_out_and_in_restores_attention(lib):
    """A preempted sequence swapped out to a CPU pool and back into other GPU blocks
    ("调度与抢占", 换出: copied out, returned when memory frees) attends exactly as
    before once its block table names the new blocks."""
    rng = np.random.default_rng(32)
    c = random_case(rng, 3, 4, 2, 32, 8, torch.float32, 60, extra_blocks=12)
    lens, tables = c["lens"], c["tables"]
    before = run_oracle(lib, c["q"], c["kc"], c["vc"], tables, lens, 0.2, 2, 8)
    victim = 1
    used = {b for t in tables for b in t}
    free = [b for b in range(c["N"]) if b not in used]
    cpu_k = torch.zeros((len(tables[victim]),) + tuple(c["kc"].shape[1:]))
    cpu_v = torch.zeros_like(cpu_k)
    out_pairs = [(b, i) for i, b in enumerate(tables[victim])]
    oracle.swap_blocks([c["kc"], c["vc"]], [cpu_k, cpu_v], out_pairs, lib=lib)
    c["kc"][tables[victim]] = float("nan")               # the GPU blocks are reused
    c["vc"][tables[victim]] = float("nan")
    new = free[:len(tables[victim])]
    oracle.swap_blocks([cpu_k, cpu_v], [c["kc"], c["vc"]], list(enumerate(new)), lib=lib)
    tables = [t if s != victim else new for s, t in enumerate(tables)]
    after = run_oracle(lib, c["q"], c["kc"], c["vc"], tables, lens, 0.2, 2, 8)
    assert np.array_equal(before, after)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
