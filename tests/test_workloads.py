"""Host-side checks of the seeded input generator (no GPU)."""
import math

import numpy as np
import torch

from paged_kv_cache_119_gb300 import workloads


def _check_tables(w):
    lens = w.context_lens.tolist()
    bt = w.block_tables
    used = []
    for s, L in enumerate(lens):
        n = math.ceil(L / w.block_size)
        row = bt[s].tolist()
        assert all(0 <= b < w.num_blocks for b in row[:n])
        assert all(b == -1 for b in row[n:])
        # internal fragmentation: at most block_size - 1 unused slots per sequence
        assert n * w.block_size - L <= w.block_size - 1
        used.extend(row[:n])
    return used


def test_tiny_shape_and_nan_fill():
    w = workloads.make("tiny")
    assert w.context_lens.tolist() == [1, 15, 16, 37]
    assert w.num_blocks == 16 and w.k_cache.shape == (16, 2, 16, 64)
    used = _check_tables(w)
    assert len(set(used)) == len(used) == 6
    # tokens 0..L-2 cached, everything else NaN (the step writes token L-1)
    for s, L in enumerate(w.context_lens.tolist()):
        for t in range(L):
            b, o = int(w.block_tables[s, t // 16]), t % 16
            assert torch.isnan(w.k_cache[b, :, o]).all() == (t == L - 1)
    assert torch.equal(w.slot_mapping,
                       torch.tensor([int(w.block_tables[s, (L - 1) // 16]) * 16 + (L - 1) % 16
                                     for s, L in enumerate(w.context_lens.tolist())]))


def test_seeded_and_reproducible():
    a, b = workloads.make("tiny"), workloads.make("tiny")
    assert torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_cache.nan_to_num(), b.k_cache.nan_to_num())
    c = workloads.make("tiny", seed=5)
    assert not torch.equal(a.q, c.q)


def test_llama_lengths_and_pool():
    w = workloads.make("llama13b", num_seqs=64)
    lens = np.array(w.context_lens.tolist())
    assert lens.min() >= 16 and lens.max() <= 2048
    used = _check_tables(w)
    assert len(set(used)) == len(used)
    assert w.num_blocks == math.ceil(1.1 * len(used))


def test_prefix_sharing_and_cow_pairs():
    w = workloads.make("prefix", num_groups=3, group_size=4, prefix_blocks=4, max_suffix=40)
    pairs = w.copy_pairs
    assert pairs.shape == (3 * 3, 2)
    dst, src = set(pairs[:, 1].tolist()), set(pairs[:, 0].tolist())
    assert len(dst) == len(pairs) and not (dst & src)
    bt = w.block_tables
    for g in range(3):
        rows = bt[g * 4:(g + 1) * 4]
        assert (rows[:, :4] == rows[0, :4]).all()          # shared prefix blocks
        tails = rows[:, 4].tolist()
        assert len(set(tails)) == 4                        # CoW split tail blocks
        assert tails[-1] in src                            # last sample keeps the original
    _check_tables(w)
    # every suffix token gets written by the step, nothing else
    assert w.slot_mapping.numel() == sum(w.meta["suffix"])
