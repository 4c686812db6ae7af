"""Host KV block manager (C++ in libpa.so) and its reference model (oracle/), pinned by
the pages' Figures 6, 8 and 9, then compared operation by operation on random workloads."""
import json
import os
import random

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, PoolExhausted
from paged_kv_cache_119_gb300 import _native as N
from paged_kv_cache_119_gb300 import build as B
from paged_kv_cache_119_gb300.block_manager import BlockManager

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


class Native:
    """The C++ manager behind the reference model's interface."""

    def __init__(self, n, bs, order=None):
        self.m = BlockManager(n, bs, order)

    def add_sequence(self, s, n):
        return list(self.m.add_sequence(s, n))

    def fork(self, p, c):
        self.m.fork(p, c)

    def append(self, seqs):
        try:
            slots, pairs = self.m.append(seqs)
        except N.PAError:
            raise PoolExhausted()
        return list(slots), [tuple(p) for p in pairs]

    def free_sequence(self, s):
        self.m.free(s)

    def table(self, s):
        t, _ = self.m.block_tables([s], 64)
        return [int(x) for x in t[0] if x >= 0]

    def refs(self, b):
        return self.m.ref_count(b)


def model_table(m, s):
    return list(m.tables[s])


IMPLS = ["model", "native"]


def make(kind, n, bs, order=None):
    return BlockManagerModel(n, bs, order) if kind == "model" else Native(n, bs, order)


def table_of(mgr, s):
    return model_table(mgr, s) if isinstance(mgr, BlockManagerModel) else mgr.table(s)


def refs_of(mgr, b):
    return mgr.refs[b] if isinstance(mgr, BlockManagerModel) else mgr.refs(b)


@pytest.mark.parametrize("kind", IMPLS)
def test_figure6_prompt_and_two_decode_steps(kind):
    g = golden("fig6_block_table.json")
    bs = g["block_size"]
    order = [7, 1, 3] + [b for b in range(8) if b not in (7, 1, 3)]
    m = make(kind, 8, bs, order)
    slots = m.add_sequence(0, g["prompt_tokens"])
    assert table_of(m, 0) == g["prefill"]["block_table"]
    assert slots == [b * bs + o for b, o in g["prefill"]["placement"]]
    for step in ("decode1", "decode2"):
        st = g[step]
        s, pairs = m.append([0])
        assert s == [st["block"] * bs + st["offset"]] and pairs == []
        assert table_of(m, 0) == st["block_table"]


@pytest.mark.parametrize("kind", IMPLS)
def test_figure8_copy_on_write(kind):
    g = golden("fig8_cow.json")
    bs = g["block_size"]
    order = [7, 1, 3] + [b for b in range(8) if b not in (7, 1, 3)]
    m = make(kind, 8, bs, order)
    m.add_sequence(1, g["prompt_tokens"])            # A1
    m.fork(1, 2)                                     # A2 shares the prompt blocks
    assert table_of(m, 2) == g["shared_table"]
    for b, r in g["refcount_before"].items():
        assert refs_of(m, int(b)) == r
    slots, pairs = m.append([1, 2])                  # A1 writes first, then A2
    assert pairs == [(g["copy"]["src"], g["copy"]["dst"])]
    assert table_of(m, 1) == g["a1_table_after"] and table_of(m, 2) == g["a2_table_after"]
    pos = g["write_position"]
    assert slots == [g["a1_table_after"][pos // bs] * bs + pos % bs,
                     g["a2_table_after"][pos // bs] * bs + pos % bs]
    for b, r in g["refcount_after"].items():
        assert refs_of(m, int(b)) == r


@pytest.mark.parametrize("kind", IMPLS)
def test_figure9_beam_search_sharing(kind):
    """Replays a beam of width 4 (block size 4, full blocks) into the state Figure 9
    describes, then the step after the dashed line."""
    g = golden("fig9_beam.json")
    bs = 4
    order = [0, 1, 2, 3, 4, 5, 8, 6, 7, 9, 10, 11, 12, 13, 14, 15]
    m = make(kind, 16, bs, order)

    def grow(seqs, tokens):
        for _ in range(tokens):
            m.append(seqs)

    m.add_sequence(0, 4)               # prompt: logical block 0
    m.fork(0, 3)                       # candidate 3 diverges from logical block 1
    grow([0], 4)
    grow([3], 4)
    grow([0], 4)
    grow([3], 8)
    m.fork(0, 1)                       # candidates 0-2 share logical blocks 1-2
    m.fork(0, 2)
    grow([0, 1, 2], 4)                 # and diverge at logical block 3
    tables = {c: table_of(m, c) for c in range(4)}
    assert all(len(t) == g["logical_blocks_before"] for t in tables.values())
    assert set.intersection(*[set(t) for t in tables.values()]) == set(g["shared_by_all_before"])
    assert tables[3][1] not in tables[0]                       # 3 diverged at logical block 1
    assert tables[0][:3] == tables[1][:3] == tables[2][:3]     # 0-2 share logical blocks 1-2
    assert len({tables[c][3] for c in (0, 1, 2)}) == 3         # and diverge at block 3
    # the dashed line: new candidates come from old 1 and 2; old 0 and 3 are dropped
    refs_before = [refs_of(m, b) for b in range(16)]
    m.free_sequence(0)
    m.free_sequence(3)
    freed = sorted(b for b in range(16) if refs_before[b] > 0 and refs_of(m, b) == 0)
    assert freed == g["freed_blocks"]
    for new, parent in ((10, 1), (11, 1), (12, 2), (13, 2)):
        m.fork(parent, new)
    m.free_sequence(1)
    m.free_sequence(2)
    slots, pairs = m.append([10, 11, 12, 13])
    assert pairs == []
    after = {i: table_of(m, c) for i, c in enumerate((10, 11, 12, 13))}
    assert sorted(t[-1] for t in after.values()) == g["new_blocks"]
    assert set.intersection(*[set(t) for t in after.values()]) == set(g["shared_by_all_after"])
    for (a, b), blk in g["shared_pairs_after"]:
        assert blk in after[a] and blk in after[b]
        assert all(blk not in after[c] for c in range(4) if c not in (a, b))


def check_invariants(m, seqs, bs, n_blocks):
    count = [0] * n_blocks
    for s in seqs:
        t = m.tables[s]
        assert len(t) == -(-m.tokens[s] // bs)          # waste <= block_size - 1 tokens
        for b in t:
            count[b] += 1
    assert count == m.refs
    assert sorted(m.free) == [b for b in range(n_blocks) if count[b] == 0]


@pytest.mark.parametrize("seed", range(6))
def test_native_matches_model_on_random_workloads(seed):
    rng = random.Random(seed)
    n_blocks, bs = rng.choice([(24, 4), (64, 16), (40, 2)])
    order = list(range(n_blocks))
    rng.shuffle(order)
    a, b = BlockManagerModel(n_blocks, bs, order), Native(n_blocks, bs, order)
    live, next_id = [], 0
    for _ in range(300):
        op = rng.random()
        try:
            if op < 0.15 or not live:
                n = rng.randrange(0, 3 * bs)
                ra = a.add_sequence(next_id, n)
                rb = b.add_sequence(next_id, n)
                assert ra == rb
                live.append(next_id)
                next_id += 1
            elif op < 0.3:
                p = rng.choice(live)
                a.fork(p, next_id)
                b.fork(p, next_id)
                live.append(next_id)
                next_id += 1
            elif op < 0.85:
                batch = rng.sample(live, rng.randint(1, len(live)))
                try:
                    ra = a.append(batch)
                except PoolExhausted:
                    with pytest.raises(PoolExhausted):
                        b.append(batch)
                    continue
                assert ra == b.append(batch)
            else:
                s = live.pop(rng.randrange(len(live)))
                a.free_sequence(s)
                b.free_sequence(s)
        except PoolExhausted:
            with pytest.raises((PoolExhausted, N.PAError)):
                if op < 0.15 or not live:
                    b.add_sequence(next_id, n)
            continue
        for s in live:
            assert table_of(a, s) == table_of(b, s)
        assert [refs_of(a, x) for x in range(n_blocks)] == [refs_of(b, x) for x in range(n_blocks)]
        check_invariants(a, live, bs, n_blocks)


def test_exhausted_pool_changes_nothing():
    m = BlockManager(4, 4)
    m.add_sequence(0, 8)
    m.add_sequence(1, 8)
    with pytest.raises(N.PAError):
        m.append([0, 1])                   # needs 2 new blocks, 0 free
    assert m.num_tokens(0) == 8 and m.num_tokens(1) == 8 and m.num_free_blocks() == 0
    with pytest.raises(N.PAError):
        m.add_sequence(2, 1)
    with pytest.raises(N.PAError):
        m.fork(7, 8)                       # unknown parent
    with pytest.raises(N.PAError):
        m.append([0, 0])                   # a sequence listed twice
    with pytest.raises(ValueError):
        BlockManager(4, 4, [0, 1, 1, 2])   # not a permutation
