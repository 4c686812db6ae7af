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


# --------------------------------------------------------------------------- swapping

def sharing_pattern(tables):
    """Which (sequence, logical block) positions name the same physical block --
    the structure swapping must preserve, whatever the ids."""
    first = {}
    out = {}
    for s in sorted(tables):
        for j, b in enumerate(tables[s]):
            out[(s, j)] = first.setdefault(b, (s, j))
    return out


def test_beam_group_swaps_out_and_back_keeping_its_sharing():
    """A beam group (Figure 9's sharing: a prefix shared by all, blocks shared by pairs)
    is preempted all-or-nothing ("调度与抢占", 换出): each distinct block goes to the CPU
    once, the references follow, the GPU blocks are free again; swapped back in, the
    group has the same sharing over new GPU blocks and decodes on."""
    m = BlockManager(24, 4)
    m.set_cpu_pool(24)
    m.add_sequence(0, 10)                      # blocks 0, 1, 2 (2 tokens in the last)
    for c in (1, 2, 3):
        m.fork(0, c)
    m.append([0, 1, 2, 3])                     # CoW of the shared partial last block
    for _ in range(4):
        m.append([0, 1, 2, 3])
    group = [0, 1, 2, 3]
    before = {s: [int(x) for x in m.block_tables([s], 16)[0][0] if x >= 0] for s in group}
    distinct = {b for t in before.values() for b in t}
    refs_before = {b: m.ref_count(b) for b in distinct}
    free_before = m.num_free_blocks()
    pairs = m.swap_out(group)
    assert sorted(int(g) for g, _ in pairs) == sorted(distinct)           # each block once
    assert len({int(c) for _, c in pairs}) == len(pairs)
    assert m.num_free_blocks() == free_before + len(distinct)
    for g, c in pairs:
        assert m.cpu_ref_count(int(c)) == refs_before[int(g)] and m.ref_count(int(g)) == 0
    assert all(m.is_swapped(s) for s in group)
    with pytest.raises(N.PAError):
        m.append([0])                          # a swapped-out sequence cannot grow
    with pytest.raises(N.PAError):
        m.block_tables([1], 16)
    with pytest.raises(N.PAError):
        m.fork(2, 9)
    # the freed GPU blocks serve someone else meanwhile
    m.add_sequence(100, 4 * m.num_free_blocks())
    with pytest.raises(N.PAError):
        m.swap_in(group)                       # no room: nothing changes
    assert all(m.is_swapped(s) for s in group)
    m.free(100)
    back = m.swap_in(group)
    assert sorted(int(c) for c, _ in back) == sorted(int(c) for _, c in pairs)
    after = {s: [int(x) for x in m.block_tables([s], 16)[0][0] if x >= 0] for s in group}
    assert sharing_pattern(after) == sharing_pattern(before)
    assert m.num_free_cpu_blocks() == 24
    slots, cow = m.append(group)               # decoding resumes
    assert len(slots) == 4


def test_swap_all_or_nothing_on_a_small_cpu_pool():
    m = BlockManager(16, 4)
    m.set_cpu_pool(3)
    m.add_sequence(0, 13)                      # 4 blocks, more than the CPU pool holds
    with pytest.raises(N.PAError):
        m.swap_out([0])
    assert not m.is_swapped(0) and m.num_free_blocks() == 12 and m.num_free_cpu_blocks() == 3
    m.add_sequence(1, 12)                      # 3 blocks fit
    pairs = m.swap_out([1])
    assert len(pairs) == 3 and m.num_free_cpu_blocks() == 0
    m.free(1)                                  # freeing a swapped-out sequence returns its CPU blocks
    assert m.num_free_cpu_blocks() == 3
    with pytest.raises(N.PAError):
        m.swap_in([0])                         # not swapped out
    with pytest.raises(N.PAError):
        BlockManager(4, 4).swap_out([0])       # no CPU pool


@pytest.mark.parametrize("seed", range(6))
def test_native_matches_model_with_swapping(seed):
    """Random add / fork / append / free / swap-out / swap-in, native against the model."""
    rng = random.Random(100 + seed)
    n_blocks, bs, n_cpu = rng.choice([(24, 4, 16), (48, 2, 48), (32, 8, 10)])
    a, b = BlockManagerModel(n_blocks, bs), BlockManager(n_blocks, bs)
    a.set_cpu_pool(n_cpu)
    b.set_cpu_pool(n_cpu)
    live, next_id = [], 0
    for _ in range(400):
        op = rng.random()
        gpu = [s for s in live if s not in a.on_cpu]
        cpu = [s for s in live if s in a.on_cpu]
        if op < 0.12 or not live:
            n = rng.randrange(0, 3 * bs)
            try:
                ra = a.add_sequence(next_id, n)
            except PoolExhausted:
                with pytest.raises(N.PAError):
                    b.add_sequence(next_id, n)
                continue
            assert ra == list(b.add_sequence(next_id, n))
            live.append(next_id)
            next_id += 1
        elif op < 0.25 and gpu:
            p = rng.choice(gpu)
            a.fork(p, next_id)
            b.fork(p, next_id)
            live.append(next_id)
            next_id += 1
        elif op < 0.65 and gpu:
            batch = rng.sample(gpu, rng.randint(1, len(gpu)))
            try:
                ra = a.append(batch)
            except PoolExhausted:
                with pytest.raises(N.PAError):
                    b.append(batch)
                continue
            rb = b.append(batch)
            assert ra == (list(rb[0]), [tuple(x) for x in rb[1].tolist()])
        elif op < 0.78 and gpu:
            group = rng.sample(gpu, rng.randint(1, min(3, len(gpu))))
            try:
                ra = a.swap_out(group)
            except PoolExhausted:
                with pytest.raises(N.PAError):
                    b.swap_out(group)
                continue
            assert ra == [tuple(x) for x in b.swap_out(group).tolist()]
        elif op < 0.9 and cpu:
            group = rng.sample(cpu, rng.randint(1, min(3, len(cpu))))
            try:
                ra = a.swap_in(group)
            except PoolExhausted:
                with pytest.raises(N.PAError):
                    b.swap_in(group)
                continue
            assert ra == [tuple(x) for x in b.swap_in(group).tolist()]
        elif live:
            s = live.pop(rng.randrange(len(live)))
            a.free_sequence(s)
            b.free(s)
        for s in live:
            assert b.is_swapped(s) == (s in a.on_cpu)
            if s not in a.on_cpu:
                t, _ = b.block_tables([s], 64)
                assert [int(x) for x in t[0] if x >= 0] == a.tables[s]
        assert [b.ref_count(x) for x in range(n_blocks)] == a.refs
        assert [b.cpu_ref_count(x) for x in range(n_cpu)] == a.cpu_refs
        assert b.num_free_blocks() == len(a.free) and b.num_free_cpu_blocks() == len(a.cpu_free)
