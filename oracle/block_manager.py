"""Reference model of the KV block manager -- TEST INFRASTRUCTURE ONLY.

Plain Python restatement of the pages' memory-management rules, used to check
the C++ manager in libpa.so operation by operation ("PagedAttention 完全拆解",
sections 原理详解（一） (Figure 6), 内存共享 / 引用计数 (Figure 8), Beam Search
(Figure 9) and 三种原语：fork、append、free):

  * tokens fill a sequence's logical blocks left to right; a new physical block
    is taken only when the last one is full;
  * each physical block counts the sequences whose tables name it;
  * fork copies the parent's table and counts each block once more;
  * append to a shared, partially filled last block first takes a new block,
    records a (old, new) copy, and moves the writer onto the new block;
  * free uncounts each block; a block whose count reaches zero is free again.

  * swapping (section 调度与抢占：内存不够时怎么办, 换出): a sequence group moves to a
    CPU pool as a whole -- each distinct block once, sharing kept -- and back.

The free lists hand blocks out first-in first-out.  Pinned by
tests/test_block_manager.py against Figures 6, 8 and 9.
"""
from __future__ import annotations

from collections import deque


class PoolExhausted(Exception):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int, alloc_order=None):
        order = list(range(num_blocks)) if alloc_order is None else list(alloc_order)
        assert sorted(order) == list(range(num_blocks))
        self.B = block_size
        self.free = deque(order)
        self.refs = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.tokens: dict[int, int] = {}
        self.cpu_free: deque = deque()
        self.cpu_refs: list[int] = []
        self.on_cpu: set = set()

    def _take(self) -> int:
        if not self.free:
            raise PoolExhausted()
        b = self.free.popleft()
        self.refs[b] = 1
        return b

    def _slot(self, seq, t):
        return self.tables[seq][t // self.B] * self.B + t % self.B

    def add_sequence(self, seq: int, num_tokens: int) -> list[int]:
        assert seq not in self.tables
        need = -(-num_tokens // self.B)
        if need > len(self.free):
            raise PoolExhausted()
        self.tables[seq] = [self._take() for _ in range(need)]
        self.tokens[seq] = num_tokens
        return [self._slot(seq, t) for t in range(num_tokens)]

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.tables and parent in self.tables and parent not in self.on_cpu
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = self.tokens[parent]
        for b in self.tables[child]:
            self.refs[b] += 1

    def append(self, seqs) -> tuple[list[int], list[tuple[int, int]]]:
        """One new token for each listed sequence, in order.  All or nothing."""
        assert len(set(seqs)) == len(seqs) and not set(seqs) & self.on_cpu
        snapshot = (deque(self.free), list(self.refs),
                    {s: list(t) for s, t in self.tables.items()}, dict(self.tokens))
        try:
            slots, pairs = [], []
            for s in seqs:
                t = self.tokens[s]
                if t % self.B == 0:
                    self.tables[s].append(self._take())
                else:
                    last = self.tables[s][-1]
                    if self.refs[last] > 1:
                        new = self._take()
                        pairs.append((last, new))
                        self.refs[last] -= 1
                        self.tables[s][-1] = new
                slots.append(self._slot(s, t))
                self.tokens[s] = t + 1
            return slots, pairs
        except PoolExhausted:
            self.free, self.refs, self.tables, self.tokens = snapshot
            raise

    def free_sequence(self, seq: int) -> None:
        cpu = seq in self.on_cpu
        refs, free = (self.cpu_refs, self.cpu_free) if cpu else (self.refs, self.free)
        for b in self.tables.pop(seq):
            refs[b] -= 1
            if refs[b] == 0:
                free.append(b)
        del self.tokens[seq]
        self.on_cpu.discard(seq)

    def set_cpu_pool(self, num_cpu_blocks: int) -> None:
        assert not self.cpu_refs and num_cpu_blocks > 0
        self.cpu_refs = [0] * num_cpu_blocks
        self.cpu_free = deque(range(num_cpu_blocks))

    def _swap(self, seqs, to_cpu: bool) -> list[tuple[int, int]]:
        assert self.cpu_refs and len(set(seqs)) == len(seqs)
        assert all((s in self.on_cpu) != to_cpu for s in seqs)
        order, uses = [], {}
        for s in seqs:
            for b in self.tables[s]:
                if b not in uses:
                    order.append(b)
                uses[b] = uses.get(b, 0) + 1
        src_refs, src_free = (self.refs, self.free) if to_cpu else (self.cpu_refs, self.cpu_free)
        dst_refs, dst_free = (self.cpu_refs, self.cpu_free) if to_cpu else (self.refs, self.free)
        if len(order) > len(dst_free):
            raise PoolExhausted()
        moved = {}
        for b in order:
            d = dst_free.popleft()
            dst_refs[d] = uses[b]
            src_refs[b] -= uses[b]
            if src_refs[b] == 0:
                src_free.append(b)
            moved[b] = d
        for s in seqs:
            self.tables[s] = [moved[b] for b in self.tables[s]]
            if to_cpu:
                self.on_cpu.add(s)
            else:
                self.on_cpu.discard(s)
        return [(b, moved[b]) for b in order]

    def swap_out(self, seqs) -> list[tuple[int, int]]:
        return self._swap(seqs, True)

    def swap_in(self, seqs) -> list[tuple[int, int]]:
        return self._swap(seqs, False)
