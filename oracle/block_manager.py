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

The free list hands blocks out first-in first-out.  Pinned by
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
        assert child not in self.tables and parent in self.tables
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = self.tokens[parent]
        for b in self.tables[child]:
            self.refs[b] += 1

    def append(self, seqs) -> tuple[list[int], list[tuple[int, int]]]:
        """One new token for each listed sequence, in order.  All or nothing."""
        assert len(set(seqs)) == len(seqs)
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
        for b in self.tables.pop(seq):
            self.refs[b] -= 1
            if self.refs[b] == 0:
                self.free.append(b)
        del self.tokens[seq]
