"""Python binding of the host-side KV block manager in libpa.so
(include/pa_block_manager.h).  Argument marshalling only."""
from __future__ import annotations

import ctypes

import numpy as np

from . import _native as N


class BlockManager:
    """Free list, reference counts, fork / append / free and copy-on-write pairs
    for a pool of ``num_blocks`` blocks of ``block_size`` tokens."""

    def __init__(self, num_blocks: int, block_size: int, alloc_order=None):
        self._lib = N.load()
        order = None
        if alloc_order is not None:
            order = np.ascontiguousarray(alloc_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("alloc_order must list every block once")
        ptr = None if order is None else order.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        self._h = self._lib.pa_bm_create(num_blocks, block_size, ptr)
        if not self._h:
            raise ValueError("invalid block manager arguments")
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    __del__ = close

    def add_sequence(self, seq_id: int, num_tokens: int) -> np.ndarray:
        slots = np.zeros(max(num_tokens, 1), dtype=np.int64)
        N.check("pa_bm_add_sequence", self._lib.pa_bm_add_sequence(
            self._h, seq_id, num_tokens, slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
        return slots[:num_tokens]

    def fork(self, parent_id: int, child_id: int) -> None:
        N.check("pa_bm_fork", self._lib.pa_bm_fork(self._h, parent_id, child_id))

    def append(self, seq_ids) -> tuple[np.ndarray, np.ndarray]:
        """One new token per sequence: returns (slots [n] int64, copy pairs [p, 2] int64)."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        slots = np.zeros(max(n, 1), dtype=np.int64)
        pairs = np.zeros(max(2 * n, 2), dtype=np.int64)
        npairs = ctypes.c_int32(0)
        i64 = ctypes.POINTER(ctypes.c_int64)
        N.check("pa_bm_append", self._lib.pa_bm_append(
            self._h, ids.ctypes.data_as(i64), n, slots.ctypes.data_as(i64),
            pairs.ctypes.data_as(i64), ctypes.byref(npairs)))
        return slots[:n], pairs[:2 * npairs.value].reshape(-1, 2)

    def free(self, seq_id: int) -> None:
        N.check("pa_bm_free", self._lib.pa_bm_free(self._h, seq_id))

    def block_tables(self, seq_ids, stride: int) -> tuple[np.ndarray, np.ndarray]:
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        table = np.zeros((max(n, 1), stride), dtype=np.int32)
        lens = np.zeros(max(n, 1), dtype=np.int32)
        N.check("pa_bm_block_tables", self._lib.pa_bm_block_tables(
            self._h, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
            table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), stride,
            lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return table[:n], lens[:n]

    def num_free_blocks(self) -> int:
        return int(self._lib.pa_bm_num_free_blocks(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._lib.pa_bm_ref_count(self._h, block))

    def num_tokens(self, seq_id: int) -> int:
        return int(self._lib.pa_bm_num_tokens(self._h, seq_id))

    # -------------------------------------------------------------------- swapping
    def set_cpu_pool(self, num_cpu_blocks: int) -> None:
        """A CPU pool of ``num_cpu_blocks`` blocks for swapped-out sequence groups."""
        N.check("pa_bm_set_cpu_pool", self._lib.pa_bm_set_cpu_pool(self._h, num_cpu_blocks))
        self.num_cpu_blocks = num_cpu_blocks

    def _swap(self, fn, seq_ids) -> np.ndarray:
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        cap = max(1, max(self.num_blocks, getattr(self, "num_cpu_blocks", 0)))
        pairs = np.zeros(2 * cap, dtype=np.int64)
        npairs = ctypes.c_int32(0)
        i64 = ctypes.POINTER(ctypes.c_int64)
        N.check(fn, getattr(self._lib, fn)(self._h, ids.ctypes.data_as(i64), n,
                                            pairs.ctypes.data_as(i64), cap, ctypes.byref(npairs)))
        return pairs[:2 * npairs.value].reshape(-1, 2)

    def swap_out(self, seq_ids) -> np.ndarray:
        """Moves a sequence group to the CPU pool; returns (gpu block, cpu block) pairs
        for pa_swap_blocks (GPU pools -> CPU pools)."""
        return self._swap("pa_bm_swap_out", seq_ids)

    def swap_in(self, seq_ids) -> np.ndarray:
        """Brings a swapped-out group back; returns (cpu block, gpu block) pairs for
        pa_swap_blocks (CPU pools -> GPU pools)."""
        return self._swap("pa_bm_swap_in", seq_ids)

    def num_free_cpu_blocks(self) -> int:
        return int(self._lib.pa_bm_num_free_cpu_blocks(self._h))

    def cpu_ref_count(self, block: int) -> int:
        return int(self._lib.pa_bm_cpu_ref_count(self._h, block))

    def is_swapped(self, seq_id: int) -> bool:
        r = int(self._lib.pa_bm_is_swapped(self._h, seq_id))
        if r < 0:
            raise KeyError(seq_id)
        return bool(r)
