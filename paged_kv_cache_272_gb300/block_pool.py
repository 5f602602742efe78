"""Python handle on the native host block manager (``pkv_pool_*`` / ``pkv_seq_*`` in
``include/pagedkv.h``).  Marshalling only; the allocator is the C++ code."""
from __future__ import annotations

import ctypes

import numpy as np

from .ops import PagedKVError, check, lib

ERR_OOM = -10


class OutOfBlocks(PagedKVError):
    pass


def _chk(code, what):
    if code == ERR_OOM:
        raise OutOfBlocks(code, what)
    check(code, what)


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class BlockPool:
    """A pool of ``num_blocks`` fixed-size KV blocks with per-sequence block tables,
    reference counts, fork and copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int = 16, free_order=None):
        h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("free_order must hold num_blocks entries")
        _chk(lib.pkv_pool_create(num_blocks, block_size, None if order is None else _p(order),
                                 ctypes.byref(h)), "pkv_pool_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def retain(self, block: int) -> None:
        """One more holder of an allocated block (as a prefix cache takes)."""
        _chk(lib.pkv_block_retain(self._h, block), "pkv_block_retain")

    def release(self, block: int) -> None:
        """One holder fewer; the block returns to the pool with its last holder."""
        _chk(lib.pkv_block_release(self._h, block), "pkv_block_release")

    def save(self) -> bytes:
        """A snapshot of the pool's state (free order, refcounts, tables, lengths)."""
        n = lib.pkv_pool_save(self._h, None, 0)
        _chk(min(int(n), 0), "pkv_pool_save")
        buf = ctypes.create_string_buffer(int(n))
        _chk(min(int(lib.pkv_pool_save(self._h, buf, n)), 0), "pkv_pool_save")
        return buf.raw

    @classmethod
    def load(cls, data: bytes) -> "BlockPool":
        """A new pool in the state a snapshot from save() recorded."""
        h = ctypes.c_void_p()
        buf = ctypes.create_string_buffer(bytes(data), len(data))
        _chk(lib.pkv_pool_load(buf, len(data), ctypes.byref(h)), "pkv_pool_load")
        self = cls.__new__(cls)
        self._h = h
        self.num_blocks = int.from_bytes(data[8:16], "little")
        self.block_size = int.from_bytes(data[16:24], "little")
        return self

    def close(self):
        if self._h:
            lib.pkv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return lib.pkv_pool_num_free(self._h)

    def refcount(self, block: int) -> int:
        r = lib.pkv_block_refcount(self._h, block)
        _chk(min(r, 0), "pkv_block_refcount")
        return r

    def add_seq(self, seq: int) -> None:
        _chk(lib.pkv_seq_add(self._h, seq), "pkv_seq_add")

    def fork(self, parent: int, child: int) -> None:
        _chk(lib.pkv_seq_fork(self._h, parent, child), "pkv_seq_fork")

    def free_seq(self, seq: int) -> None:
        _chk(lib.pkv_seq_free(self._h, seq), "pkv_seq_free")

    def num_tokens(self, seq: int) -> int:
        n = ctypes.c_int()
        _chk(lib.pkv_seq_num_tokens(self._h, seq, ctypes.byref(n)), "pkv_seq_num_tokens")
        return n.value

    def num_seq_blocks(self, seq: int) -> int:
        n = ctypes.c_int()
        _chk(lib.pkv_seq_num_blocks(self._h, seq, ctypes.byref(n)), "pkv_seq_num_blocks")
        return n.value

    def append_slot(self, seq: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _chk(lib.pkv_seq_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                     ctypes.byref(dst)), "pkv_seq_append_slot")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def append_tokens(self, seq: int, count: int):
        slots = np.empty(max(count, 1), np.int64)
        pairs = np.empty((max(count, 1), 2), np.int32)
        n = ctypes.c_int()
        _chk(lib.pkv_seq_append_tokens(self._h, seq, count, _p(slots), _p(pairs),
                                       ctypes.byref(n)), "pkv_seq_append_tokens")
        return slots[:count], pairs[:n.value]

    def step(self, seqs):
        """One decode step: a slot per listed sequence.  Returns (slot_mapping int64[n],
        cow_pairs int32[P][2])."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        n = seqs.shape[0]
        slots = np.empty(max(n, 1), np.int64)
        pairs = np.empty((max(n, 1), 2), np.int32)
        ncow = ctypes.c_int()
        _chk(lib.pkv_pool_step(self._h, _p(seqs), n, _p(slots), _p(pairs), ctypes.byref(ncow)),
             "pkv_pool_step")
        return slots[:n], pairs[:ncow.value]

    def export(self, seqs, max_blocks: int, pad: int = -1):
        """(block_tables int32[n][max_blocks], context_lens int32[n])."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        n = seqs.shape[0]
        tables = np.empty((max(n, 1), max_blocks), np.int32)
        lens = np.empty(max(n, 1), np.int32)
        _chk(lib.pkv_pool_export(self._h, _p(seqs), n, max_blocks, pad, _p(tables), _p(lens)),
             "pkv_pool_export")
        return tables[:n], lens[:n]

    def block_table(self, seq: int):
        nb = self.num_seq_blocks(seq)
        t, _ = self.export([seq], max(nb, 1))
        return t[0, :nb].tolist()
