"""Python handle on the native prefix cache and continuous-batching scheduler
(``pkv_pcache_*`` / ``pkv_sched_*`` in ``include/pagedkv.h``).  Marshalling only: the
trie, the LRU policy and the scheduling decisions are the C++ code."""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from .block_pool import BlockPool, _chk, _p
from .ops import lib

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


class StepPlan(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int), ("num_decode", ctypes.c_int),
                ("num_tokens", ctypes.c_int), ("max_blocks", ctypes.c_int),
                ("num_cow", ctypes.c_int), ("finished", ctypes.c_int),
                ("preempted", ctypes.c_int), ("running", ctypes.c_int),
                ("waiting", ctypes.c_int), ("seq_ids", _i64p), ("query_lens", _i32p),
                ("context_lens", _i32p), ("query_start", _i32p), ("slot_mapping", _i64p),
                ("block_tables", _i32p), ("cow_pairs", _i32p)]


class StepPack(ctypes.Structure):
    """Layout and counts of a packed step (pkv_step_pack): byte offsets of the arrays in
    the staging buffer, and the step's sizes."""
    _fields_ = [("slot_mapping", ctypes.c_int64), ("token_seq", ctypes.c_int64),
                ("last_rows", ctypes.c_int64), ("block_tables", ctypes.c_int64),
                ("context_lens", ctypes.c_int64), ("cow_pairs", ctypes.c_int64),
                ("prefill_start", ctypes.c_int64), ("token_ids", ctypes.c_int64),
                ("positions", ctypes.c_int64), ("kv_rows", ctypes.c_int64),
                ("q_rows", ctypes.c_int64), ("total", ctypes.c_int64),
                ("num_seqs", ctypes.c_int), ("num_decode", ctypes.c_int),
                ("num_tokens", ctypes.c_int), ("num_cow", ctypes.c_int),
                ("decode_max_context", ctypes.c_int), ("prefill_max_query", ctypes.c_int),
                ("outputs", ctypes.c_int)]


class StepIO(ctypes.Structure):
    """Buffers and constants of the device half of a packed step (pkv_step_io)."""
    _P = ctypes.c_void_p
    _fields_ = [("host_stage", _P * 2), ("dev_stage", _P), ("stage_bytes", ctypes.c_int64),
                ("k_table", _P), ("v_table", _P), ("q_table", _P),
                ("table_rows", ctypes.c_int64), ("k_new", _P), ("v_new", _P), ("q", _P),
                ("prefill_out", _P), ("out", _P), ("out_host", _P * 2), ("k_cache", _P),
                ("v_cache", _P), ("max_tokens", ctypes.c_int), ("max_seqs", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("num_q_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("block_size", ctypes.c_int), ("table_stride", ctypes.c_int),
                ("partition_size", ctypes.c_int), ("scale", ctypes.c_float),
                ("workspace", _P), ("workspace_bytes", ctypes.c_size_t), ("err_flag", _P)]


class SchedStats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("finished", ctypes.c_int64),
                ("preemptions", ctypes.c_int64), ("decode_tokens", ctypes.c_int64),
                ("prefill_tokens", ctypes.c_int64), ("busy_steps", ctypes.c_int64),
                ("fill_sum", ctypes.c_double), ("busy_fill_sum", ctypes.c_double),
                ("slots_held", ctypes.c_int64), ("slots_unused", ctypes.c_int64)]


def _arr(ptr, n, dtype):
    """A numpy copy of n elements at a C array (one memmove)."""
    a = np.empty(max(n, 0), dtype)
    if n > 0:
        ctypes.memmove(a.ctypes.data, ptr, a.nbytes)
    return a


@dataclass
class Plan:
    """One step's work (copies of the scheduler's arrays)."""
    seq_ids: np.ndarray        # int64 [n], decode entries first
    num_decode: int
    query_lens: np.ndarray     # int32 [n]
    context_lens: np.ndarray   # int32 [n]
    query_start: np.ndarray    # int32 [n+1]
    slot_mapping: np.ndarray   # int64 [tokens]
    block_tables: np.ndarray   # int32 [n][max_blocks]
    cow_pairs: np.ndarray      # int32 [c][2]
    finished: int
    preempted: int
    running: int
    waiting: int


class PrefixCache:
    def __init__(self, pool: BlockPool, max_entries: int):
        h = ctypes.c_void_p()
        _chk(lib.pkv_pcache_create(pool._h, max_entries, ctypes.byref(h)), "pkv_pcache_create")
        self._h, self.pool = h, pool

    def close(self):
        if self._h:
            lib.pkv_pcache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def lookup(self, tokens) -> list[int]:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(max(1, t.shape[0] // self.pool.block_size), np.int32)
        n = lib.pkv_pcache_lookup(self._h, _p(t), t.shape[0], _p(out), out.shape[0])
        _chk(min(n, 0), "pkv_pcache_lookup")
        return out[:n].tolist()

    def use(self, tokens, num_matched: int) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _chk(lib.pkv_pcache_use(self._h, _p(t), t.shape[0], num_matched), "pkv_pcache_use")

    def insert(self, tokens, table) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        tb = np.ascontiguousarray(table, dtype=np.int32)
        _chk(lib.pkv_pcache_insert(self._h, _p(t), t.shape[0], _p(tb), tb.shape[0]),
             "pkv_pcache_insert")

    def evict_free_one(self) -> bool:
        r = lib.pkv_pcache_evict_free_one(self._h)
        _chk(min(r, 0), "pkv_pcache_evict_free_one")
        return r == 1

    def stats(self) -> dict:
        out = np.zeros(6, np.int64)
        _chk(lib.pkv_pcache_stats(self._h, _p(out)), "pkv_pcache_stats")
        keys = ("lookups", "hits", "query_tokens", "matched_tokens", "entries", "evictions")
        return dict(zip(keys, (int(x) for x in out)))


class Scheduler:
    """Continuous (or static) batching over a BlockPool, optionally with a PrefixCache."""

    def __init__(self, pool: BlockPool, max_num_seqs: int, max_batched_tokens: int,
                 static: bool = False, cache: PrefixCache | None = None):
        h = ctypes.c_void_p()
        _chk(lib.pkv_sched_create(pool._h, cache._h if cache is not None else None,
                                  max_num_seqs, max_batched_tokens, int(static),
                                  ctypes.byref(h)), "pkv_sched_create")
        self._h, self.pool, self.cache = h, pool, cache
        self.max_num_seqs = max_num_seqs
        self.max_batched_tokens = max_batched_tokens
        self._pl = StepPlan()

    def close(self):
        if self._h:
            lib.pkv_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_request(self, rid: int, prompt, output_len: int, use_tokens: bool = True) -> None:
        t = np.ascontiguousarray(prompt, dtype=np.int32)
        _chk(lib.pkv_sched_add_request(self._h, rid, t.shape[0], _p(t) if use_tokens else None,
                                       output_len), "pkv_sched_add_request")

    def done(self) -> bool:
        return lib.pkv_sched_done(self._h) == 1

    def step(self) -> Plan:
        pl = StepPlan()
        n = lib.pkv_sched_step(self._h, ctypes.byref(pl))
        _chk(min(n, 0), "pkv_sched_step")
        tables = _arr(pl.block_tables, pl.num_seqs * pl.max_blocks, np.int32)
        return Plan(seq_ids=_arr(pl.seq_ids, pl.num_seqs, np.int64), num_decode=pl.num_decode,
                    query_lens=_arr(pl.query_lens, pl.num_seqs, np.int32),
                    context_lens=_arr(pl.context_lens, pl.num_seqs, np.int32),
                    query_start=_arr(pl.query_start, pl.num_seqs + 1, np.int32),
                    slot_mapping=_arr(pl.slot_mapping, pl.num_tokens, np.int64),
                    block_tables=tables.reshape(pl.num_seqs, pl.max_blocks),
                    cow_pairs=_arr(pl.cow_pairs, 2 * pl.num_cow, np.int32).reshape(-1, 2),
                    finished=pl.finished, preempted=pl.preempted, running=pl.running,
                    waiting=pl.waiting)

    def step_only(self) -> int:
        """Run one step without copying its plan out (see pack); returns the number of
        scheduled sequences."""
        n = lib.pkv_sched_step(self._h, ctypes.byref(self._pl))
        _chk(min(n, 0), "pkv_sched_step")
        return n

    def pack(self, buf_ptr: int, buf_bytes: int, max_tokens: int, max_seqs: int,
             table_stride: int, out: StepPack | None = None) -> StepPack:
        """Write the last step's plan into host memory at buf_ptr (pkv_sched_pack)."""
        pk = out if out is not None else StepPack()
        _chk(lib.pkv_sched_pack(self._h, buf_ptr, buf_bytes, max_tokens, max_seqs,
                                table_stride, ctypes.byref(pk)), "pkv_sched_pack")
        return pk

    def stats(self) -> dict:
        s = SchedStats()
        _chk(lib.pkv_sched_get_stats(self._h, ctypes.byref(s)), "pkv_sched_get_stats")
        return {f: getattr(s, f) for f, _ in SchedStats._fields_}
