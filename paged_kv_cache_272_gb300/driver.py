"""Continuous-batching step driver: runs the native scheduler's steps on the GPU.

Each step the C++ scheduler (``serving.Scheduler``) decides which requests run and
reserves their slots; the driver copies the step's arrays to the device, forms the new
tokens' q/K/V there and launches the library's kernels on one stream:

    paged_block_copy        copy-on-write pairs (if any)
    paged_kv_write          K/V of every new token (decode tokens and prefill chunks)
    paged_attention_decode  the decode entries (one query token each)
    paged_attention_prefill the prefill chunks (causal, tensor cores)

There is no model: the new tokens' K/V rows and query rows are taken from fixed seeded
tables kept on the device (standing in for the layers that would produce them there);
a step copies only the row indices and gathers the rows on the device.  A token's K/V
depend only on its token id and position, so two requests with the same prompt prefix
hold the same K/V there and a cached prefix block is valid for both; a query row
depends on the request and position.  Output tokens get synthetic ids from (request,
position).
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import numpy as np
import torch

from . import ops
from .serving import Plan, Scheduler

BS = 16


def _i64(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.int64)  # no copy when already int64


def kv_row(token_ids: np.ndarray, positions: np.ndarray, rows: int) -> np.ndarray:
    """Row of the K/V tables for (token id, position)."""
    return (_i64(token_ids) * 1000003 + _i64(positions) * 7919) % rows


def q_row(rids: np.ndarray, positions: np.ndarray, rows: int) -> np.ndarray:
    return (_i64(rids) * 2654435761 + _i64(positions) * 40503) % rows


def output_token(rids: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """Synthetic id of the output token at a position (>= prompt length)."""
    return ((_i64(rids) * 7777 + _i64(positions) * 131) % 32000).astype(np.int32)


@dataclass
class StepInputs:
    """Host arrays of one step (everything the kernels read besides the caches)."""
    plan: Plan
    token_ids: np.ndarray      # int32 [T] ids of the new tokens, in slot order
    positions: np.ndarray      # int32 [T]
    kv_rows: np.ndarray        # int64 [T] rows of the K/V tables
    q_rows: np.ndarray         # int64 [T] rows of the query table
    num_decode: int
    decode_ctx_max: int
    prefill_query_start: np.ndarray  # int32 [n_prefill + 1], offsets within the prefill rows
    prefill_max_query: int


def prepare(plan: Plan, prompts: dict, kv_rows_n: int, q_rows_n: int,
            prompt_lens: np.ndarray | None = None) -> StepInputs:
    """Token ids, positions and table rows of a step's new tokens (host only).  Entry i
    covers positions context_lens[i] - query_lens[i] .. context_lens[i] - 1; a position
    inside the request's prompt takes the prompt's token, any later one a generated id.
    prompt_lens: optional array of prompt lengths indexed by request id (a faster lookup
    than the prompts dict when the ids are small integers)."""
    seq = _i64(plan.seq_ids)
    L = plan.query_lens.astype(np.int64)
    c = plan.context_lens.astype(np.int64)
    T = int(L.sum())
    first = c - L  # each entry's first new position
    starts = np.cumsum(L) - L
    rid_of = np.repeat(seq, L)
    pos = np.repeat(first - starts, L) + np.arange(T, dtype=np.int64)
    ids = output_token(rid_of, pos)
    if prompt_lens is not None:
        plen = prompt_lens[seq]
    else:
        plen = np.fromiter((len(prompts[r]) for r in seq.tolist()), dtype=np.int64,
                           count=len(seq))
    for i in np.flatnonzero(first < plen).tolist():  # entries that reach into their prompt
        lo, hi = int(first[i]), int(min(c[i], plen[i]))
        ids[starts[i]:starts[i] + hi - lo] = prompts[int(seq[i])][lo:hi]
    nd = plan.num_decode
    pq = plan.query_start[nd:] - plan.query_start[nd]
    return StepInputs(plan=plan, token_ids=ids, positions=pos.astype(np.int32),
                      kv_rows=kv_row(ids, pos, kv_rows_n), q_rows=q_row(rid_of, pos, q_rows_n),
                      num_decode=nd,
                      decode_ctx_max=int(plan.context_lens[:nd].max()) if nd else 0,
                      prefill_query_start=pq.astype(np.int32),
                      prefill_max_query=int(plan.query_lens[nd:].max()) if len(pq) > 1 else 0)


class ServingDriver:
    def __init__(self, sched: Scheduler, num_blocks: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, max_context: int, seed: int = 0, table_rows: int = 4096,
                 device="cuda", partition_size: int = 0):
        self.sched = sched
        self.Hq, self.Hkv, self.D = num_q_heads, num_kv_heads, head_dim
        self.dev = torch.device(device)
        self.scale = head_dim ** -0.5
        g = torch.Generator().manual_seed(seed)
        bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
        # tables (the "model"): K/V rows by (token, position), q rows by (request, pos);
        # host copies for checking, device copies for the steps
        self.k_tab, self.v_tab = bf(table_rows, num_kv_heads, head_dim), bf(table_rows, num_kv_heads, head_dim)
        self.q_tab = bf(table_rows, num_q_heads, head_dim)
        self.k_tab_d, self.v_tab_d, self.q_tab_d = (t.to(self.dev) for t in
                                                     (self.k_tab, self.v_tab, self.q_tab))
        self.rows = table_rows
        self.k_cache = torch.zeros(num_blocks, num_kv_heads, BS, head_dim, dtype=torch.bfloat16,
                                   device=self.dev)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.prompts: dict[int, np.ndarray] = {}
        self._plen: np.ndarray | None = np.zeros(1024, np.int64)
        self.max_context = max_context
        self.P = partition_size  # 0: each decode call picks its split on the device
        self.P_ws = partition_size if partition_size > 0 else 512  # the workspace's partitions
        self.ws = ops.alloc_workspace(sched.max_num_seqs, num_q_heads, head_dim, max_context,
                                      partition_size, device=self.dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.stream = torch.cuda.current_stream(self.dev)
        self.launches = 0
        self._bufs = {}
        self._dbufs = {}
        self._views = {}
        self._host = {}
        self.h2d_bytes = 0
        self.d2h_bytes = 0
        self.on_decode = None  # optional hook(0 before / 1 after) around decode attention
        self.on_start = None   # optional hook called before the step's first copy

    def add_request(self, rid: int, prompt, output_len: int) -> None:
        self.prompts[rid] = np.ascontiguousarray(prompt, dtype=np.int32)
        if self._plen is not None:  # prompt lengths by id while the ids are small
            if 0 <= rid < (1 << 20):
                if rid >= self._plen.shape[0]:
                    self._plen = np.concatenate(
                        [self._plen, np.zeros(max(rid + 1, 2 * self._plen.shape[0]) -
                                              self._plen.shape[0], np.int64)])
                self._plen[rid] = self.prompts[rid].shape[0]
            else:
                self._plen = None
        self.sched.add_request(rid, self.prompts[rid], output_len)

    def done(self) -> bool:
        return self.sched.done()

    def _pack(self, arrays, slot):
        """Stage host arrays [(name, numpy array, torch dtype)] in one pinned buffer of
        `slot`, each at a 256-byte aligned offset, so a step needs one host-to-device
        copy.  Returns (pinned bytes, device bytes, {name: (offset, shape, dtype)})."""
        layout, off = {}, 0
        for name, arr, dt in arrays:
            nb = arr.size * torch.empty(0, dtype=dt).element_size()
            layout[name] = (off, tuple(arr.shape), dt, nb)
            off += (nb + 255) & ~255
        total = max(off, 256)
        h = self._bufs.get(slot)
        if h is None or h.numel() < total:
            h = torch.empty(total * 2, dtype=torch.uint8).pin_memory()
            self._bufs[slot] = h
        d = self._dbufs.get("in")
        if d is None or d.numel() < total:
            d = torch.empty(total * 2, dtype=torch.uint8, device=self.dev)
            self._dbufs["in"] = d
        hn = h.numpy()
        for name, arr, dt in arrays:
            o, shape, _, nb = layout[name]
            np_dt = {torch.int64: np.int64, torch.int32: np.int32}[dt]
            hn[o:o + nb].view(np_dt)[:] = np.ascontiguousarray(arr, dtype=np_dt).ravel()
        return h[:total], d[:total], layout

    def _dev(self, name, shape, dtype):
        """A device buffer, grown on demand; returns a view of the requested shape (views
        are kept per shape until the buffer grows)."""
        v = self._views.get((name, shape))
        if v is not None:
            return v
        n = math.prod(shape)
        buf = self._dbufs.get(name)
        if buf is None or buf.numel() < n:
            buf = torch.empty(max(n, 1) * 2, dtype=dtype, device=self.dev)
            self._dbufs[name] = buf
            self._views = {k: t for k, t in self._views.items() if k[0] != name}
        if len(self._views) > 4096:
            self._views.clear()
        v = buf[:n].view(shape)
        self._views[(name, shape)] = v
        return v

    def fetch(self, *outs, slot=0):
        """Copy a step's outputs to pinned host memory (what a sampler would read), into
        the buffers of `slot` (so a step's outputs stay readable while the next step,
        using the other slot, runs)."""
        res = []
        for i, t in enumerate(outs):
            if t is None:
                res.append(None)
                continue
            n = t.numel()
            h = self._host.get((i, slot))
            if h is None or h.numel() < n:
                h = torch.empty(max(n, 1) * 2, dtype=t.dtype).pin_memory()
                self._host[(i, slot)] = h
            v = h[:n].view(t.shape)
            v.copy_(t, non_blocking=True)
            self.d2h_bytes += n * t.element_size()
            res.append(v)
        return res

    def plan_step(self, slot=0):
        """Host part of one step: the scheduler's plan, the new tokens' ids, positions and
        table rows, and the step's arrays in pinned staging buffers of `slot`.  Touches
        no device memory, so it may run while the previous step's kernels execute (use
        another slot than a step whose copies may still be pending).  Returns the staged
        step, or its inputs alone when the plan has no new token."""
        plan = self.sched.step()
        x = prepare(plan, self.prompts, self.rows, self.rows, self._plen)
        if x.token_ids.shape[0] == 0:
            return x, None
        arrays = [("kvr", x.kv_rows, torch.int64), ("qr", x.q_rows, torch.int64),
                  ("slots", plan.slot_mapping, torch.int64),
                  ("tables", plan.block_tables, torch.int32),
                  ("ctx", plan.context_lens, torch.int32)]
        if plan.cow_pairs.size:
            arrays.append(("pairs", plan.cow_pairs, torch.int32))
        if plan.seq_ids.shape[0] > x.num_decode:
            arrays.append(("pq", x.prefill_query_start, torch.int32))
        staged = self._pack(arrays, slot)
        return x, staged

    def launch_step(self, x, staged):
        """Device part of one step, queued on the stream: the copies of the staged arrays,
        the row gathers and the library's kernels.  Returns (decode_out, prefill_out)
        (device tensors; decode_out is [num_decode][Hq][D], prefill_out [tokens][Hq][D])."""
        if staged is None:
            return None, None
        plan = x.plan
        T = x.token_ids.shape[0]
        if self.on_start is not None:
            self.on_start()
        hbuf, dbuf, layout = staged
        dbuf.copy_(hbuf, non_blocking=True)
        self.h2d_bytes += hbuf.numel()
        typed = {torch.int64: (dbuf.view(torch.int64), 8), torch.int32: (dbuf.view(torch.int32), 4)}
        dv = {}
        for name, (o, shape, dt, nb) in layout.items():
            t, es = typed[dt]
            v = t[o // es:(o + nb) // es]
            dv[name] = v if len(shape) == 1 else v.view(shape)
        k_new = self._dev("k", (T, self.Hkv, self.D), torch.bfloat16)
        v_new = self._dev("v", (T, self.Hkv, self.D), torch.bfloat16)
        q = self._dev("q", (T, self.Hq, self.D), torch.bfloat16)
        torch.index_select(self.k_tab_d, 0, dv["kvr"], out=k_new)
        torch.index_select(self.v_tab_d, 0, dv["kvr"], out=v_new)
        torch.index_select(self.q_tab_d, 0, dv["qr"], out=q)
        slots, tables, ctx = dv["slots"], dv["tables"], dv["ctx"]
        if "pairs" in dv:
            ops.paged_block_copy(self.k_cache, self.v_cache, dv["pairs"], err_flag=self.err,
                                 stream=self.stream)
            self.launches += 1
        ops.paged_kv_write(k_new, v_new, slots, self.k_cache, self.v_cache, err_flag=self.err,
                           stream=self.stream)
        self.launches += 1
        nd = x.num_decode
        dec_out = pre_out = None
        if nd:
            dec_out = self._dev("dec_out", (nd, self.Hq, self.D), torch.bfloat16)
            if self.on_decode is not None:
                self.on_decode(0)
            ops.paged_attention_decode(dec_out, q[:nd], self.k_cache, self.v_cache, tables[:nd],
                                       ctx[:nd], self.scale, x.decode_ctx_max, self.ws, self.P,
                                       err_flag=self.err, stream=self.stream)
            if self.on_decode is not None:
                self.on_decode(1)
            self.launches += 3 if x.decode_ctx_max > self.P_ws else 2
        if plan.seq_ids.shape[0] > nd:
            pre_out = self._dev("pre_out", (T - nd, self.Hq, self.D), torch.bfloat16)
            ops.paged_attention_prefill(pre_out, q[nd:], self.k_cache, self.v_cache, tables[nd:],
                                        ctx[nd:], dv["pq"], self.scale, x.prefill_max_query,
                                        err_flag=self.err, stream=self.stream)
            self.launches += 1
        return dec_out, pre_out

    def step(self):
        """One scheduler step and its kernels: plan_step then launch_step.  Returns
        (inputs, decode_out, prefill_out).  The caller synchronises (or reads the
        outputs) before the next step reuses the staging buffers."""
        x, staged = self.plan_step()
        dec, pre = self.launch_step(x, staged)
        return x, dec, pre

    # ---- the packed path: the plan written straight into pinned staging by the native
    # scheduler (pkv_sched_pack) at fixed offsets, and the device half of each step
    # queued by one native call (pkv_step_launch) over buffers made once, sized for the
    # capacities --------------------------------------------------------------------
    def _fast_setup(self):
        from .serving import StepIO, StepPack
        self.f_tokens = self.sched.max_batched_tokens + self.sched.max_num_seqs
        self.f_seqs = self.sched.max_num_seqs
        self.f_stride = (self.max_context + BS - 1) // BS
        lay = StepPack()
        try:  # layout only (a NULL buffer is refused after the layout is filled)
            self.sched.pack(None, 0, self.f_tokens, self.f_seqs, self.f_stride, lay)
        except ops.PagedKVError:
            pass
        self.f_bytes = lay.total
        self.f_host = [torch.empty(self.f_bytes, dtype=torch.uint8).pin_memory()
                       for _ in range(2)]
        self.f_dev = torch.empty(self.f_bytes, dtype=torch.uint8, device=self.dev)
        self.f_packs = [StepPack(), StepPack()]
        T, S = self.f_tokens, self.f_seqs
        # the staging's context lengths, per slot (read by callers that count bytes)
        self.f_np = [h[lay.context_lens:lay.context_lens + 4 * S].view(torch.int32).numpy()
                     for h in self.f_host]
        self.f_knew = torch.empty(T, self.Hkv, self.D, dtype=torch.bfloat16, device=self.dev)
        self.f_vnew = torch.empty_like(self.f_knew)
        self.f_q = torch.empty(T, self.Hq, self.D, dtype=torch.bfloat16, device=self.dev)
        self.f_pre = torch.empty(T, self.Hq, self.D, dtype=torch.bfloat16, device=self.dev)
        # what a sampler reads, in one device buffer: the decode rows, then the last row
        # of each prefill chunk (copied to the host in one copy)
        self.f_out = torch.empty(S, self.Hq, self.D, dtype=torch.bfloat16, device=self.dev)
        self.f_out_h = [torch.empty(S, self.Hq, self.D, dtype=torch.bfloat16).pin_memory()
                        for _ in range(2)]
        self.f_row = self.Hq * self.D * 2  # bytes of one q / output row
        NB = self.k_cache.shape[0]
        io = StepIO()
        io.host_stage[0], io.host_stage[1] = (h.data_ptr() for h in self.f_host)
        io.dev_stage, io.stage_bytes = self.f_dev.data_ptr(), self.f_bytes
        io.k_table, io.v_table = self.k_tab_d.data_ptr(), self.v_tab_d.data_ptr()
        io.q_table, io.table_rows = self.q_tab_d.data_ptr(), self.rows
        io.k_new, io.v_new, io.q = (t.data_ptr() for t in (self.f_knew, self.f_vnew, self.f_q))
        io.prefill_out, io.out = self.f_pre.data_ptr(), self.f_out.data_ptr()
        io.out_host[0], io.out_host[1] = (h.data_ptr() for h in self.f_out_h)
        io.k_cache, io.v_cache = self.k_cache.data_ptr(), self.v_cache.data_ptr()
        io.max_tokens, io.max_seqs, io.num_blocks = T, S, NB
        io.num_q_heads, io.num_kv_heads, io.head_dim = self.Hq, self.Hkv, self.D
        io.block_size, io.table_stride, io.partition_size = BS, self.f_stride, self.P
        io.scale = self.scale
        io.workspace, io.workspace_bytes = self.ws.data_ptr(), self.ws.numel()
        io.err_flag = self.err.data_ptr()
        self.f_io = io
        self.f_io_ref = ctypes.byref(io)
        self.f_stream = ctypes.c_void_p(self.stream.cuda_stream)

    def plan_packed(self, slot=0):
        """Host part of one step on the packed path: the native scheduler steps, packs its
        plan into pinned staging buffer `slot` (fixed offsets) and fills in the synthetic
        model's generated token ids and table rows.  Returns the StepPack (counts and
        layout)."""
        if not hasattr(self, "f_host"):
            self._fast_setup()
        self.sched.step_only()
        pk = self.f_packs[slot]
        ptr = self.f_host[slot].data_ptr()
        self.sched.pack(ptr, self.f_bytes, self.f_tokens, self.f_seqs, self.f_stride, pk)
        if pk.num_tokens:
            ops.check(ops.lib.pkv_step_synthetic_rows(ptr, ctypes.byref(pk), self.rows),
                      "pkv_step_synthetic_rows")
        return pk

    def launch_packed(self, pk, slot=0, events=None):
        """Device part of a packed step, queued on the stream by one native call
        (pkv_step_launch): the copy of the packed plan, the synthetic model's row gathers,
        paged_decode_step (copies, write, decode attention), the prefill call, the
        gather of each chunk's last row and one copy of what a sampler reads (every
        decode row, the last row of every prefill chunk) into pinned buffers of `slot`.
        events: None or a ctypes array of three cudaEvent_t handles (each may be None)
        recorded before the first copy, before and after the decode step.  Returns
        (decode rows, prefill last rows) as host tensors, valid once the stream reaches
        this point."""
        T = pk.num_tokens
        if T == 0:
            return None, None
        ops.check(ops.lib.pkv_step_launch(self.f_io_ref, ctypes.byref(pk), slot, events,
                                          self.f_stream), "pkv_step_launch")
        return self._launched(pk, slot)

    def engine_step(self, slot=0, events=None):
        """One whole serving iteration in one native call (pkv_engine_step): the scheduler
        step, its pack into pinned staging `slot`, the synthetic model's rows and the
        device half of the step (see launch_packed).  Returns (pack, decode rows, prefill
        last rows); the rows are host tensors valid once the stream reaches this point,
        None when the step launched nothing (pack.num_tokens == 0)."""
        if not hasattr(self, "f_host"):
            self._fast_setup()
        pk = self.f_packs[slot]
        n = ops.lib.pkv_engine_step(self.sched._h, self.f_io_ref, ctypes.byref(pk), slot, events,
                                    self.f_stream)
        ops.check(min(n, 0), "pkv_engine_step")
        if pk.num_tokens == 0:
            return pk, None, None
        return (pk, *self._launched(pk, slot))

    def _launched(self, pk, slot):
        """Counts of a launched packed step; its host output views."""
        n, nd = pk.num_seqs, pk.num_decode
        self.h2d_bytes += pk.total
        self.d2h_bytes += n * self.f_row
        launches = 1  # the row gathers
        if nd:  # prologue (copies, write, plan), partition, merge if split, extra copies
            launches += 2 + (pk.decode_max_context > self.P_ws) + (pk.num_cow > 1024)
        else:  # no decode entry: the copies (if any) and the write alone
            launches += 1 + (pk.num_cow > 0)
        if n > nd:  # the prefill and its last-row gather
            launches += 2
        self.launches += launches
        out_h = self.f_out_h[slot]
        return (out_h[:nd] if nd else None), (out_h[nd:n] if n > nd else None)
