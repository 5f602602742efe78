"""The continuous-batching driver on the GPU: every step's decode and prefill outputs
against the fp64 oracle run on a host copy of the cache that receives the same
copy-on-write pairs and K/V writes (|err| <= 1e-2 + 1e-2 |ref|, mean <= 2e-3)."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
from paged_kv_cache_272_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _steps(drv, overlap):
    """(inputs, decode_out, prefill_out) of every step, in order.  Without overlap the
    host waits for each step before the next; with overlap it keeps two steps in flight
    as the serving benchmark does (step k + 1 planned and queued before step k's outputs,
    read back into the other slot's pinned buffers, are waited for)."""
    if not overlap:
        while not drv.done():
            x, dec, pre = drv.step()
            torch.cuda.synchronize()
            yield x, dec, pre
        return
    slot, pending = 0, []
    while not drv.done():
        x, staged = drv.plan_step(slot)
        if staged is None:
            continue
        dec, pre = drv.launch_step(x, staged)
        hd, hp = drv.fetch(dec, pre, slot=slot)
        ev = torch.cuda.Event()
        ev.record()
        pending.append((x, hd, hp, ev))
        slot ^= 1
        if len(pending) == 2:
            x0, hd0, hp0, ev0 = pending.pop(0)
            ev0.synchronize()
            yield x0, hd0, hp0
    for x0, hd0, hp0, ev0 in pending:
        ev0.synchronize()
        yield x0, hd0, hp0


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("cache_entries,blocks", [(None, 400), (40, 400), (30, 60)])
def test_driver_steps_match_oracle(cache_entries, blocks, overlap):
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.driver import ServingDriver
    from paged_kv_cache_272_gb300.serving import PrefixCache, Scheduler
    Hq, Hkv, D = 8, 2, 128
    reqs = workloads.make_requests("shared-prefix", seed=21, n=24)
    for r in reqs:
        r.output_len = min(r.output_len, 40)
    pool = BlockPool(blocks)
    cache = PrefixCache(pool, cache_entries) if cache_entries else None
    sched = Scheduler(pool, 6, 96, cache=cache)
    max_ctx = max(len(r.prompt) + r.output_len for r in reqs)
    drv = ServingDriver(sched, blocks, Hq, Hkv, D, max_ctx, seed=3)
    for r in reqs:
        drv.add_request(r.rid, r.prompt, r.output_len)
    kh = np.zeros((blocks, Hkv, 16, D), np.uint16)
    vh = np.zeros_like(kh)
    steps = 0
    for x, dec, pre in _steps(drv, overlap):
        steps += 1
        p = x.plan
        if x.token_ids.shape[0] == 0:
            continue
        if p.cow_pairs.size:
            oracle.block_copy(kh, vh, p.cow_pairs)
        oracle.kv_write(kh, vh, u16(drv.k_tab[torch.from_numpy(x.kv_rows)]),
                        u16(drv.v_tab[torch.from_numpy(x.kv_rows)]), p.slot_mapping)
        q = u16(drv.q_tab[torch.from_numpy(x.q_rows)])
        nd = x.num_decode
        if nd:
            ref = oracle.attention(q[:nd], kh, vh, p.block_tables[:nd], p.context_lens[:nd],
                                   drv.scale, nthreads=H.NTHREADS)
            H.assert_attention_close(dec, ref, f"decode step {steps}")
        if p.seq_ids.shape[0] > nd:
            ref = oracle.attention_prefill(q[nd:], kh, vh, p.block_tables[nd:],
                                           p.context_lens[nd:], x.prefill_query_start,
                                           drv.scale, nthreads=H.NTHREADS)
            H.assert_attention_close(pre, ref, f"prefill step {steps}")
    assert int(drv.err.item()) == 0
    assert sched.stats()["finished"] == len(reqs)
    # the device cache equals the host replica for every block the host wrote
    assert np.array_equal(u16(drv.k_cache.cpu()), kh) and np.array_equal(u16(drv.v_cache.cpu()), vh)
    if cache is not None:
        assert cache.stats()["hits"] > 0


@pytest.mark.parametrize("engine", [False, True])
@pytest.mark.parametrize("cache_entries,blocks", [(None, 400), (30, 60)])
def test_packed_path_equals_the_checked_path(cache_entries, blocks, engine):
    """The packed serving path (native pack into pinned staging, fused decode step, two
    steps in flight; its device half in one native call, or the whole iteration in one,
    pkv_engine_step) gives, step by step, the same bits as the path checked against the
    oracle above: every decode row, the last row of every prefill chunk, and the caches."""
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.driver import ServingDriver
    from paged_kv_cache_272_gb300.serving import PrefixCache, Scheduler
    Hq, Hkv, D = 8, 2, 128
    reqs = workloads.make_requests("shared-prefix", seed=22, n=24)
    for r in reqs:
        r.output_len = min(r.output_len, 40)
    max_ctx = max(len(r.prompt) + r.output_len for r in reqs)

    def make():
        pool = BlockPool(blocks)
        cache = PrefixCache(pool, cache_entries) if cache_entries else None
        drv = ServingDriver(Scheduler(pool, 6, 96, cache=cache), blocks, Hq, Hkv, D, max_ctx,
                            seed=3)
        for r in reqs:
            drv.add_request(r.rid, r.prompt, r.output_len)
        return drv

    ref = []
    a = make()
    for x, dec, pre in _steps(a, overlap=False):
        if x.token_ids.shape[0] == 0:
            continue
        last = (pre[torch.as_tensor(x.prefill_query_start[1:].astype(np.int64) - 1,
                                    device=pre.device)].cpu() if pre is not None else None)
        ref.append((dec.cpu() if dec is not None else None, last))
    b = make()
    got, slot, pending = [], 0, []
    while not b.done():
        if engine:  # one native call per step
            pk, hd, hl = b.engine_step(slot)
            if pk.num_tokens == 0:
                continue
        else:
            pk = b.plan_packed(slot)
            if pk.num_tokens == 0:
                continue
            hd, hl = b.launch_packed(pk, slot)
        ev = torch.cuda.Event()
        ev.record()
        pending.append((hd, hl, ev))
        slot ^= 1
        if len(pending) == 2:
            hd0, hl0, ev0 = pending.pop(0)
            ev0.synchronize()
            got.append((None if hd0 is None else hd0.clone(), None if hl0 is None else hl0.clone()))
    for hd0, hl0, ev0 in pending:
        ev0.synchronize()
        got.append((None if hd0 is None else hd0.clone(), None if hl0 is None else hl0.clone()))
    assert len(got) == len(ref)
    for k, ((rd, rl), (gd, gl)) in enumerate(zip(ref, got)):
        for r_, g_, what in ((rd, gd, "decode"), (rl, gl, "prefill last rows")):
            assert (r_ is None) == (g_ is None), (k, what)
            if r_ is not None:
                assert torch.equal(r_.view(torch.int16), g_.view(torch.int16)), (k, what)
    assert int(a.err.item()) == 0 and int(b.err.item()) == 0
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))


def test_gather_rows_bit_exact_and_flags_bad_rows():
    """paged_gather_rows moves whole rows bit for bit; a row index outside the table sets
    PKV_DEV_BAD_ROW and leaves that destination row as it was."""
    from paged_kv_cache_272_gb300 import ops
    g = torch.Generator().manual_seed(9)
    src = torch.randint(-32768, 32767, (300, 8, 128), generator=g, dtype=torch.int16)
    idx = torch.randint(0, 300, (517,), generator=g)
    idx[5], idx[9] = 300, -1
    dst = torch.zeros(517, 8, 128, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_gather_rows(dst, src.cuda().view(torch.bfloat16), idx.cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == ops.DEV_BAD_ROW
    ok = torch.ones(517, dtype=torch.bool)
    ok[5] = ok[9] = False
    got = dst.cpu().view(torch.int16)
    assert torch.equal(got[ok], src[idx[ok]])
    assert (got[~ok] == 0).all()
    # a one-row table, 16-byte rows, and nothing to gather
    one = torch.arange(8, dtype=torch.int16).reshape(1, 8)
    d1 = torch.zeros(3, 8, dtype=torch.int16, device="cuda")
    ops.paged_gather_rows(d1, one.cuda(), torch.zeros(3, dtype=torch.int64, device="cuda"))
    ops.paged_gather_rows(d1, one.cuda(), torch.zeros(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(d1.cpu(), one.expand(3, 8))


def test_engine_step_records_its_events():
    """pkv_engine_step records the caller's events (before the staging copy, around the
    decode step) on the stream, in order, and records none for a step with no tokens."""
    import ctypes
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.driver import ServingDriver
    from paged_kv_cache_272_gb300.serving import Scheduler
    reqs = workloads.make_requests("pareto", seed=23, n=6)
    pool = BlockPool(200)
    drv = ServingDriver(Scheduler(pool, 4, 64), 200, 8, 2, 128,
                        max(len(r.prompt) + min(r.output_len, 12) for r in reqs), seed=4)
    for r in reqs:
        drv.add_request(r.rid, r.prompt, min(r.output_len, 12))
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:
        e.record(stream)  # creates the events
    stream.synchronize()
    handles = (ctypes.c_void_p * 3)(ev[0].cuda_event, ev[1].cuda_event, ev[2].cuda_event)
    timed = 0
    slot = 0
    while not drv.done():
        pk, hd, hl = drv.engine_step(slot, handles)
        if pk.num_tokens == 0:
            continue
        ev[3].record(stream)
        ev[3].synchronize()
        t_all = ev[0].elapsed_time(ev[3])
        t_dec = ev[1].elapsed_time(ev[2])
        assert 0.0 < t_dec <= t_all and ev[0].elapsed_time(ev[1]) >= 0.0
        timed += 1
        slot ^= 1
    assert timed > 3 and int(drv.err.item()) == 0
