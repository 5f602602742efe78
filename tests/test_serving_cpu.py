"""Continuous-batching scheduler and prefix cache (host code, CPU only).

* The plain-Python references (``oracle/scheduler.py``, ``oracle/prefix_trie.py``)
  against what the pages state: slot fill above 80% under continuous batching with
  Pareto output lengths ("Inference optimization", exercise 2), prefix-cache hit rate
  above 55% for 1000 requests of which 60% share 5 prefixes with at most 500 LRU
  entries (exercise 4), near-zero KV waste with paging ("Inference optimization",
  PagedAttention), continuous batching ahead of static batching ("Continuous batching
  and PagedAttention", section 2) -- plus conservation invariants and brute force.
* The C++ scheduler and cache against those references, step by step.
"""
import numpy as np
import pytest

from oracle.block_manager import BlockManager
from oracle.prefix_trie import PrefixTrie
from oracle.scheduler import Scheduler as RefScheduler
from paged_kv_cache_272_gb300 import workloads

BS = 16


def ref_run(reqs, num_blocks, max_seqs, budget, static=False, cache_entries=None,
            free_order=None, max_steps=200000):
    bm = BlockManager(num_blocks, BS, free_order=free_order)
    cache = PrefixTrie(bm, cache_entries) if cache_entries is not None else None
    s = RefScheduler(bm, max_seqs, budget, static=static, cache=cache)
    for r in reqs:
        s.add_request(r.rid, r.prompt.tolist(), r.output_len)
    plans = []
    while not s.done():
        plans.append(s.step())
        assert len(plans) < max_steps
    return s, bm, cache, plans


# -------------------------------------------------------------------------------------
# Pins of the references
# -------------------------------------------------------------------------------------
def test_exercise2_continuous_fill_above_80_percent():
    reqs = workloads.make_requests("pareto", seed=1)
    cont, bm, _, _ = ref_run(reqs, 4000, 8, 512)
    stat, _, _, _ = ref_run(reqs, 4000, 8, 512, static=True)
    assert cont.finished == stat.finished == len(reqs)
    assert cont.busy_fill_sum / cont.busy_steps > 0.80
    assert cont.fill_sum / cont.steps > stat.fill_sum / stat.steps
    assert cont.steps < stat.steps                     # more tokens per step
    assert bm.num_free() == bm.num_blocks              # nothing leaked


def test_outputs_and_prompts_are_conserved():
    """Without preemption or caching every request computes its prompt once and writes
    the K/V of all its outputs but the last."""
    reqs = workloads.make_requests("pareto", seed=2, n=40)
    s, _, _, plans = ref_run(reqs, 4000, 6, 300)
    assert s.preemptions == 0
    assert s.prefill_tokens == sum(len(r.prompt) for r in reqs)
    assert s.decode_tokens == sum(r.output_len - 1 for r in reqs)
    # a request's tokens appear at consecutive positions, each position once
    seen = {}
    for p in plans:
        for rid, q, c in zip(p.seqs, p.query_lens, p.context_lens):
            seen.setdefault(rid, []).append((c - q, c))
    for r in reqs:
        spans = seen[r.rid]
        assert spans[0][0] == 0 and all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        assert spans[-1][1] == len(r.prompt) + r.output_len - 1


def test_waste_is_below_one_block_per_request():
    reqs = workloads.make_requests("pareto", seed=3)
    s, _, _, _ = ref_run(reqs, 4000, 8, 512)
    frac = s.slots_unused / s.slots_held
    assert frac < 0.05  # the pages quote about 4% with paging
    # each running request wastes at most block_size - 1 slots per step
    assert s.slots_unused <= (BS - 1) * s.fill_sum * 8 + 1e-9


def test_budget_and_slots_are_respected():
    reqs = workloads.make_requests("pareto", seed=4, n=60)
    s, _, _, plans = ref_run(reqs, 4000, 5, 64)
    for p in plans:
        assert sum(p.query_lens) <= 64
        assert len(p.seqs) <= 5
        assert all(q == 1 for q in p.query_lens[:p.num_decode])


def test_preemption_under_block_pressure_completes_everything():
    reqs = workloads.make_requests("pareto", seed=5, n=30)
    s, bm, _, plans = ref_run(reqs, 40, 8, 128)
    assert s.preemptions > 0
    assert s.finished == len(reqs)
    assert bm.num_free() == bm.num_blocks


def test_pool_too_small_is_reported():
    from oracle.block_manager import BlockManagerError
    reqs = [workloads.Request(0, np.arange(100, dtype=np.int32), 5)]
    with pytest.raises(BlockManagerError):
        ref_run(reqs, 4, 2, 256)


def test_exercise4_prefix_hit_rate_above_55_percent():
    reqs = workloads.make_requests("shared-prefix", seed=6)
    s, bm, cache, _ = ref_run(reqs, 8000, 32, 2048, cache_entries=500)
    assert cache.lookups == len(reqs)
    assert cache.hits / cache.lookups > 0.55
    assert len(cache.entries) <= 500
    # prefill work saved = matched tokens
    assert s.prefill_tokens == sum(len(r.prompt) for r in reqs) - cache.matched_tokens


def test_trie_lookup_equals_brute_force_longest_prefix():
    rng = np.random.default_rng(7)
    bm = BlockManager(400)
    trie = PrefixTrie(bm, 10 ** 6)
    base = rng.integers(0, 5, 160).tolist()       # few symbols: many shared prefixes
    prompts = []
    for i in range(40):
        cut = int(rng.integers(0, 160))
        p = base[:cut] + rng.integers(0, 5, int(rng.integers(1, 80))).tolist()
        bm.add_seq(i)
        bm.append_tokens(i, len(p))
        trie.insert(p, bm.block_table(i))
        prompts.append(p)
    for q in prompts + [base, base[:33], [9] * 40]:
        want = 0
        for p in prompts:          # longest common full-block prefix with any inserted
            k = 0
            while (k + 1) * BS <= min(len(p), len(q)) and p[:(k + 1) * BS] == q[:(k + 1) * BS]:
                k += 1
            want = max(want, k)
        assert len(trie.lookup(q)) == min(want, (len(q) - 1) // BS)


def test_trie_lru_evicts_least_recent_leaf_first():
    bm = BlockManager(64)
    trie = PrefixTrie(bm, 3)
    a = list(range(48))             # three full blocks: a chain of three entries
    bm.add_seq(0)
    bm.append_tokens(0, 48)
    trie.insert(a, bm.block_table(0))
    b = list(range(100, 132))       # two more entries: over the limit of 3
    bm.add_seq(1)
    bm.append_tokens(1, 32)
    trie.insert(b, bm.block_table(1))
    # the leaves were a's third block (older) and b's second block; the older goes
    # first, then a's second block (now a leaf), leaving a[0], b[0], b[1]
    assert set(len(k) for k in trie.entries) == {16, 32}
    assert tuple(a[:16]) in trie.entries and tuple(b[:32]) in trie.entries
    assert tuple(a[:32]) not in trie.entries


# -------------------------------------------------------------------------------------
# The C++ scheduler and cache against the references
# -------------------------------------------------------------------------------------
def native_run(reqs, num_blocks, max_seqs, budget, static=False, cache_entries=None,
               free_order=None):
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.serving import PrefixCache, Scheduler
    pool = BlockPool(num_blocks, BS, free_order=free_order)
    cache = PrefixCache(pool, cache_entries) if cache_entries is not None else None
    s = Scheduler(pool, max_seqs, budget, static=static, cache=cache)
    for r in reqs:
        s.add_request(r.rid, r.prompt, r.output_len)
    plans = []
    while not s.done():
        plans.append(s.step())
    return s, pool, cache, plans


CASES = {
    "continuous": dict(kind="pareto", n=50, blocks=4000, seqs=8, budget=512),
    "static": dict(kind="pareto", n=50, blocks=4000, seqs=8, budget=512, static=True),
    "small-budget": dict(kind="pareto", n=40, blocks=4000, seqs=6, budget=40),
    "preemption": dict(kind="pareto", n=30, blocks=40, seqs=8, budget=128),
    "prefix-cache": dict(kind="shared-prefix", n=300, blocks=3000, seqs=16, budget=1024,
                         cache=100),
    "prefix-cache-pressure": dict(kind="shared-prefix", n=200, blocks=120, seqs=8,
                                  budget=512, cache=60),
}


@pytest.mark.parametrize("name", list(CASES))
def test_native_scheduler_matches_reference(name):
    c = CASES[name]
    reqs = workloads.make_requests(c["kind"], seed=11, n=c["n"])
    order = np.random.default_rng(12).permutation(c["blocks"])
    ref, bm, rcache, rplans = ref_run(reqs, c["blocks"], c["seqs"], c["budget"],
                                      c.get("static", False), c.get("cache"), order)
    nat, pool, ncache, nplans = native_run(reqs, c["blocks"], c["seqs"], c["budget"],
                                           c.get("static", False), c.get("cache"), order)
    assert len(nplans) == len(rplans)
    for i, (a, b) in enumerate(zip(nplans, rplans)):
        assert a.seq_ids.tolist() == b.seqs, i
        assert a.num_decode == b.num_decode, i
        assert a.query_lens.tolist() == b.query_lens, i
        assert a.context_lens.tolist() == b.context_lens, i
        assert a.slot_mapping.tolist() == b.slots, i
        assert a.query_start.tolist() == [0] + np.cumsum(b.query_lens).tolist(), i
        assert [tuple(x) for x in a.cow_pairs.tolist()] == [tuple(x) for x in b.cow_pairs], i
        assert (a.finished, a.preempted) == (b.finished, b.preempted), i
        for row, rid in zip(a.block_tables, a.seq_ids):
            t = bm.tables.get(int(rid))
            if t is not None and b is rplans[-1]:
                assert row[:len(t)].tolist() == t
    st = nat.stats()
    assert st["steps"] == ref.steps and st["finished"] == ref.finished
    assert st["preemptions"] == ref.preemptions
    assert st["decode_tokens"] == ref.decode_tokens
    assert st["prefill_tokens"] == ref.prefill_tokens
    assert st["slots_held"] == ref.slots_held and st["slots_unused"] == ref.slots_unused
    assert st["busy_steps"] == ref.busy_steps
    assert abs(st["fill_sum"] - ref.fill_sum) < 1e-9
    if rcache is not None:
        cs = ncache.stats()
        assert (cs["lookups"], cs["hits"], cs["matched_tokens"], cs["evictions"]) == (
            rcache.lookups, rcache.hits, rcache.matched_tokens, rcache.evictions)
        assert cs["entries"] == len(rcache.entries)
    assert pool.num_free() + (ncache.stats()["entries"] if ncache else 0) >= 0


def test_native_block_tables_match_reference_each_step():
    """The exported tables of every step equal the reference pool's tables then."""
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.serving import PrefixCache, Scheduler
    reqs = workloads.make_requests("shared-prefix", seed=13, n=120)
    bm = BlockManager(400)
    rs = RefScheduler(bm, 8, 256, cache=PrefixTrie(bm, 50))
    pool = BlockPool(400)
    ns = Scheduler(pool, 8, 256, cache=PrefixCache(pool, 50))
    for r in reqs:
        rs.add_request(r.rid, r.prompt.tolist(), r.output_len)
        ns.add_request(r.rid, r.prompt, r.output_len)
    while not rs.done():
        b = rs.step()
        a = ns.step()
        for row, rid in zip(a.block_tables, a.seq_ids):
            t = bm.tables[int(rid)]
            assert row[:len(t)].tolist() == t and (row[len(t):] == -1).all()
    assert ns.done()


def test_native_cache_api_matches_reference():
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.serving import PrefixCache
    rng = np.random.default_rng(14)
    bm, pool = BlockManager(200), BlockPool(200)
    trie, cache = PrefixTrie(bm, 12), PrefixCache(pool, 12)
    base = rng.integers(0, 3, 128).tolist()
    for i in range(30):
        p = base[:int(rng.integers(0, 128))] + rng.integers(0, 3, int(rng.integers(1, 60))).tolist()
        assert cache.lookup(p) == trie.lookup(p)
        m = trie.lookup(p)
        trie.use(p, len(m))
        cache.use(p, len(m))
        bm.add_seq(i)
        bm.append_tokens(i, len(p))
        pool.add_seq(i)
        pool.append_tokens(i, len(p))
        trie.insert(p, bm.block_table(i))
        cache.insert(p, pool.block_table(i))
        if i % 3 == 2:
            bm.free_seq(i - 1)
            pool.free_seq(i - 1)
            assert cache.evict_free_one() == trie.evict_free_one()
        assert pool.num_free() == bm.num_free()
        assert cache.stats()["entries"] == len(trie.entries)


@pytest.mark.parametrize("num_blocks", [2000, 40])
def test_driver_step_inputs_follow_the_plan(num_blocks):
    """The driver's host preparation: prompt tokens for prefill chunks, synthetic output
    tokens for decode entries, K/V rows that depend only on (token, position); with a
    small pool requests are preempted and prefilled again from the start."""
    from paged_kv_cache_272_gb300 import driver
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.serving import Scheduler
    reqs = workloads.make_requests("pareto", seed=15, n=10)
    pool = BlockPool(num_blocks)
    s = Scheduler(pool, 4, 64)
    prompts = {}
    for r in reqs:
        prompts[r.rid] = r.prompt
        s.add_request(r.rid, r.prompt, r.output_len)
    plen = np.zeros(max(prompts) + 1, np.int64)  # the driver's lookup by request id
    for rid, pr in prompts.items():
        plen[rid] = len(pr)
    while not s.done():
        plan = s.step()
        x = driver.prepare(plan, prompts, 4096, 4096)
        y = driver.prepare(plan, prompts, 4096, 4096, plen)
        for f in ("token_ids", "positions", "kv_rows", "q_rows", "prefill_query_start"):
            assert np.array_equal(getattr(x, f), getattr(y, f)), f
        assert x.token_ids.shape[0] == plan.slot_mapping.shape[0]
        for i, rid in enumerate(plan.seq_ids.tolist()):
            a, b = int(plan.query_start[i]), int(plan.query_start[i + 1])
            c, L = int(plan.context_lens[i]), int(plan.query_lens[i])
            assert x.positions[a:b].tolist() == list(range(c - L, c))
            P = len(prompts[rid])
            if i < plan.num_decode:
                assert L == 1 and c - 1 >= P
                assert x.token_ids[a] == driver.output_token(np.array([rid]), np.array([c - 1]))[0]
            else:
                pos = np.arange(c - L, c)
                want = [int(prompts[rid][p]) if p < P else
                        int(driver.output_token(np.array([rid]), np.array([p]))[0]) for p in pos]
                assert x.token_ids[a:b].tolist() == want
        nd = plan.num_decode
        assert x.prefill_query_start.tolist() == (plan.query_start[nd:] - plan.query_start[nd]).tolist()
        assert (x.kv_rows == driver.kv_row(x.token_ids, x.positions, 4096)).all()
    if num_blocks == 40:
        assert s.stats()["preemptions"] > 0


@pytest.mark.parametrize("kind,num_blocks", [("pareto", 2000), ("pareto", 40),
                                             ("shared-prefix", 3000)])
def test_native_pack_equals_the_host_preparation(kind, num_blocks):
    """pkv_sched_pack writes, at fixed offsets, exactly what the driver's numpy
    preparation derives from a plan: slots, tables (padded with -1), context lengths,
    copy pairs, chunk offsets and last rows, and per new token the request id, the
    position and the prompt token (-1 past the prompt, where the synthetic sampler's id
    goes); plus the step's maxima and its output-token count."""
    import ctypes
    from paged_kv_cache_272_gb300 import driver
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.serving import PrefixCache, Scheduler, StepPack
    reqs = workloads.make_requests(kind, seed=21, n=40)
    pool = BlockPool(num_blocks)
    cache = PrefixCache(pool, 256) if kind == "shared-prefix" else None
    s = Scheduler(pool, 8, 96, cache=cache)
    prompts = {}
    for r in reqs:
        prompts[r.rid] = np.ascontiguousarray(r.prompt, dtype=np.int32)
        s.add_request(r.rid, prompts[r.rid], r.output_len)
    maxT, maxS, stride = 96 + 8, 8, 200
    pk = StepPack()
    buf = (ctypes.c_uint8 * (1 << 20))()
    base = ctypes.addressof(buf)
    raw = np.frombuffer(buf, dtype=np.uint8)
    view = lambda off, n, dt: raw[off:off + n * np.dtype(dt).itemsize].view(dt)
    steps = outputs = 0
    while not s.done():
        plan = s.step()
        s.pack(base, len(buf), maxT, maxS, stride, pk)
        x = driver.prepare(plan, prompts, 4096, 4096)
        T, n, nd = pk.num_tokens, pk.num_seqs, pk.num_decode
        assert (T, n, nd, pk.num_cow) == (plan.slot_mapping.shape[0], plan.seq_ids.shape[0],
                                          plan.num_decode, plan.cow_pairs.shape[0])
        assert np.array_equal(view(pk.slot_mapping, T, np.int64), plan.slot_mapping)
        tb = view(pk.block_tables, n * stride, np.int32).reshape(n, stride)
        mb = plan.block_tables.shape[1]
        assert np.array_equal(tb[:, :mb], plan.block_tables) and (tb[:, mb:] == -1).all()
        assert np.array_equal(view(pk.context_lens, n, np.int32), plan.context_lens)
        assert np.array_equal(view(pk.cow_pairs, 2 * pk.num_cow, np.int32).reshape(-1, 2),
                              plan.cow_pairs)
        assert np.array_equal(view(pk.positions, T, np.int32), x.positions)
        rid = view(pk.token_seq, T, np.int64)
        assert np.array_equal(rid, np.repeat(plan.seq_ids, plan.query_lens))
        tok = view(pk.token_ids, T, np.int32).copy()
        gen = tok < 0
        tok[gen] = driver.output_token(rid[gen], x.positions[gen])
        assert np.array_equal(tok, x.token_ids)
        # the synthetic model's ids and table rows, natively, equal the driver's numpy ones
        from paged_kv_cache_272_gb300 import ops
        ops.check(ops.lib.pkv_step_synthetic_rows(base, ctypes.byref(pk), 4096), "rows")
        assert np.array_equal(view(pk.token_ids, T, np.int32), x.token_ids)
        assert np.array_equal(view(pk.kv_rows, T, np.int64), x.kv_rows)
        assert np.array_equal(view(pk.q_rows, T, np.int64), x.q_rows)
        ch = n - nd
        if ch:
            assert np.array_equal(view(pk.prefill_start, ch + 1, np.int32),
                                  x.prefill_query_start)
            assert np.array_equal(view(pk.last_rows, ch, np.int64),
                                  x.prefill_query_start[1:].astype(np.int64) - 1)
        assert pk.prefill_max_query == x.prefill_max_query
        assert pk.decode_max_context == x.decode_ctx_max
        want = nd + sum(1 for i in range(nd, n)
                        if plan.context_lens[i] == len(prompts[int(plan.seq_ids[i])]))
        assert pk.outputs == want
        steps += 1
        outputs += pk.outputs
    assert steps > 10
    if s.stats()["preemptions"] == 0:  # (a recomputed request's outputs count again)
        assert outputs == sum(r.output_len for r in reqs)
    # a capacity below the step's needs is refused
    pool2 = BlockPool(2000)
    s2 = Scheduler(pool2, 8, 96)
    for r in reqs[:8]:
        s2.add_request(r.rid, prompts[r.rid], r.output_len)
    s2.step()
    with pytest.raises(Exception):
        s2.pack(base, len(buf), 4, maxS, stride)
    with pytest.raises(Exception):
        s2.pack(base, 16, maxT, maxS, stride)


@pytest.mark.parametrize("seed", range(12))
def test_native_scheduler_fuzz(seed):
    """Random pools, slot counts, budgets, cache sizes and request mixes (including pools
    small enough to force preemption and cache eviction): the native scheduler takes
    the reference's decisions at every step."""
    rng = np.random.default_rng(100 + seed)
    kind = "shared-prefix" if seed % 2 else "pareto"
    reqs = workloads.make_requests(kind, seed=200 + seed, n=int(rng.integers(10, 60)))
    for r in reqs:
        r.output_len = int(min(r.output_len, rng.integers(1, 200)))
    seqs = int(rng.integers(1, 12))
    budget = int(rng.integers(seqs, 600))
    need = max((len(r.prompt) + r.output_len + 15) // 16 for r in reqs)
    blocks = int(rng.integers(need + 1, need * 6))
    cache = int(rng.integers(0, 200)) if kind == "shared-prefix" else None
    static = bool(seed % 3 == 0)
    order = rng.permutation(blocks)
    ref, bm, rcache, rplans = ref_run(reqs, blocks, seqs, budget, static, cache, order)
    nat, pool, ncache, nplans = native_run(reqs, blocks, seqs, budget, static, cache, order)
    assert len(nplans) == len(rplans)
    for a, b in zip(nplans, rplans):
        assert a.seq_ids.tolist() == b.seqs
        assert a.slot_mapping.tolist() == b.slots
        assert a.context_lens.tolist() == b.context_lens
        assert (a.finished, a.preempted) == (b.finished, b.preempted)
    st = nat.stats()
    assert (st["preemptions"], st["finished"]) == (ref.preemptions, ref.finished)
    assert ref.finished == len(reqs)
    if rcache is not None:
        assert ncache.stats()["evictions"] == rcache.evictions


def test_native_serving_api_rejects_bad_arguments():
    import ctypes
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.ops import lib
    from paged_kv_cache_272_gb300.serving import PrefixCache, Scheduler
    ERR_NULL, ERR_ARG, ERR_DUP = -1, -14, -12
    h = ctypes.c_void_p()
    assert lib.pkv_pcache_create(None, 4, ctypes.byref(h)) == ERR_NULL
    pool = BlockPool(8)
    assert lib.pkv_pcache_create(pool._h, -1, ctypes.byref(h)) == ERR_ARG
    assert lib.pkv_sched_create(pool._h, None, 0, 16, 0, ctypes.byref(h)) == ERR_ARG
    assert lib.pkv_sched_create(pool._h, None, 8, 4, 0, ctypes.byref(h)) == ERR_ARG  # budget < slots
    other = BlockPool(8)
    c_other = PrefixCache(other, 4)
    assert lib.pkv_sched_create(pool._h, c_other._h, 2, 16, 0, ctypes.byref(h)) == ERR_ARG
    s = Scheduler(pool, 2, 16)
    assert lib.pkv_sched_add_request(s._h, 1, 0, None, 3) == ERR_ARG      # empty prompt
    assert lib.pkv_sched_add_request(s._h, 1, 4, None, 0) == ERR_ARG      # no output token
    assert lib.pkv_sched_add_request(s._h, 1, 4, None, 3) == 0
    assert lib.pkv_sched_add_request(s._h, 1, 4, None, 3) == ERR_DUP
    # a cached block must be allocated; a table too short for the prompt is refused
    cache = PrefixCache(pool, 4)
    toks = np.arange(32, dtype=np.int32)
    table = np.array([0], dtype=np.int32)
    assert lib.pkv_pcache_insert(cache._h, toks.ctypes.data, 32, table.ctypes.data, 1) == ERR_ARG
    assert lib.pkv_block_retain(pool._h, 3) == ERR_ARG   # free block
    assert lib.pkv_block_release(pool._h, 99) == ERR_ARG
    assert lib.pkv_seq_add_shared(pool._h, 5, table.ctypes.data, 1) == ERR_ARG  # block 0 free


def test_pool_too_small_native():
    from paged_kv_cache_272_gb300.block_pool import BlockPool, OutOfBlocks
    from paged_kv_cache_272_gb300.serving import Scheduler
    pool = BlockPool(4)
    s = Scheduler(pool, 2, 256)
    s.add_request(0, np.arange(100, dtype=np.int32), 5)
    with pytest.raises(OutOfBlocks):
        while not s.done():
            s.step()


def test_scheduler_plans_pass_the_slot_check():
    """Every step's slot mapping from the native scheduler is in range and race free."""
    from paged_kv_cache_272_gb300 import ops
    reqs = workloads.make_requests("shared-prefix", seed=31, n=80)
    nat, pool, cache, plans = native_run(reqs, 300, 8, 256, cache_entries=40)
    for p in plans:
        ops.paged_kv_check_slots(p.slot_mapping, 300)


def test_driver_prompt_length_table_grows_and_falls_back():
    """The driver's prompt-length table (request id -> length) grows past its first
    size, and ids it cannot index (negative, huge) switch it off in favour of the
    prompts dict (logic only: a stand-in object, no device)."""
    from types import SimpleNamespace
    from paged_kv_cache_272_gb300 import driver
    added = []
    fake = SimpleNamespace(prompts={}, _plen=np.zeros(4, np.int64),
                           sched=SimpleNamespace(add_request=lambda *a: added.append(a[0])))
    for rid, n in ((0, 5), (3, 7), (9, 2), (40, 11)):
        driver.ServingDriver.add_request(fake, rid, np.arange(n), 3)
    assert fake._plen.shape[0] >= 41
    assert [int(fake._plen[r]) for r in (0, 3, 9, 40)] == [5, 7, 2, 11]
    assert int(fake._plen[1]) == 0 and added == [0, 3, 9, 40]
    driver.ServingDriver.add_request(fake, 1 << 40, np.arange(3), 3)
    assert fake._plen is None and len(fake.prompts[1 << 40]) == 3
    driver.ServingDriver.add_request(fake, 5, np.arange(6), 3)  # stays off
    assert fake._plen is None
