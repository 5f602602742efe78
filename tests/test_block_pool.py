"""The native block manager against the plain-Python reference: identical block
tables, slots, copy-on-write pairs, refcounts and errors on seeded operation
sequences (CPU only)."""
import random

import numpy as np
import pytest

from oracle.block_manager import BlockManager, OutOfBlocks as RefOOM, BlockManagerError
from paged_kv_cache_272_gb300.block_pool import BlockPool, OutOfBlocks
from paged_kv_cache_272_gb300.ops import PagedKVError

BS = 16


def same_state(ref: BlockManager, pool: BlockPool, live):
    assert pool.num_free() == ref.num_free()
    for b in range(ref.num_blocks):
        assert pool.refcount(b) == ref.refcount[b]
    for s in live:
        assert pool.block_table(s) == ref.block_table(s)
        assert pool.num_tokens(s) == ref.num_tokens[s]
    if live:
        mb = max(len(ref.block_table(s)) for s in live) + 2
        t_ref, l_ref = ref.export(live, mb)
        t, l = pool.export(live, mb)
        assert t.tolist() == t_ref and l.tolist() == l_ref


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_operations_match_reference(seed):
    rng = random.Random(seed)
    nb = rng.choice([8, 40, 200])
    order = rng.sample(range(nb), nb)
    ref = BlockManager(nb, BS, free_order=order)
    pool = BlockPool(nb, BS, free_order=order)
    live, nid = [], 0
    for _ in range(1500):
        op = rng.random()
        if op < 0.12 or not live:
            ref.add_seq(nid)
            pool.add_seq(nid)
            live.append(nid)
            nid += 1
        elif op < 0.45:
            s, c = rng.choice(live), rng.randint(0, 40)
            try:
                want = ref.append_tokens(s, c)
            except RefOOM:
                with pytest.raises(OutOfBlocks):
                    pool.append_tokens(s, c)
            else:
                slots, pairs = pool.append_tokens(s, c)
                assert slots.tolist() == want[0]
                assert [tuple(p) for p in pairs.tolist()] == want[1]
        elif op < 0.70:
            batch = [rng.choice(live) for _ in range(rng.randint(1, 6))]
            try:
                want = ref.step(batch)
            except RefOOM:
                with pytest.raises(OutOfBlocks):
                    pool.step(batch)
            else:
                slots, pairs = pool.step(batch)
                assert slots.tolist() == want[0]
                assert [tuple(p) for p in pairs.tolist()] == want[1]
        elif op < 0.80:
            s = rng.choice(live)
            try:
                want = ref.append_slot(s)
            except RefOOM:
                with pytest.raises(OutOfBlocks):
                    pool.append_slot(s)
            else:
                assert pool.append_slot(s) == want
        elif op < 0.90:
            p = rng.choice(live)
            ref.fork(p, nid)
            pool.fork(p, nid)
            live.append(nid)
            nid += 1
        else:
            s = rng.choice(live)
            ref.free_seq(s)
            pool.free_seq(s)
            live.remove(s)
        same_state(ref, pool, live)


def test_errors_match():
    pool = BlockPool(4, BS)
    pool.add_seq(1)
    with pytest.raises(PagedKVError):
        pool.add_seq(1)
    with pytest.raises(PagedKVError):
        pool.append_slot(2)
    with pytest.raises(PagedKVError):
        pool.fork(9, 10)
    with pytest.raises(PagedKVError):
        pool.free_seq(3)
    with pytest.raises(PagedKVError):
        BlockPool(4, BS, free_order=[0, 0, 1, 2])
    with pytest.raises(PagedKVError):
        pool.refcount(4)


def test_step_with_shared_last_block():
    """Two forks share a partly filled block: the first to append copies it, the
    second then owns the original alone and appends in place."""
    order = list(range(10))
    ref = BlockManager(10, BS, free_order=order)
    pool = BlockPool(10, BS, free_order=order)
    for m in (ref, pool):
        m.add_seq(0)
        m.append_tokens(0, 20)
        m.fork(0, 1)
        m.fork(0, 2)
    want = ref.step([1, 2, 0, 1])
    slots, pairs = pool.step([1, 2, 0, 1])
    assert slots.tolist() == want[0]
    assert [tuple(p) for p in pairs.tolist()] == want[1]
    assert len(want[1]) == 2
    same_state(ref, pool, [0, 1, 2])


def test_step_oom_is_atomic():
    ref = BlockManager(3, BS)
    pool = BlockPool(3, BS)
    for m in (ref, pool):
        m.add_seq(0)
        m.append_tokens(0, 16)
        m.add_seq(1)
        m.append_tokens(1, 16)
    with pytest.raises(RefOOM):
        ref.step([0, 1])
    with pytest.raises(OutOfBlocks):
        pool.step([0, 1])
    same_state(ref, pool, [0, 1])


# -------------------------------------------------------------------------------------
# Snapshot (checkpoint / resume) of the native pool
# -------------------------------------------------------------------------------------
def _random_op(rng, pool, live, nid):
    """One random operation; returns (what happened, next id).  Out-of-blocks is an
    outcome like any other."""
    op = rng.random()
    try:
        if op < 0.12 or not live:
            pool.add_seq(nid)
            live.append(nid)
            return ("add", nid), nid + 1
        if op < 0.45:
            s, c = rng.choice(live), rng.randint(0, 40)
            slots, pairs = pool.append_tokens(s, c)
            return ("append", slots.tolist(), pairs.tolist()), nid
        if op < 0.70:
            slots, pairs = pool.step([rng.choice(live) for _ in range(rng.randint(1, 6))])
            return ("step", slots.tolist(), pairs.tolist()), nid
        if op < 0.80:
            return ("slot", pool.append_slot(rng.choice(live))), nid
        if op < 0.88:
            pool.fork(rng.choice(live), nid)
            live.append(nid)
            return ("fork", nid), nid + 1
        if op < 0.93:  # an extra holder, as a prefix cache takes
            s = rng.choice(live)
            t = pool.block_table(s)
            if t:
                pool.retain(t[0])
            return ("retain", t[:1]), nid
        s = rng.choice(live)
        pool.free_seq(s)
        live.remove(s)
        return ("free", s), nid
    except OutOfBlocks:
        return ("oom",), nid


def _state(pool, live):
    return (pool.num_free(), [pool.refcount(b) for b in range(pool.num_blocks)],
            {s: (pool.block_table(s), pool.num_tokens(s)) for s in live})


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_snapshot_resumes_identically(seed):
    """A pool rebuilt from a snapshot at random points answers every later operation
    exactly as the original does, and snapshots itself to the same bytes."""
    rng = random.Random(100 + seed)
    nb = rng.choice([12, 60, 300])
    pool = BlockPool(nb, BS, free_order=rng.sample(range(nb), nb))
    live, nid = [], 0
    for round_ in range(6):
        for _ in range(rng.randint(50, 250)):
            _, nid = _random_op(rng, pool, live, nid)
        snap = pool.save()
        copy = BlockPool.load(snap)
        assert copy.save() == snap
        assert (copy.num_blocks, copy.block_size) == (nb, BS)
        assert _state(copy, live) == _state(pool, live)
        r1, r2 = random.Random(seed * 7 + round_), random.Random(seed * 7 + round_)
        live1, live2, n1, n2 = list(live), list(live), nid, nid
        for _ in range(200):
            a, n1 = _random_op(r1, pool, live1, n1)
            b, n2 = _random_op(r2, copy, live2, n2)
            assert a == b
        assert live1 == live2 and _state(copy, live2) == _state(pool, live1)
        live, nid = live1, n1
        copy.close()


def test_snapshot_rejects_inconsistent_bytes():
    pool = BlockPool(10, BS)
    pool.add_seq(1)
    pool.append_tokens(1, 20)  # two blocks
    pool.fork(1, 2)
    snap = bytearray(pool.save())
    w = np.frombuffer(bytes(snap), dtype="<i8").copy()
    nfree = int(w[3])
    ref_at = 4 + nfree  # the refcounts
    seq_at = ref_at + 10 + 1  # first sequence record
    table0 = int(w[seq_at + 3])

    def bad(words):
        with pytest.raises(PagedKVError):
            BlockPool.load(np.asarray(words, dtype="<i8").tobytes())

    bad(w[:-1])                                   # truncated
    bad(np.concatenate([w, [0]]))                 # trailing word
    x = w.copy(); x[0] ^= 1; bad(x)               # magic
    x = w.copy(); x[1] = 0; bad(x)                # no blocks
    x = w.copy(); x[4] = x[5]; bad(x)             # a block twice on the free stack
    x = w.copy(); x[ref_at + table0] = 1; bad(x)  # refcount below the two tables' uses
    x = w.copy(); x[ref_at + int(w[4])] = 1; bad(x)  # a free block with a holder
    x = w.copy(); x[seq_at + 3] = 99; bad(x)      # table entry out of range
    x = w.copy(); x[seq_at + 3] = w[4]; bad(x)    # a free block in a table
    x = w.copy(); x[seq_at + 1] = 40; bad(x)      # length does not match the table
    with pytest.raises(PagedKVError):
        BlockPool.load(bytes(snap[:20]))          # shorter than the header
    # counts the buffer cannot hold are refused before anything is allocated for them
    bad([w[0], 2**31 - 1, BS, 0, 0])              # INT32_MAX blocks in a 40-byte buffer
    bad([w[0], 2**31 - 1, BS, 2**31 - 1, 0])      # ... and as many free blocks
    x = w.copy(); x[3] = 10; bad(x)               # a free stack that runs past the buffer
    # a token count near INT64_MAX (its block count would overflow) is refused
    x = w.copy(); x[seq_at + 1] = 2**63 - 1; bad(x)
    x = w.copy(); x[seq_at + 1] = 10 * BS + 1; bad(x)  # more tokens than the pool holds
