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
