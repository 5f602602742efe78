"""The plain-Python block manager against the pages' block-manager rules (CPU only)."""
import collections
import random

import pytest

from oracle.block_manager import BlockManager, BlockManagerError, OutOfBlocks

BS = 16


def check_invariants(bm: BlockManager):
    counts = collections.Counter()
    for seq, table in bm.tables.items():
        counts.update(table)
        n = bm.num_tokens[seq]
        assert len(table) == (n + BS - 1) // BS
        assert 0 <= bm.internal_waste(seq) < BS          # at most one partly filled block
    for b in range(bm.num_blocks):
        assert bm.refcount[b] == counts.get(b, 0)
    free = set(bm._free)
    assert len(free) == len(bm._free)
    assert free.isdisjoint(counts)
    assert len(free) + len(counts) == bm.num_blocks


def test_figure_requests_and_reuse():
    """Requests A (200 tokens) and B (150 tokens) take 13 and 10 blocks; when A
    finishes its blocks go straight to the next request C ("System-level
    optimization", section 2.3 figure)."""
    bm = BlockManager(40, BS)
    bm.add_seq(0)
    bm.add_seq(1)
    bm.append_tokens(0, 200)
    bm.append_tokens(1, 150)
    a_blocks = bm.block_table(0)
    assert len(a_blocks) == 13 and len(bm.block_table(1)) == 10
    assert set(a_blocks).isdisjoint(bm.block_table(1))
    bm.free_seq(0)
    bm.add_seq(2)
    bm.append_tokens(2, 200)
    assert bm.block_table(2) == a_blocks
    check_invariants(bm)


def test_block_table_non_contiguous():
    """Physical blocks need not be contiguous; the table restores the logical order
    ("Continuous batching and PagedAttention", section 3: A -> [7, 3, 15])."""
    order = [7, 3, 15, 2, 9] + [b for b in range(16) if b not in (7, 3, 15, 2, 9)]
    bm = BlockManager(16, BS, free_order=order)
    bm.add_seq("A")
    bm.append_tokens("A", 40)
    bm.add_seq("B")
    bm.append_tokens("B", 20)
    assert bm.block_table("A") == [7, 3, 15]
    assert bm.block_table("B") == [2, 9]
    assert bm.append_slot("A")[0] == 15 * BS + 40 % BS


def test_fork_and_copy_on_write():
    """Forked requests share blocks read-only; writing into a shared, partly filled
    block copies it first ("Continuous batching and PagedAttention", section 3,
    copy-on-write)."""
    bm = BlockManager(8, BS)
    bm.add_seq(0)
    bm.append_tokens(0, 20)               # blocks [0, 1], block 1 partly filled
    bm.fork(0, 1)
    assert bm.refcount[0] == 2 and bm.refcount[1] == 2
    slot, cow = bm.append_slot(1)
    assert cow == (1, 2)
    assert bm.block_table(1) == [0, 2] and slot == 2 * BS + 4
    assert bm.refcount[1] == 1 and bm.refcount[2] == 1 and bm.refcount[0] == 2
    slot, cow = bm.append_slot(0)         # parent now owns block 1 alone: no copy
    assert cow is None and slot == 1 * BS + 4
    check_invariants(bm)


def test_fork_full_block_needs_no_copy():
    bm = BlockManager(8, BS)
    bm.add_seq(0)
    bm.append_tokens(0, 32)
    bm.fork(0, 1)
    slot, cow = bm.append_slot(1)
    assert cow is None and bm.block_table(1)[:2] == bm.block_table(0)
    check_invariants(bm)


def test_shared_prefix_refcount():
    """50 requests sharing one system prompt store its blocks once with refcount 50."""
    bm = BlockManager(400, BS)
    bm.add_seq("p")
    bm.append_tokens("p", 2000)
    for i in range(50):
        bm.fork("p", i)
    bm.free_seq("p")
    prefix = bm.block_table(0)
    assert len(prefix) == 125
    assert all(bm.refcount[b] == 50 for b in prefix)
    assert bm.num_free() == 400 - 125
    check_invariants(bm)


def test_out_of_blocks_leaves_state():
    bm = BlockManager(3, BS)
    bm.add_seq(0)
    bm.append_tokens(0, 40)               # 3 blocks
    before = bm._snapshot()
    with pytest.raises(OutOfBlocks):
        bm.append_tokens(0, 9)
    assert bm._snapshot() == before
    bm.fork(0, 1)
    with pytest.raises(OutOfBlocks):      # COW needs a block too
        bm.append_slot(1)
    check_invariants(bm)


def test_errors():
    bm = BlockManager(4, BS)
    bm.add_seq(0)
    with pytest.raises(BlockManagerError):
        bm.add_seq(0)
    with pytest.raises(BlockManagerError):
        bm.append_slot(5)
    with pytest.raises(BlockManagerError):
        bm.fork(0, 0)
    with pytest.raises(BlockManagerError):
        bm.free_seq(9)
    with pytest.raises(BlockManagerError):
        BlockManager(4, BS, free_order=[0, 1, 1, 2])


def test_random_ops_keep_invariants():
    rng = random.Random(7)
    bm = BlockManager(64, BS, free_order=rng.sample(range(64), 64))
    live = []
    next_id = 0
    for _ in range(3000):
        op = rng.random()
        try:
            if op < 0.15 or not live:
                bm.add_seq(next_id)
                live.append(next_id)
                next_id += 1
            elif op < 0.75:
                bm.append_tokens(rng.choice(live), rng.randint(1, 20))
            elif op < 0.85:
                bm.fork(rng.choice(live), next_id)
                live.append(next_id)
                next_id += 1
            else:
                s = rng.choice(live)
                bm.free_seq(s)
                live.remove(s)
        except OutOfBlocks:
            s = rng.choice(live)
            bm.free_seq(s)
            live.remove(s)
        check_invariants(bm)
