"""Plain-Python reference of the host block manager (test infrastructure only).

It restates the pages' block manager as directly as possible:

* The KV cache is cut into fixed-size blocks (usually 16 tokens), all the same size,
  handed out on demand from one global pool by a single block manager; a request's
  blocks need not be contiguous ("System-level optimization: batching, PagedAttention
  and FlashAttention", section 2.3 PagedAttention solution; "Continuous batching and
  PagedAttention", section 3 PagedAttention).
* Each request owns a block table mapping its logical block i to a physical block
  (same sections; "Request A's block table: [7, 3, 15]").
* Blocks a finished request releases can be reused by the next request at once
  (section 2.3 figure: A's pages are freed and C reuses them).
* Blocks are reference counted; several requests may share read-only blocks (prefix
  sharing, parallel sampling), and a private copy is made only when a request writes
  into a shared block -- copy-on-write ("Continuous batching and PagedAttention",
  section 3, copy-on-write sharing).
* Internal waste is at most one partly filled block per request (section 3, effects).

Readings where the pages are silent (each fixed so two implementations can be
compared exactly):

* Allocation order: the free pool is a stack.  It starts as ``free_order`` with its
  first element handed out first; a freed block is pushed on top, so the most
  recently freed block is the next one handed out.
* ``free_seq`` releases a request's blocks from its last logical block to its first,
  so a new request's logical block 0 lands on the freed request's old block 0.
* A slot is ``physical_block * block_size + offset``.
* A copy-on-write happens only inside ``append_slot``, when the block that the new
  token falls in has refcount > 1; the new block takes the table entry and the old
  block's refcount drops by one.
* Every failing call leaves the state unchanged.
"""
from __future__ import annotations


class BlockManagerError(RuntimeError):
    pass


class OutOfBlocks(BlockManagerError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise BlockManagerError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise BlockManagerError("free_order must be a permutation of range(num_blocks)")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self._free = list(reversed(order))  # top of stack = end of list
        self.refcount = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.num_tokens: dict[int, int] = {}

    # -- pool ---------------------------------------------------------------------
    def num_free(self) -> int:
        return len(self._free)

    def _alloc(self) -> int:
        if not self._free:
            raise OutOfBlocks("block pool exhausted")
        b = self._free.pop()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        if self.refcount[b] <= 0:
            raise BlockManagerError(f"refcount underflow on block {b}")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self._free.append(b)

    # -- sequences ----------------------------------------------------------------
    def add_seq(self, seq: int) -> None:
        if seq in self.tables:
            raise BlockManagerError(f"sequence {seq} already exists")
        self.tables[seq] = []
        self.num_tokens[seq] = 0

    def _need(self, seq: int):
        if seq not in self.tables:
            raise BlockManagerError(f"unknown sequence {seq}")
        return self.tables[seq]

    def append_slot(self, seq: int):
        """Reserve the slot of the sequence's next token.  Returns (slot, cow) where cow
        is None or the (src, dst) block pair the caller must copy before writing."""
        table = self._need(seq)
        n = self.num_tokens[seq]
        bs = self.block_size
        cow = None
        if n % bs == 0:
            table.append(self._alloc())
        else:
            last = table[n // bs]
            if self.refcount[last] > 1:
                dst = self._alloc()
                self.refcount[last] -= 1
                table[n // bs] = dst
                cow = (last, dst)
        self.num_tokens[seq] = n + 1
        return table[n // bs] * bs + n % bs, cow

    def append_tokens(self, seq: int, count: int):
        """``count`` append_slot calls; returns (slots, cow_pairs).  All or nothing."""
        snapshot = self._snapshot()
        slots, pairs = [], []
        try:
            for _ in range(count):
                slot, cow = self.append_slot(seq)
                slots.append(slot)
                if cow is not None:
                    pairs.append(cow)
        except BlockManagerError:
            self._restore(snapshot)
            raise
        return slots, pairs

    def step(self, seqs):
        """One decode step: append_slot for each listed sequence in order, all or
        nothing.  Returns (slot_mapping, cow_pairs)."""
        snapshot = self._snapshot()
        slots, pairs = [], []
        try:
            for s in seqs:
                slot, cow = self.append_slot(s)
                slots.append(slot)
                if cow is not None:
                    pairs.append(cow)
        except BlockManagerError:
            self._restore(snapshot)
            raise
        return slots, pairs

    def add_seq_shared(self, seq: int, blocks) -> None:
        """A new sequence whose table starts with the given full blocks, already holding
        their tokens (a prefix shared with a cache or another request)."""
        if seq in self.tables:
            raise BlockManagerError(f"sequence {seq} already exists")
        for b in blocks:
            if not 0 <= b < self.num_blocks or self.refcount[b] <= 0:
                raise BlockManagerError(f"block {b} is not allocated")
        for b in blocks:
            self.refcount[b] += 1
        self.tables[seq] = list(blocks)
        self.num_tokens[seq] = len(blocks) * self.block_size

    def retain(self, b: int) -> None:
        """One more holder of an allocated block."""
        if not 0 <= b < self.num_blocks or self.refcount[b] <= 0:
            raise BlockManagerError(f"block {b} is not allocated")
        self.refcount[b] += 1

    def release(self, b: int) -> None:
        """One holder fewer; the block returns to the pool when none is left."""
        if not 0 <= b < self.num_blocks:
            raise BlockManagerError(f"bad block {b}")
        self._release(b)

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (refcount + 1 each)."""
        table = self._need(parent)
        if child in self.tables:
            raise BlockManagerError(f"sequence {child} already exists")
        for b in table:
            self.refcount[b] += 1
        self.tables[child] = list(table)
        self.num_tokens[child] = self.num_tokens[parent]

    def free_seq(self, seq: int) -> None:
        table = self._need(seq)
        for b in reversed(table):
            self._release(b)
        del self.tables[seq]
        del self.num_tokens[seq]

    # -- export -------------------------------------------------------------------
    def block_table(self, seq: int) -> list[int]:
        return list(self._need(seq))

    def export(self, seqs, max_blocks: int, pad: int = -1):
        """(block_tables[len(seqs)][max_blocks], context_lens[len(seqs)]) as lists."""
        tables, lens = [], []
        for s in seqs:
            t = self._need(s)
            if len(t) > max_blocks:
                raise BlockManagerError("max_blocks too small")
            tables.append(list(t) + [pad] * (max_blocks - len(t)))
            lens.append(self.num_tokens[s])
        return tables, lens

    def internal_waste(self, seq: int) -> int:
        """Unused token slots in the sequence's blocks (< block_size)."""
        return len(self._need(seq)) * self.block_size - self.num_tokens[seq]

    def _snapshot(self):
        return (list(self._free), list(self.refcount),
                {k: list(v) for k, v in self.tables.items()}, dict(self.num_tokens))

    def _restore(self, snap):
        self._free, self.refcount, self.tables, self.num_tokens = (
            snap[0], snap[1], snap[2], snap[3])
