"""Plain-Python reference of the prefix cache (test infrastructure only).

What the pages give:

* A trie-based prefix cache stores the KV entries of shared prompt prefixes and
  supports lookup, insertion and hit-rate statistics ("Inference optimization", Step 3:
  prefix cache (trie)); an LRU-evicting variant holds at most max_entries entries, and
  with 1000 requests of which 60% share 5 common prefixes its hit rate should stay
  above 55% ("Inference optimization", exercise 4).
* With a paged cache the shared prefix is a run of shared, read-only blocks that many
  requests' block tables point at, reference counted (block sharing and copy-on-write,
  "Continuous batching and PagedAttention", section 3).

Readings where the pages are silent (fixed so that the C++ cache can be compared with
this one decision by decision):

* Granularity: an entry is one FULL block of a prompt, keyed by the prompt's whole
  token prefix up to the end of that block.  Entry i of a prompt can exist only if
  entry i - 1 does (a trie whose edges are 16-token blocks).  Partly filled blocks are
  never cached.
* A lookup matches the longest run of cached entries from the start of the prompt,
  leaving at least one prompt token to compute (the model needs the last prompt
  token's output to sample the first new token): at most (P - 1) // 16 blocks.
* The cache holds one reference on each cached block.  A request that uses a matched
  block holds another.
* LRU: every entry carries a stamp from one counter that increases by one per touch.
  A lookup that is used touches its matched entries from the shortest prefix to the
  longest; an insertion touches each entry of the prompt in the same order (creating
  the missing ones).  Only leaves (entries with no longer cached prefix) are evicted,
  least recently touched first.  After an insertion the cache evicts until it holds
  at most max_entries entries.  To free pool blocks, it evicts only leaves whose block
  no request holds (refcount 1), least recently touched first.
* Statistics: request hit rate = lookups that matched at least one block / lookups;
  token hit rate = matched tokens / prompt tokens looked up.
"""
from __future__ import annotations


class PrefixTrie:
    def __init__(self, manager, max_entries: int, block_size: int = 16):
        self.bm = manager                      # oracle.block_manager.BlockManager
        self.max_entries = max_entries
        self.bs = block_size
        self.entries: dict[tuple, list] = {}   # prefix tokens -> [block, stamp]
        self.children: dict[tuple, int] = {}   # prefix tokens -> cached one-block extensions
        self.clock = 0
        self.lookups = self.hits = self.query_tokens = self.matched_tokens = 0
        self.evictions = 0

    # -- helpers --------------------------------------------------------------------
    def _key(self, tokens, i):
        return tuple(tokens[: self.bs * (i + 1)])

    def _is_leaf(self, key) -> bool:
        return self.children.get(key, 0) == 0

    def _touch(self, key):
        self.clock += 1
        self.entries[key][1] = self.clock

    # -- lookup / insert ------------------------------------------------------------
    def lookup(self, tokens) -> list[int]:
        """Blocks of the longest cached prefix (no side effects)."""
        out = []
        limit = (len(tokens) - 1) // self.bs
        for i in range(limit):
            e = self.entries.get(self._key(tokens, i))
            if e is None:
                break
            out.append(e[0])
        return out

    def use(self, tokens, nmatched: int) -> None:
        """Record a lookup whose first nmatched blocks a request now uses."""
        for i in range(nmatched):
            self._touch(self._key(tokens, i))
        self.lookups += 1
        self.hits += 1 if nmatched else 0
        self.query_tokens += len(tokens)
        self.matched_tokens += nmatched * self.bs

    def insert(self, tokens, table) -> None:
        """Cache every full block of a completely computed prompt (table = the request's
        block table), then evict down to max_entries."""
        for i in range(len(tokens) // self.bs):
            key = self._key(tokens, i)
            if key not in self.entries:
                self.bm.retain(table[i])
                self.entries[key] = [table[i], 0]
                parent = key[:-self.bs]
                self.children[parent] = self.children.get(parent, 0) + 1
            self._touch(key)
        while len(self.entries) > self.max_entries:
            if not self._evict(require_free=False):
                break

    def _evict(self, require_free: bool) -> bool:
        best = None
        for key, (block, stamp) in self.entries.items():
            if require_free and self.bm.refcount[block] != 1:
                continue
            if not self._is_leaf(key):
                continue
            if best is None or stamp < self.entries[best][1]:
                best = key
        if best is None:
            return False
        block = self.entries.pop(best)[0]
        self.children[best[:-self.bs]] -= 1
        self.bm.release(block)
        self.evictions += 1
        return True

    def evict_free_one(self) -> bool:
        """Evict the least recently touched leaf that only the cache holds (frees one
        pool block).  False if there is none."""
        return self._evict(require_free=True)
