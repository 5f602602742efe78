// Host block manager: one pool of fixed-size KV blocks, a block table per sequence,
// reference counts, fork (shared prefixes, parallel sampling) and copy-on-write.
//
// The pages' rules ("Continuous batching and PagedAttention", section 3 PagedAttention;
// "System-level optimization", section 2.3 PagedAttention solution): blocks of one
// size come from a single pool on demand, a request's blocks need not be contiguous,
// released blocks are reused at once, shared blocks are read-only and a private copy
// is made only when a request writes into a shared block.
//
// Allocation policy (the pages leave it open): the free pool is a stack seeded with
// free_order (first element handed out first); a freed block goes on top.  Every
// failing call leaves the pool unchanged: the block demand of a call is counted before
// anything is modified.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <memory>
#include <new>
#include <unordered_map>
#include <vector>

#include "block_pool.hpp"

extern "C" {

int pkv_pool_create(int num_blocks, int block_size, const int32_t *free_order, pkv_pool **out) {
  if (!out) return PKV_ERR_NULL;
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0) return PKV_ERR_ARG;
  pkv_pool *p = new (std::nothrow) pkv_pool();
  if (!p) return PKV_ERR_OOM;
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->refcount.assign(num_blocks, 0);
  p->free_stack.resize(num_blocks);
  std::vector<char> seen(num_blocks, 0);
  for (int i = 0; i < num_blocks; ++i) {
    int32_t b = free_order ? free_order[i] : i;
    if (b < 0 || b >= num_blocks || seen[b]) {
      delete p;
      return PKV_ERR_ARG;
    }
    seen[b] = 1;
    p->free_stack[num_blocks - 1 - i] = b;
  }
  *out = p;
  return PKV_OK;
}

void pkv_pool_destroy(pkv_pool *pool) { delete pool; }

int pkv_pool_num_free(const pkv_pool *pool) {
  return pool ? (int)pool->free_stack.size() : PKV_ERR_NULL;
}

int pkv_block_refcount(const pkv_pool *pool, int block) {
  if (!pool) return PKV_ERR_NULL;
  if (block < 0 || block >= pool->num_blocks) return PKV_ERR_ARG;
  return pool->refcount[block];
}

int pkv_seq_add(pkv_pool *pool, int64_t seq) {
  if (!pool) return PKV_ERR_NULL;
  if (pool->seqs.count(seq)) return PKV_ERR_DUP_SEQ;
  pool->seqs.emplace(seq, pkv_pool::Seq());
  return PKV_OK;
}

int pkv_seq_add_shared(pkv_pool *pool, int64_t seq, const int32_t *blocks, int num_blocks) {
  if (!pool || (num_blocks > 0 && !blocks)) return PKV_ERR_NULL;
  if (num_blocks < 0) return PKV_ERR_ARG;
  if (pool->seqs.count(seq)) return PKV_ERR_DUP_SEQ;
  for (int i = 0; i < num_blocks; ++i)
    if (blocks[i] < 0 || blocks[i] >= pool->num_blocks || pool->refcount[blocks[i]] <= 0)
      return PKV_ERR_ARG;
  pkv_pool::Seq sq;
  sq.table.assign(blocks, blocks + num_blocks);
  sq.num_tokens = (int64_t)num_blocks * pool->block_size;
  for (int32_t b : sq.table) pool->refcount[b] += 1;
  pool->seqs.emplace(seq, std::move(sq));
  return PKV_OK;
}

int pkv_block_retain(pkv_pool *pool, int block) {
  if (!pool) return PKV_ERR_NULL;
  if (block < 0 || block >= pool->num_blocks || pool->refcount[block] <= 0) return PKV_ERR_ARG;
  pool->refcount[block] += 1;
  return PKV_OK;
}

int pkv_block_release(pkv_pool *pool, int block) {
  if (!pool) return PKV_ERR_NULL;
  if (block < 0 || block >= pool->num_blocks) return PKV_ERR_ARG;
  if (pool->refcount[block] <= 0) return PKV_ERR_REFCOUNT;
  pool->release(block);
  return PKV_OK;
}

int pkv_seq_fork(pkv_pool *pool, int64_t parent, int64_t child) {
  if (!pool) return PKV_ERR_NULL;
  auto it = pool->seqs.find(parent);
  if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  if (pool->seqs.count(child)) return PKV_ERR_DUP_SEQ;
  pkv_pool::Seq copy = it->second;
  for (int32_t b : copy.table) pool->refcount[b] += 1;
  pool->seqs.emplace(child, std::move(copy));
  return PKV_OK;
}

int pkv_seq_free(pkv_pool *pool, int64_t seq) {
  if (!pool) return PKV_ERR_NULL;
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  const auto &table = it->second.table;
  for (int32_t b : table)
    if (pool->refcount[b] <= 0) return PKV_ERR_REFCOUNT;
  for (auto r = table.rbegin(); r != table.rend(); ++r) pool->release(*r);
  pool->seqs.erase(it);
  return PKV_OK;
}

int pkv_seq_num_tokens(const pkv_pool *pool, int64_t seq, int *num_tokens) {
  if (!pool || !num_tokens) return PKV_ERR_NULL;
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  *num_tokens = (int)it->second.num_tokens;
  return PKV_OK;
}

int pkv_seq_num_blocks(const pkv_pool *pool, int64_t seq, int *num_blocks) {
  if (!pool || !num_blocks) return PKV_ERR_NULL;
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  *num_blocks = (int)it->second.table.size();
  return PKV_OK;
}

int pkv_seq_append_slot(pkv_pool *pool, int64_t seq, int64_t *slot, int32_t *cow_src,
                        int32_t *cow_dst) {
  if (!pool || !slot || !cow_src || !cow_dst) return PKV_ERR_NULL;
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  if (pool->demand1(it->second, it->second.num_tokens) > (int)pool->free_stack.size())
    return PKV_ERR_OOM;
  *slot = pool->append(it->second, cow_src, cow_dst);
  return PKV_OK;
}

int pkv_seq_append_tokens(pkv_pool *pool, int64_t seq, int count, int64_t *slots,
                          int32_t *cow_pairs, int *num_cow) {
  if (!pool) return PKV_ERR_NULL;
  if (count < 0) return PKV_ERR_ARG;
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  auto &sq = it->second;
  // Demand: a copy only for the first token (afterwards the block is private), plus
  // one block per block boundary crossed.
  int64_t need = 0;
  if (count > 0) {
    const int64_t n = sq.num_tokens, bs = pool->block_size;
    const int64_t have = (n + bs - 1) / bs, want = (n + count + bs - 1) / bs;
    need = want - have;
    if (n % bs != 0) need += pool->demand1(sq, n);
  }
  if (need > (int64_t)pool->free_stack.size()) return PKV_ERR_OOM;
  int ncow = 0;
  for (int i = 0; i < count; ++i) {
    int32_t src, dst;
    int64_t s = pool->append(sq, &src, &dst);
    if (slots) slots[i] = s;
    if (src >= 0) {
      if (cow_pairs) {
        cow_pairs[2 * ncow] = src;
        cow_pairs[2 * ncow + 1] = dst;
      }
      ++ncow;
    }
  }
  if (num_cow) *num_cow = ncow;
  return PKV_OK;
}

int pkv_pool_step(pkv_pool *pool, const int64_t *seqs, int n, int64_t *slot_mapping,
                  int32_t *cow_pairs, int *num_cow) {
  if (!pool || (n > 0 && (!seqs || !slot_mapping))) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_ARG;
  // Count the demand of the whole step first (a sequence may appear more than once).
  std::unordered_map<int32_t, int> delta;
  std::unordered_map<int64_t, int64_t> extra_tokens;
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    auto it = pool->seqs.find(seqs[i]);
    if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
    // Only a sequence's first append of the step can land in a shared block; later
    // ones land in the block that append made private or allocated.
    const int64_t k = extra_tokens[seqs[i]]++;
    const int64_t pos = it->second.num_tokens + k;
    if (pos % pool->block_size == 0) {
      need += 1;
    } else if (k == 0) {
      need += pool->demand(it->second, pos, delta);
    }
  }
  if (need > (int64_t)pool->free_stack.size()) return PKV_ERR_OOM;
  int ncow = 0;
  for (int i = 0; i < n; ++i) {
    auto &sq = pool->seqs.find(seqs[i])->second;
    int32_t src, dst;
    slot_mapping[i] = pool->append(sq, &src, &dst);
    if (src >= 0) {
      if (cow_pairs) {
        cow_pairs[2 * ncow] = src;
        cow_pairs[2 * ncow + 1] = dst;
      }
      ++ncow;
    }
  }
  if (num_cow) *num_cow = ncow;
  return PKV_OK;
}

int pkv_pool_export(const pkv_pool *pool, const int64_t *seqs, int n, int max_blocks,
                    int32_t pad, int32_t *block_tables, int32_t *context_lens) {
  if (!pool || (n > 0 && (!seqs || !block_tables || !context_lens))) return PKV_ERR_NULL;
  if (n < 0 || max_blocks <= 0) return PKV_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    auto it = pool->seqs.find(seqs[i]);
    if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
    if ((int)it->second.table.size() > max_blocks) return PKV_ERR_ARG;
  }
  for (int i = 0; i < n; ++i) {
    const auto &sq = pool->seqs.find(seqs[i])->second;
    int32_t *row = block_tables + (size_t)i * max_blocks;
    size_t nb = sq.table.size();
    if (nb) std::memcpy(row, sq.table.data(), nb * sizeof(int32_t));
    for (int j = (int)nb; j < max_blocks; ++j) row[j] = pad;
    context_lens[i] = (int32_t)sq.num_tokens;
  }
  return PKV_OK;
}

// Snapshot of the pool (checkpoint / resume of the host allocator): little-endian int64
// words -- magic, num_blocks, block_size, the free stack (bottom to top), every block's
// refcount, then each sequence (ascending id) as id, num_tokens, table length, table.
static const int64_t kPoolMagic = 0x314C4F4F5056504BLL;  // "PKVPOOL1"

int64_t pkv_pool_save(const pkv_pool *pool, void *buf, int64_t buf_bytes) {
  if (!pool) return PKV_ERR_NULL;
  std::vector<int64_t> ids;
  ids.reserve(pool->seqs.size());
  int64_t words = 4 + (int64_t)pool->free_stack.size() + pool->num_blocks + 1;
  for (const auto &kv : pool->seqs) {
    ids.push_back(kv.first);
    words += 3 + (int64_t)kv.second.table.size();
  }
  const int64_t bytes = words * 8;
  if (!buf) return bytes;
  if (buf_bytes < bytes) return PKV_ERR_ARG;
  std::sort(ids.begin(), ids.end());
  std::vector<int64_t> w;
  w.reserve(words);
  w.push_back(kPoolMagic);
  w.push_back(pool->num_blocks);
  w.push_back(pool->block_size);
  w.push_back((int64_t)pool->free_stack.size());
  for (int32_t b : pool->free_stack) w.push_back(b);
  for (int32_t r : pool->refcount) w.push_back(r);
  w.push_back((int64_t)ids.size());
  for (int64_t id : ids) {
    const pkv_pool::Seq &sq = pool->seqs.at(id);
    w.push_back(id);
    w.push_back(sq.num_tokens);
    w.push_back((int64_t)sq.table.size());
    for (int32_t b : sq.table) w.push_back(b);
  }
  std::memcpy(buf, w.data(), (size_t)bytes);
  return bytes;
}

}  // extern "C"

namespace {

// The body of pkv_pool_load once the header words have been read and the buffer is known
// to hold the free stack, the refcounts and the sequence count.  May throw
// std::bad_alloc (caught by the caller); the partly built pool is then freed.
int pool_load_checked(const std::vector<int64_t> &w, int64_t at, int64_t nb, int64_t bs,
                      int64_t nfree, pkv_pool **out) {
  const int64_t n = (int64_t)w.size();
  auto next = [&](int64_t &v) -> bool {
    if (at >= n) return false;
    v = w[(size_t)at++];
    return true;
  };
  std::unique_ptr<pkv_pool> p(new pkv_pool());
  p->num_blocks = (int)nb;
  p->block_size = (int)bs;
  std::vector<char> is_free((size_t)nb, 0);
  p->free_stack.reserve((size_t)nfree);
  for (int64_t i = 0; i < nfree; ++i) {
    int64_t b;
    if (!next(b) || b < 0 || b >= nb || is_free[(size_t)b]) return PKV_ERR_ARG;
    is_free[(size_t)b] = 1;
    p->free_stack.push_back((int32_t)b);
  }
  p->refcount.resize((size_t)nb);
  for (int64_t b = 0; b < nb; ++b) {
    int64_t r;
    if (!next(r) || r < 0 || r > INT32_MAX || (r == 0) != (is_free[(size_t)b] != 0))
      return PKV_ERR_ARG;
    p->refcount[(size_t)b] = (int32_t)r;
  }
  int64_t nseq;
  if (!next(nseq) || nseq < 0) return PKV_ERR_ARG;
  std::vector<int64_t> uses((size_t)nb, 0);
  for (int64_t i = 0; i < nseq; ++i) {
    int64_t id, ntok, len;
    // No table covers more tokens than the pool holds (this also keeps the length
    // arithmetic from overflowing).
    if (!next(id) || !next(ntok) || !next(len) || ntok < 0 || ntok > nb * bs ||
        len != ntok / bs + (ntok % bs != 0) || len > n - at || p->seqs.count(id))
      return PKV_ERR_ARG;
    pkv_pool::Seq sq;
    sq.num_tokens = ntok;
    sq.table.reserve((size_t)len);
    for (int64_t j = 0; j < len; ++j) {
      int64_t b;
      if (!next(b) || b < 0 || b >= nb || is_free[(size_t)b] ||
          ++uses[(size_t)b] > p->refcount[(size_t)b])
        return PKV_ERR_ARG;
      sq.table.push_back((int32_t)b);
    }
    p->seqs.emplace(id, std::move(sq));
  }
  if (at != n) return PKV_ERR_ARG;
  *out = p.release();
  return PKV_OK;
}

}  // namespace

extern "C" {

// Rebuild a pool from pkv_pool_save's bytes.  The snapshot is checked before anything
// is built: sizes and ids in range, the buffer long enough for the counts it declares,
// the free stack without repeats, free blocks (and only they) at refcount 0, every
// table of length ceil(num_tokens / block_size) naming blocks in use, and no block
// referenced by more tables than its refcount.  Running out of host memory while
// building returns PKV_ERR_OOM (no exception crosses the C boundary).
int pkv_pool_load(const void *buf, int64_t buf_bytes, pkv_pool **out) {
  if (!out) return PKV_ERR_NULL;
  *out = nullptr;
  if (!buf) return PKV_ERR_NULL;
  if (buf_bytes < 40 || buf_bytes % 8 != 0) return PKV_ERR_ARG;
  try {
    const int64_t n = buf_bytes / 8;
    std::vector<int64_t> w((size_t)n);
    std::memcpy(w.data(), buf, (size_t)buf_bytes);
    const int64_t magic = w[0], nb = w[1], bs = w[2], nfree = w[3];
    if (magic != kPoolMagic) return PKV_ERR_ARG;
    if (nb <= 0 || nb > INT32_MAX || bs <= 0 || bs > INT32_MAX || nfree < 0 || nfree > nb)
      return PKV_ERR_ARG;
    // The free stack, one refcount per block and the sequence count must all be in the
    // buffer: checked before any allocation sized by the snapshot's own numbers.
    if (nfree + nb + 1 > n - 4) return PKV_ERR_ARG;
    return pool_load_checked(w, 4, nb, bs, nfree, out);
  } catch (const std::bad_alloc &) {
    return PKV_ERR_OOM;
  }
}

int paged_kv_check_slots(const int64_t *slot_mapping, int num_tokens, int num_blocks,
                         int block_size) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0) return PKV_ERR_ARG;
  if (num_tokens > 0 && !slot_mapping) return PKV_ERR_NULL;
  const int64_t limit = (int64_t)num_blocks * block_size;
  std::vector<int64_t> live;
  live.reserve((size_t)num_tokens);
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;  // padding
    if (s >= limit) return PKV_ERR_ARG;
    live.push_back(s);
  }
  std::sort(live.begin(), live.end());
  return std::adjacent_find(live.begin(), live.end()) == live.end() ? PKV_OK : PKV_ERR_ARG;
}

}  // extern "C"
