// Serving structures on top of the host block pool: a prefix cache (a trie of full
// prompt blocks with LRU eviction) and a continuous-batching scheduler with chunked
// prefill.  Host code; each scheduler step produces the arrays the GPU kernels take
// (block tables, context lengths, slot mapping, copy-on-write pairs, chunk offsets).
//
// Prefix cache ("Inference optimization", Step 3: a trie-based prefix cache with
// lookup, insertion and hit-rate statistics; exercise 4: LRU eviction bounded by
// max_entries; "Continuous batching and PagedAttention", section 3: shared read-only
// blocks with reference counts).  An entry is one full block of a prompt; its trie
// edge is the block's 16 token ids, so a path from the root spells a prompt prefix.
// The cache holds one reference on each cached block.  A lookup matches at most
// (P - 1) / 16 blocks, so the last prompt token is always computed.  Stamps from one
// counter order the entries by last use; only leaves are evicted, least recently used
// first; after an insertion the cache evicts down to max_entries; to free a pool block
// it evicts a leaf whose block no request holds.  The leaves are kept ordered by stamp,
// so an eviction visits leaves oldest first instead of scanning every entry.
//
// Scheduler ("Continuous batching and PagedAttention", section 2: iteration-level
// scheduling -- finished requests leave and waiting requests join at every step --
// and chunked prefill with a per-step token budget; "Inference optimization",
// continuous batching and exercise 2: slot fill rate per step).  One step: retire
// finished requests; one decode token per running request whose prompt is complete
// (admission order); the next prefill chunk of requests still prefilling; admit
// waiting requests first come first served while slots and budget remain (static
// batching admits only into an empty batch).  Out of blocks: evict an unused cached
// block, else preempt the most recently admitted request (recomputed later).
#include <algorithm>
#include <cstring>
#include <deque>
#include <new>
#include <set>
#include <string>
#include <unordered_map>
#include <vector>

#include "block_pool.hpp"

struct pkv_prefix_cache {
  struct Node {
    int32_t block = -1;
    int parent = -1;
    int nchild = 0;
    uint64_t stamp = 0;
    std::string key;  // the edge from the parent: parent id + 16 token ids
    bool alive = false;
  };
  pkv_pool *pool = nullptr;
  int max_entries = 0;
  int bs = 16;
  std::vector<Node> nodes;  // nodes[0] is the root (no block)
  std::vector<int> free_ids;
  std::unordered_map<std::string, int> edges;
  std::set<std::pair<uint64_t, int>> leaves;  // (stamp, id) of every live leaf
  mutable std::string probe;  // lookup key buffer (no allocation per lookup)
  uint64_t clock = 0;
  int64_t entries = 0, lookups = 0, hits = 0, query_tokens = 0, matched_tokens = 0,
          evictions = 0;

  std::string edge(int parent, const int32_t *toks) const {
    std::string k(sizeof(int) + sizeof(int32_t) * bs, '\0');
    std::memcpy(&k[0], &parent, sizeof(int));
    std::memcpy(&k[sizeof(int)], toks, sizeof(int32_t) * bs);
    return k;
  }

  int child(int parent, const int32_t *toks) const {
    probe.resize(sizeof(int) + sizeof(int32_t) * bs);
    std::memcpy(&probe[0], &parent, sizeof(int));
    std::memcpy(&probe[sizeof(int)], toks, sizeof(int32_t) * bs);
    auto it = edges.find(probe);
    return it == edges.end() ? -1 : it->second;
  }

  // Nodes of the longest cached prefix (at most (n - 1) / bs of them).
  int match(const int32_t *toks, int n, std::vector<int> &path) const {
    path.clear();
    const int limit = n > 0 ? (n - 1) / bs : 0;
    int at = 0;
    for (int i = 0; i < limit; ++i) {
      const int c = child(at, toks + (size_t)i * bs);
      if (c < 0) break;
      path.push_back(c);
      at = c;
    }
    return (int)path.size();
  }

  void touch(int id) {
    Node &nd = nodes[id];
    const bool leaf = id != 0 && nd.alive && nd.nchild == 0;
    if (leaf) leaves.erase({nd.stamp, id});
    nd.stamp = ++clock;
    if (leaf) leaves.insert({nd.stamp, id});
  }

  void use(const int32_t *toks, int n, int nmatched) {
    std::vector<int> path;
    match(toks, n, path);
    for (int i = 0; i < nmatched && i < (int)path.size(); ++i) touch(path[i]);
    lookups += 1;
    hits += nmatched > 0 ? 1 : 0;
    query_tokens += n;
    matched_tokens += (int64_t)nmatched * bs;
  }

  // Cache the full blocks of a completely computed prompt; table = its block table.
  void insert(const int32_t *toks, int n, const int32_t *table) {
    int at = 0;
    for (int i = 0; i < n / bs; ++i) {
      int c = child(at, toks + (size_t)i * bs);
      if (c < 0) {
        if (free_ids.empty()) {
          free_ids.push_back((int)nodes.size());
          nodes.emplace_back();
        }
        c = free_ids.back();
        free_ids.pop_back();
        Node &nd = nodes[c];
        nd.block = table[i];
        nd.parent = at;
        nd.nchild = 0;
        nd.alive = true;
        nd.stamp = 0;
        nd.key = edge(at, toks + (size_t)i * bs);
        edges.emplace(nd.key, c);
        if (at != 0 && nodes[at].nchild == 0) leaves.erase({nodes[at].stamp, at});
        nodes[at].nchild += 1;
        leaves.insert({0, c});
        pool->refcount[table[i]] += 1;  // the cache's own reference
        entries += 1;
      }
      touch(c);
      at = c;
    }
    while (entries > max_entries)
      if (!evict(false)) break;
  }

  // Evict the least recently used leaf (whose block only the cache holds, if
  // require_free).  Returns false if there is none.
  bool evict(bool require_free) {
    int best = -1;
    for (const auto &e : leaves)  // oldest first
      if (!require_free || pool->refcount[nodes[e.second].block] == 1) {
        best = e.second;
        break;
      }
    if (best < 0) return false;
    Node &nd = nodes[best];
    leaves.erase({nd.stamp, best});
    edges.erase(nd.key);
    Node &up = nodes[nd.parent];
    up.nchild -= 1;
    if (nd.parent != 0 && up.nchild == 0) leaves.insert({up.stamp, nd.parent});
    pool->release(nd.block);
    nd.alive = false;
    nd.key.clear();
    free_ids.push_back(best);
    entries -= 1;
    evictions += 1;
    return true;
  }

  void clear() {
    for (int id = 1; id < (int)nodes.size(); ++id)
      if (nodes[id].alive) pool->release(nodes[id].block);
    nodes.assign(1, Node());
    nodes[0].alive = true;
    free_ids.clear();
    edges.clear();
    leaves.clear();
    entries = 0;
  }
};

struct pkv_sched {
  struct Req {
    int64_t id = 0;
    std::vector<int32_t> prompt;  // empty: the request does not use the prefix cache
    int P = 0, O = 0, computed = 0, generated = 0;
    bool active = false;  // in `running`
  };
  struct Entry {
    int64_t rid;
    int off, n;  // its new tokens' slots: step_slots[off .. off + n)
  };
  enum Room { kOk, kSelf, kStuck };

  pkv_pool *pool = nullptr;
  pkv_prefix_cache *cache = nullptr;
  int max_num_seqs = 0, budget_per_step = 0, static_policy = 0;
  std::unordered_map<int64_t, Req> reqs;
  std::deque<int64_t> waiting;
  std::vector<int64_t> running;
  // plan of the last step
  std::vector<int64_t> p_seqs, p_slots;
  std::vector<int32_t> p_qlens, p_ctx, p_qstart, p_tables, p_cow;
  int p_num_decode = 0, p_max_blocks = 1, p_finished = 0, p_preempted = 0;
  pkv_sched_stats st = {};
  // per-step scratch, kept between steps (no allocation once warm)
  std::vector<Entry> dec, pre;
  std::vector<int64_t> step_slots, order;
  std::vector<int32_t> step_pairs;

  bool is_running(int64_t rid) const {
    auto it = reqs.find(rid);
    return it != reqs.end() && it->second.active;
  }

  void preempt(int64_t rid) {
    pkv_seq_free(pool, rid);
    Req &r = reqs.at(rid);
    r.computed = r.generated = 0;
    r.active = false;
    running.erase(std::find(running.begin(), running.end(), rid));
    waiting.push_front(rid);
    p_preempted += 1;
    st.preemptions += 1;
  }

  Room make_room(int64_t rid, const std::vector<Entry> &a, const std::vector<Entry> *b) {
    if (cache && cache->evict(true)) return kOk;
    const int64_t victim = running.back();
    for (const Entry &e : a)
      if (e.rid == victim) return kStuck;
    if (b)
      for (const Entry &e : *b)
        if (e.rid == victim) return kStuck;
    preempt(victim);
    return victim == rid ? kSelf : kOk;
  }

  int step() {
    p_seqs.clear();
    p_slots.clear();
    p_qlens.clear();
    p_ctx.clear();
    p_qstart.assign(1, 0);
    p_tables.clear();
    p_cow.clear();
    p_num_decode = p_finished = p_preempted = 0;
    // (1) retire
    for (size_t i = 0; i < running.size();) {
      const int64_t rid = running[i];
      const Req &r = reqs.at(rid);
      if (r.generated == r.O) {
        const int rc = pkv_seq_free(pool, rid);
        if (rc != PKV_OK) return rc;
        reqs.erase(rid);
        running.erase(running.begin() + (long)i);
        p_finished += 1;
        st.finished += 1;
      } else {
        ++i;
      }
    }
    int budget = budget_per_step;
    const bool was_empty = running.empty();
    dec.clear();
    pre.clear();
    step_slots.clear();
    // (2) one decode token per request whose prompt is complete
    order = running;
    for (int64_t rid : order) {
      if (!is_running(rid)) continue;
      Req &r = reqs.at(rid);
      if (r.computed < r.P) continue;
      int64_t slot = -1;
      int32_t src = -1, dst = -1;
      bool ok = false;
      while (true) {
        const int rc = pkv_seq_append_slot(pool, rid, &slot, &src, &dst);
        if (rc == PKV_OK) {
          ok = true;
          break;
        }
        if (rc != PKV_ERR_OOM) return rc;
        if (make_room(rid, dec, nullptr) != kOk) break;
      }
      if (!ok) continue;
      r.computed += 1;
      step_slots.push_back(slot);
      dec.push_back({rid, (int)step_slots.size() - 1, 1});
      if (src >= 0) {
        p_cow.push_back(src);
        p_cow.push_back(dst);
      }
      budget -= 1;
    }
    // (3) the next chunk of requests still prefilling
    order = running;
    for (int64_t rid : order) {
      if (!is_running(rid)) continue;
      Req &r = reqs.at(rid);
      if (r.computed >= r.P || budget <= 0) continue;
      const int chunk = std::min(r.P - r.computed, budget);
      const size_t off = step_slots.size();
      step_slots.resize(off + chunk);
      step_pairs.resize(2 * (size_t)chunk);
      int ncow = 0;
      bool ok = false;
      while (true) {
        const int rc = pkv_seq_append_tokens(pool, rid, chunk, step_slots.data() + off,
                                             step_pairs.data(), &ncow);
        if (rc == PKV_OK) {
          ok = true;
          break;
        }
        if (rc != PKV_ERR_OOM) return rc;
        if (make_room(rid, dec, &pre) != kOk) break;
      }
      if (!ok) {
        step_slots.resize(off);
        continue;
      }
      r.computed += chunk;
      pre.push_back({rid, (int)off, chunk});
      p_cow.insert(p_cow.end(), step_pairs.begin(), step_pairs.begin() + 2 * ncow);
      budget -= chunk;
    }
    // (4) admission, first come first served
    const bool admit = !static_policy || was_empty;
    std::vector<int> path;
    std::vector<int32_t> matched;
    while (admit && !waiting.empty() && (int)running.size() < max_num_seqs && budget > 0) {
      const int64_t rid = waiting.front();
      Req &r = reqs.at(rid);
      const bool cached = cache && !r.prompt.empty();
      int nm = cached ? cache->match(r.prompt.data(), r.P, path) : 0;
      matched.resize(nm);
      for (int i = 0; i < nm; ++i) matched[i] = cache->nodes[path[i]].block;
      const int bs = pool->block_size;
      const int start = nm * bs;
      const int chunk = std::min(r.P - start, budget);
      const int need = (start + chunk + bs - 1) / bs - nm;
      int rc = pkv_seq_add_shared(pool, rid, matched.data(), nm);
      if (rc != PKV_OK) return rc;
      while ((int)pool->free_stack.size() < need && cache && cache->evict(true)) {
      }
      if ((int)pool->free_stack.size() < need) {
        pkv_seq_free(pool, rid);
        break;
      }
      if (cached) cache->use(r.prompt.data(), r.P, nm);
      const size_t off = step_slots.size();
      step_slots.resize(off + chunk);
      step_pairs.resize(2 * (size_t)chunk);
      int ncow = 0;
      rc = pkv_seq_append_tokens(pool, rid, chunk, step_slots.data() + off, step_pairs.data(),
                                 &ncow);
      if (rc != PKV_OK) return rc;
      r.computed = start + chunk;
      waiting.pop_front();
      running.push_back(rid);
      r.active = true;
      pre.push_back({rid, (int)off, chunk});
      p_cow.insert(p_cow.end(), step_pairs.begin(), step_pairs.begin() + 2 * ncow);
      budget -= chunk;
    }
    // (5) sampling: decode entries produce a token; a completed prompt produces its first
    for (const Entry &e : dec) reqs.at(e.rid).generated += 1;
    for (const Entry &e : pre) {
      Req &r = reqs.at(e.rid);
      if (r.computed == r.P) {
        r.generated = 1;
        if (cache && !r.prompt.empty())
          cache->insert(r.prompt.data(), r.P, pool->seqs.at(e.rid).table.data());
      }
    }
    // (6) the plan: decode entries, then prefill entries
    p_num_decode = (int)dec.size();
    p_max_blocks = 1;
    for (const std::vector<Entry> *list : {&dec, &pre})
      for (const Entry &e : *list) {
        p_seqs.push_back(e.rid);
        p_qlens.push_back((int32_t)e.n);
        p_ctx.push_back(reqs.at(e.rid).computed);
        p_slots.insert(p_slots.end(), step_slots.begin() + e.off,
                       step_slots.begin() + e.off + e.n);
        p_qstart.push_back((int32_t)p_slots.size());
        p_max_blocks = std::max(p_max_blocks, (int)pool->seqs.at(e.rid).table.size());
      }
    p_tables.assign(p_seqs.size() * (size_t)p_max_blocks, -1);
    if (!p_seqs.empty())
      pkv_pool_export(pool, p_seqs.data(), (int)p_seqs.size(), p_max_blocks, -1,
                      p_tables.data(), p_ctx.data());
    if (p_seqs.empty() && !(waiting.empty() && running.empty()) && p_finished == 0)
      return PKV_ERR_OOM;
    // statistics
    st.steps += 1;
    const double fill = (double)running.size() / max_num_seqs;
    st.fill_sum += fill;
    if (!waiting.empty()) {
      st.busy_steps += 1;
      st.busy_fill_sum += fill;
    }
    for (int64_t rid : running) {
      const auto &sq = pool->seqs.at(rid);
      const int64_t held = (int64_t)sq.table.size() * pool->block_size;
      st.slots_held += held;
      st.slots_unused += held - sq.num_tokens;
    }
    st.decode_tokens += (int64_t)dec.size();
    for (const Entry &e : pre) st.prefill_tokens += (int64_t)e.n;
    return (int)p_seqs.size();
  }
};

extern "C" {

int pkv_pcache_create(pkv_pool *pool, int max_entries, pkv_prefix_cache **out) {
  if (!pool || !out) return PKV_ERR_NULL;
  *out = nullptr;
  if (max_entries < 0) return PKV_ERR_ARG;
  pkv_prefix_cache *c = new (std::nothrow) pkv_prefix_cache();
  if (!c) return PKV_ERR_OOM;
  c->pool = pool;
  c->max_entries = max_entries;
  c->bs = pool->block_size;
  c->clear();
  *out = c;
  return PKV_OK;
}

void pkv_pcache_destroy(pkv_prefix_cache *cache) {
  if (!cache) return;
  cache->clear();
  delete cache;
}

int pkv_pcache_lookup(const pkv_prefix_cache *cache, const int32_t *tokens, int num_tokens,
                      int32_t *blocks, int max_blocks) {
  if (!cache || (num_tokens > 0 && !tokens)) return PKV_ERR_NULL;
  if (num_tokens < 0) return PKV_ERR_ARG;
  std::vector<int> path;
  const int n = cache->match(tokens, num_tokens, path);
  if (n > 0 && (!blocks || max_blocks < n)) return PKV_ERR_ARG;
  for (int i = 0; i < n; ++i) blocks[i] = cache->nodes[path[i]].block;
  return n;
}

int pkv_pcache_use(pkv_prefix_cache *cache, const int32_t *tokens, int num_tokens,
                   int num_matched) {
  if (!cache || (num_tokens > 0 && !tokens)) return PKV_ERR_NULL;
  if (num_tokens < 0 || num_matched < 0) return PKV_ERR_ARG;
  cache->use(tokens, num_tokens, num_matched);
  return PKV_OK;
}

int pkv_pcache_insert(pkv_prefix_cache *cache, const int32_t *tokens, int num_tokens,
                      const int32_t *table, int table_len) {
  if (!cache || (num_tokens > 0 && (!tokens || !table))) return PKV_ERR_NULL;
  if (num_tokens < 0 || table_len < num_tokens / cache->bs) return PKV_ERR_ARG;
  for (int i = 0; i < num_tokens / cache->bs; ++i)
    if (table[i] < 0 || table[i] >= cache->pool->num_blocks ||
        cache->pool->refcount[table[i]] <= 0)
      return PKV_ERR_ARG;
  cache->insert(tokens, num_tokens, table);
  return PKV_OK;
}

int pkv_pcache_evict_free_one(pkv_prefix_cache *cache) {
  if (!cache) return PKV_ERR_NULL;
  return cache->evict(true) ? 1 : 0;
}

int pkv_pcache_stats(const pkv_prefix_cache *cache, int64_t *out6) {
  if (!cache || !out6) return PKV_ERR_NULL;
  out6[0] = cache->lookups;
  out6[1] = cache->hits;
  out6[2] = cache->query_tokens;
  out6[3] = cache->matched_tokens;
  out6[4] = cache->entries;
  out6[5] = cache->evictions;
  return PKV_OK;
}

int pkv_sched_create(pkv_pool *pool, pkv_prefix_cache *cache, int max_num_seqs,
                     int max_batched_tokens, int static_batching, pkv_sched **out) {
  if (!pool || !out) return PKV_ERR_NULL;
  *out = nullptr;
  if (max_num_seqs <= 0 || max_batched_tokens < max_num_seqs) return PKV_ERR_ARG;
  if (cache && cache->pool != pool) return PKV_ERR_ARG;
  pkv_sched *s = new (std::nothrow) pkv_sched();
  if (!s) return PKV_ERR_OOM;
  s->pool = pool;
  s->cache = cache;
  s->max_num_seqs = max_num_seqs;
  s->budget_per_step = max_batched_tokens;
  s->static_policy = static_batching ? 1 : 0;
  *out = s;
  return PKV_OK;
}

void pkv_sched_destroy(pkv_sched *s) {
  if (!s) return;
  for (int64_t rid : s->running) pkv_seq_free(s->pool, rid);
  delete s;
}

int pkv_sched_add_request(pkv_sched *s, int64_t id, int prompt_len,
                          const int32_t *prompt_tokens, int output_len) {
  if (!s) return PKV_ERR_NULL;
  if (prompt_len < 1 || output_len < 1) return PKV_ERR_ARG;
  if (s->reqs.count(id) || s->pool->seqs.count(id)) return PKV_ERR_DUP_SEQ;
  pkv_sched::Req r;
  r.id = id;
  r.P = prompt_len;
  r.O = output_len;
  if (prompt_tokens) r.prompt.assign(prompt_tokens, prompt_tokens + prompt_len);
  s->reqs.emplace(id, std::move(r));
  s->waiting.push_back(id);
  return PKV_OK;
}

int pkv_sched_step(pkv_sched *s, pkv_step_plan *plan) {
  if (!s || !plan) return PKV_ERR_NULL;
  const int rc = s->step();
  if (rc < 0) return rc;
  plan->num_seqs = (int)s->p_seqs.size();
  plan->num_decode = s->p_num_decode;
  plan->num_tokens = (int)s->p_slots.size();
  plan->max_blocks = s->p_max_blocks;
  plan->num_cow = (int)(s->p_cow.size() / 2);
  plan->finished = s->p_finished;
  plan->preempted = s->p_preempted;
  plan->running = (int)s->running.size();
  plan->waiting = (int)s->waiting.size();
  plan->seq_ids = s->p_seqs.data();
  plan->query_lens = s->p_qlens.data();
  plan->context_lens = s->p_ctx.data();
  plan->query_start = s->p_qstart.data();
  plan->slot_mapping = s->p_slots.data();
  plan->block_tables = s->p_tables.data();
  plan->cow_pairs = s->p_cow.data();
  return rc;
}

int pkv_sched_pack(const pkv_sched *s, void *buf, int64_t buf_bytes, int max_tokens,
                   int max_seqs, int table_stride, pkv_step_pack *pack) {
  if (!s || !pack) return PKV_ERR_NULL;
  if (max_tokens < 1 || max_seqs < 1 || table_stride < 1) return PKV_ERR_ARG;
  // Fixed offsets (from the capacities alone), each 256-byte aligned.
  auto al = [](int64_t x) { return (x + 255) & ~(int64_t)255; };
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = al(off + bytes);
    return o;
  };
  const int64_t T = max_tokens, S = max_seqs;
  pack->slot_mapping = take(8 * T);
  pack->token_seq = take(8 * T);
  pack->last_rows = take(8 * S);
  pack->block_tables = take(4 * S * table_stride);
  pack->context_lens = take(4 * S);
  pack->cow_pairs = take(4 * 2 * S);
  pack->prefill_start = take(4 * (S + 1));
  pack->token_ids = take(4 * T);
  pack->positions = take(4 * T);
  pack->kv_rows = take(8 * T);
  pack->q_rows = take(8 * T);
  pack->total = off;
  const int n = (int)s->p_seqs.size(), nd = s->p_num_decode;
  const int ntok = (int)s->p_slots.size(), ncow = (int)(s->p_cow.size() / 2);
  pack->num_seqs = n;
  pack->num_decode = nd;
  pack->num_tokens = ntok;
  pack->num_cow = ncow;
  if (ntok > max_tokens || n > max_seqs || ncow > max_seqs || s->p_max_blocks > table_stride)
    return PKV_ERR_ARG;
  if (!buf) return PKV_ERR_NULL;
  if (buf_bytes < off) return PKV_ERR_ARG;
  char *b = static_cast<char *>(buf);
  int64_t *slots = reinterpret_cast<int64_t *>(b + pack->slot_mapping);
  int64_t *tseq = reinterpret_cast<int64_t *>(b + pack->token_seq);
  int64_t *last = reinterpret_cast<int64_t *>(b + pack->last_rows);
  int32_t *tables = reinterpret_cast<int32_t *>(b + pack->block_tables);
  int32_t *ctx = reinterpret_cast<int32_t *>(b + pack->context_lens);
  int32_t *cow = reinterpret_cast<int32_t *>(b + pack->cow_pairs);
  int32_t *pstart = reinterpret_cast<int32_t *>(b + pack->prefill_start);
  int32_t *tok = reinterpret_cast<int32_t *>(b + pack->token_ids);
  int32_t *pos = reinterpret_cast<int32_t *>(b + pack->positions);
  if (ntok) std::memcpy(slots, s->p_slots.data(), sizeof(int64_t) * (size_t)ntok);
  if (ncow) std::memcpy(cow, s->p_cow.data(), sizeof(int32_t) * 2 * (size_t)ncow);
  if (n) std::memcpy(ctx, s->p_ctx.data(), sizeof(int32_t) * (size_t)n);
  const int mb = s->p_max_blocks;
  for (int i = 0; i < n; ++i) {
    int32_t *row = tables + (size_t)i * table_stride;
    std::memcpy(row, s->p_tables.data() + (size_t)i * mb, sizeof(int32_t) * (size_t)mb);
    for (int c = mb; c < table_stride; ++c) row[c] = -1;
  }
  int dmax = 0, qmax = 0, outs = nd;
  const int base = n > nd ? s->p_qstart[nd] : 0;
  for (int i = 0; i < n; ++i) {
    const int64_t rid = s->p_seqs[i];
    const int L = s->p_qlens[i], c = s->p_ctx[i];
    const int q0 = s->p_qstart[i];
    const auto &rq = s->reqs.at(rid);
    const int P = rq.P;
    const bool toks = !rq.prompt.empty();
    for (int k = 0; k < L; ++k) {
      const int p = c - L + k;
      tseq[q0 + k] = rid;
      pos[q0 + k] = p;
      tok[q0 + k] = (toks && p < P) ? rq.prompt[(size_t)p] : -1;
    }
    if (i < nd) {
      dmax = std::max(dmax, c);
    } else {
      pstart[i - nd] = q0 - base;
      last[i - nd] = (int64_t)(s->p_qstart[i + 1] - 1 - base);
      qmax = std::max(qmax, L);
      if (c == P) ++outs;  // the chunk completes the prompt: its first output token
    }
  }
  if (n > nd) pstart[n - nd] = s->p_qstart[n] - base;
  pack->decode_max_context = dmax;
  pack->prefill_max_query = qmax;
  pack->outputs = outs;
  return PKV_OK;
}

int pkv_step_synthetic_rows(void *buf, const pkv_step_pack *pack, int64_t table_rows) {
  if (!buf || !pack) return PKV_ERR_NULL;
  if (table_rows <= 0) return PKV_ERR_ARG;
  char *b = static_cast<char *>(buf);
  int32_t *tok = reinterpret_cast<int32_t *>(b + pack->token_ids);
  const int32_t *pos = reinterpret_cast<const int32_t *>(b + pack->positions);
  const int64_t *rid = reinterpret_cast<const int64_t *>(b + pack->token_seq);
  int64_t *kvr = reinterpret_cast<int64_t *>(b + pack->kv_rows);
  int64_t *qr = reinterpret_cast<int64_t *>(b + pack->q_rows);
  for (int t = 0; t < pack->num_tokens; ++t) {
    const int64_t p = pos[t], r = rid[t];
    if (tok[t] < 0) tok[t] = (int32_t)((r * 7777 + p * 131) % 32000);
    kvr[t] = ((int64_t)tok[t] * 1000003 + p * 7919) % table_rows;
    qr[t] = (r * 2654435761LL + p * 40503) % table_rows;
  }
  return PKV_OK;
}

int pkv_sched_done(const pkv_sched *s) {
  if (!s) return PKV_ERR_NULL;
  return s->waiting.empty() && s->running.empty() ? 1 : 0;
}

int pkv_sched_get_stats(const pkv_sched *s, pkv_sched_stats *out) {
  if (!s || !out) return PKV_ERR_NULL;
  *out = s->st;
  return PKV_OK;
}

}  // extern "C"
