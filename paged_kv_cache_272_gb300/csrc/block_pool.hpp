// Internal definition of the host block pool, shared by the pool's C entry points
// (block_pool.cpp) and the serving structures built on it (serving.cpp).
#pragma once

#include <cstdint>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

struct pkv_pool {
  int num_blocks = 0;
  int block_size = 16;
  std::vector<int32_t> free_stack;  // back() is handed out next
  std::vector<int32_t> refcount;
  struct Seq {
    std::vector<int32_t> table;
    int64_t num_tokens = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;

  void release(int32_t b) {
    if (--refcount[b] == 0) free_stack.push_back(b);
  }

  int32_t alloc() {
    int32_t b = free_stack.back();
    free_stack.pop_back();
    refcount[b] = 1;
    return b;
  }

  // Blocks one append at token position n of one sequence needs (a fresh block at a
  // block boundary, a copy when the last block is shared, else none).
  int demand1(const Seq &sq, int64_t n) const {
    if (n % block_size == 0) return 1;
    return refcount[sq.table[n / block_size]] > 1 ? 1 : 0;
  }

  // Blocks one append at token position n needs, given pending refcount changes.
  int demand(const Seq &sq, int64_t n, std::unordered_map<int32_t, int> &delta) const {
    if (n % block_size == 0) return 1;
    int32_t last = sq.table[n / block_size];
    int rc = refcount[last] + delta[last];
    if (rc > 1) {
      delta[last] -= 1;
      return 1;
    }
    return 0;
  }

  // One append (demand already checked).  Returns the slot; fills the COW pair.
  int64_t append(Seq &sq, int32_t *src, int32_t *dst) {
    const int64_t n = sq.num_tokens;
    *src = -1;
    *dst = -1;
    if (n % block_size == 0) {
      sq.table.push_back(alloc());
    } else {
      int32_t &last = sq.table[n / block_size];
      if (refcount[last] > 1) {
        int32_t fresh = alloc();
        refcount[last] -= 1;
        *src = last;
        *dst = fresh;
        last = fresh;
      }
    }
    sq.num_tokens = n + 1;
    return (int64_t)sq.table[n / block_size] * block_size + n % block_size;
  }
};
