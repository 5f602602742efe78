// One decode step of one layer in three launches: the copy-on-write block copies, the
// paged write of the step's new tokens and the split-K plan share the first launch (the
// "prologue"); the partition kernel and the LSE merge follow as in
// paged_attention_decode.
//
// What is computed is exactly paged_block_copy, then paged_kv_write, then
// paged_attention_decode ("Continuous batching and PagedAttention", section 3: copy a
// shared block before a request writes into it; "Inference optimization", section "KV
// cache": append only the new token's K/V; attention as in attention.cu).  The order
// "copies before writes" is kept inside the one launch by ownership: every copy pair and
// every new token whose block is a pair's source or destination belong to one CTA,
// chosen by the pair's source block, which does that CTA's copies first and those
// tokens' writes after a CTA barrier.  All other tokens are written by other CTAs at the
// same time, and one CTA builds the attention plan meanwhile (the plan reads only
// context_lens).  Pairs sharing a source block land on the same CTA, so a write into a
// source block also waits for every copy out of it.
#include <algorithm>
#include <climits>

#include "attention.cuh"
#include "kv_rows.cuh"
#include "plan.cuh"

namespace pkv {
namespace {

constexpr int kStepThreads = 512;
constexpr int kStepMaxPairs = 1024;  // pairs the prologue takes (more: a copy launch first)
constexpr int kStepMaxWindow = 64;   // most tokens a write CTA takes at a time
constexpr int kCopyBatch = 8;        // 16-byte vectors a thread loads before it stores

// Tokens a write CTA takes at a time: about one 16-byte vector per thread.
__host__ __device__ constexpr int step_window(int per_tok) {
  return per_tok >= kStepThreads ? 1
                                 : (kStepThreads / per_tok < kStepMaxWindow ? kStepThreads / per_tok
                                                                            : kStepMaxWindow);
}

struct StepIO {
  const uint4 *k_new, *v_new;  // [T][Hkv][D] bf16, 16-byte vectors
  const int64_t *slots;        // [T]
  int num_tokens;
  const int32_t *pairs;        // [P][2] (src, dst)
  int num_pairs;
  void *k_cache, *v_cache;
  int heads, row_vecs, num_blocks;
  int64_t num_slots;   // num_blocks * 16
  int64_t block_vecs;  // 16-byte vectors of one block of one cache
  int kv8;
  float k_scale, v_scale;
  const float *k_scales, *v_scales;
  int pair_ctas, write_ctas;
  int win;          // tokens a write CTA takes at a time
  int table_slots;  // entries of the block -> owner hash table (a power of two)
  int32_t *err;
};

// Block id -> owner (the smallest index of a pair whose source block it is, or whose
// destination it is through that pair's source), open addressing in shared memory (load
// factor <= 1/2).  The owning CTA is owner % pair_ctas, so pairs with distinct sources
// spread evenly and pairs sharing a source land on one CTA.
__device__ __forceinline__ uint32_t table_hash(int32_t key, int mask) {
  return ((uint32_t)key * 2654435761u) & (uint32_t)mask;
}
__device__ __forceinline__ void table_insert(int2 *tab, int mask, int32_t key, int owner) {
  for (uint32_t h = table_hash(key, mask);; h = (h + 1) & (uint32_t)mask) {
    const int prev = atomicCAS(&tab[h].x, -1, key);
    if (prev == -1 || prev == key) {
      atomicMin(&tab[h].y, owner);  // the entry starts at INT_MAX
      return;
    }
  }
}
__device__ __forceinline__ int table_find(const int2 *tab, int mask, int32_t key) {
  for (uint32_t h = table_hash(key, mask);; h = (h + 1) & (uint32_t)mask) {
    const int2 e = tab[h];
    if (e.x == key) return e.y;
    if (e.x == -1) return -1;
  }
}

__device__ __forceinline__ void put_vec(const StepIO &io, int64_t i, int64_t slot, int h, int e) {
  if (io.kv8)
    put_row_vec_e4m3(io.k_new, io.v_new, i, slot, h, e, io.heads, io.row_vecs,
                     static_cast<uint2 *>(io.k_cache), static_cast<uint8_t *>(io.v_cache),
                     io.k_scale, io.v_scale, io.k_scales, io.v_scales, io.err);
  else
    put_row_vec_bf16(io.k_new, io.v_new, i, slot, h, e, io.heads, io.row_vecs,
                     static_cast<uint4 *>(io.k_cache), static_cast<uint4 *>(io.v_cache));
}

// Block 0: the attention plan.  Blocks 1 .. pair_ctas: copy pairs, then the writes into
// their blocks.  The rest: every other new token, io.win tokens at a time.
__global__ void __launch_bounds__(kStepThreads) step_prologue_kernel(const AttnArgs a,
                                                                     int head_dim,
                                                                     const StepIO io) {
  extern __shared__ int2 tab[];  // io.table_slots entries when there are pairs
  __shared__ int list[kStepThreads];
  __shared__ long long wslot[kStepMaxWindow];
  __shared__ int nlist;
  pdl_trigger();
  pdl_wait();
  if (blockIdx.x == 0) {
    attn_plan_cta(a, head_dim);
    return;
  }
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int mask = io.table_slots - 1;
  const int C = io.pair_ctas;
  const int per_tok = io.heads * io.row_vecs;
  auto valid_pair = [&](int j) {
    const int src = io.pairs[2 * j], dst = io.pairs[2 * j + 1];
    return (unsigned)src < (unsigned)io.num_blocks && (unsigned)dst < (unsigned)io.num_blocks;
  };
  if (io.num_pairs > 0) {
    for (int i = tid; i < io.table_slots; i += nthr) tab[i] = make_int2(-1, INT_MAX);
    __syncthreads();
    for (int j = tid; j < io.num_pairs; j += nthr)  // sources: the smallest pair index
      if (valid_pair(j)) table_insert(tab, mask, io.pairs[2 * j], j);
    __syncthreads();
    for (int j = tid; j < io.num_pairs; j += nthr)  // destinations: their source's owner
      if (valid_pair(j))
        table_insert(tab, mask, io.pairs[2 * j + 1], table_find(tab, mask, io.pairs[2 * j]));
    __syncthreads();
  }
  const int b = (int)blockIdx.x - 1;
  if (b < C) {
    // Phase 1: this CTA's copies (a pair with a block outside the pool is flagged by
    // pair CTA 0 and skipped).
    for (int j0 = 0; j0 < io.num_pairs; j0 += nthr) {
      if (tid == 0) nlist = 0;
      __syncthreads();
      const int j = j0 + tid;
      if (j < io.num_pairs) {
        const int src = io.pairs[2 * j], dst = io.pairs[2 * j + 1];
        if ((unsigned)src >= (unsigned)io.num_blocks || (unsigned)dst >= (unsigned)io.num_blocks) {
          if (b == 0) flag_error(io.err, PKV_DEV_BAD_BLOCK);
        } else if (table_find(tab, mask, src) % C == b) {
          list[atomicAdd(&nlist, 1)] = j;
        }
      }
      __syncthreads();
      const int n = nlist;
      const int64_t bv = io.block_vecs, total = (int64_t)n * bv;
      uint4 *kc = static_cast<uint4 *>(io.k_cache);
      uint4 *vc = static_cast<uint4 *>(io.v_cache);
      // kCopyBatch vectors of K and of V in flight per thread before the stores
      for (int64_t i0 = 0; i0 < total; i0 += (int64_t)nthr * kCopyBatch) {
        uint4 kv[kCopyBatch], vv[kCopyBatch];
        int64_t to[kCopyBatch];
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
          const int64_t i = i0 + (int64_t)u * nthr + tid;
          to[u] = -1;
          if (i < total) {
            const int jj = list[i / bv];
            const int64_t e = i % bv;
            const int64_t src = io.pairs[2 * jj];
            to[u] = (int64_t)io.pairs[2 * jj + 1] * bv + e;
            kv[u] = kc[src * bv + e];
            vv[u] = vc[src * bv + e];
          }
        }
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u)
          if (to[u] >= 0) {
            kc[to[u]] = kv[u];
            vc[to[u]] = vv[u];
          }
      }
      __syncthreads();
    }
    // Phase 2: the new tokens whose block is one of this CTA's sources or destinations
    // (after every copy above: the CTA barrier orders them).
    for (int t0 = 0; t0 < io.num_tokens; t0 += nthr) {
      if (tid == 0) nlist = 0;
      __syncthreads();
      const int t = t0 + tid;
      if (t < io.num_tokens) {
        const int64_t slot = io.slots[t];
        if (slot >= 0 && slot < io.num_slots) {
          const int own = table_find(tab, mask, (int32_t)(slot >> 4));
          if (own >= 0 && own % C == b) list[atomicAdd(&nlist, 1)] = t;
        }
      }
      __syncthreads();
      const int n = nlist;
      for (int i = tid; i < n * per_tok; i += nthr) {
        const int tt = list[i / per_tok], r = i % per_tok;
        put_vec(io, (int64_t)tt * per_tok + r, io.slots[tt], r / io.row_vecs, r % io.row_vecs);
      }
      __syncthreads();
    }
    return;
  }
  // Write CTAs: windows of io.win tokens; tokens owned by a pair CTA are skipped.
  const int win = io.win;
  for (int t0 = (b - C) * win; t0 < io.num_tokens; t0 += io.write_ctas * win) {
    if (tid < win) {
      const int t = t0 + tid;
      long long keep = -1;
      if (t < io.num_tokens) {
        const int64_t slot = io.slots[t];
        if (slot >= io.num_slots) {
          flag_error(io.err, PKV_DEV_BAD_SLOT);
        } else if (slot >= 0 &&
                   (io.num_pairs == 0 || table_find(tab, mask, (int32_t)(slot >> 4)) < 0)) {
          keep = slot;
        }
      }
      wslot[tid] = keep;
    }
    __syncthreads();
    for (int i = tid; i < win * per_tok; i += nthr) {
      const int lt = i / per_tok, r = i % per_tok;
      const long long slot = wslot[lt];
      if (slot < 0) continue;
      put_vec(io, (int64_t)(t0 + lt) * per_tok + r, slot, r / io.row_vecs, r % io.row_vecs);
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

static int step_impl(uint16_t *out, const uint16_t *q, void *k_cache, void *v_cache,
                     const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                     int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                     int block_size, int num_blocks, float scale, int partition_size,
                     int max_context_len, const uint16_t *k_new, const uint16_t *v_new,
                     const int64_t *slot_mapping, int num_tokens, const int32_t *block_pairs,
                     int num_pairs, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                     void *stream, bool kv8, float k_scale, float v_scale,
                     const float *k_scales, const float *v_scales) {
  if (num_tokens < 0 || num_pairs < 0) return PKV_ERR_SHAPE;
  DecodeCall d;
  int rc = decode_prepare(&d, out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                          max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, scale, partition_size, max_context_len, workspace,
                          workspace_bytes, err_flag, kv8, k_scale, v_scale, k_scales, v_scales);
  if (rc != PKV_OK) return rc;
  if (num_tokens > 0 && (!k_new || !v_new || !slot_mapping)) return PKV_ERR_NULL;
  if (num_pairs > 0 && !block_pairs) return PKV_ERR_NULL;
  if (num_tokens > 0 && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_ALIGN;
  if ((num_tokens > 0 || num_pairs > 0) && (!k_cache || !v_cache)) return PKV_ERR_NULL;
  if ((num_tokens > 0 || num_pairs > 0) && (!aligned16(k_cache) || !aligned16(v_cache)))
    return PKV_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d.empty) {  // no sequences: the copies and the write alone
    if (kv8) {
      rc = paged_block_copy_fp8(static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache),
                                block_pairs, num_pairs, num_blocks, num_kv_heads, head_dim,
                                block_size, err_flag, stream);
      if (rc == PKV_OK)
        rc = k_scales ? paged_kv_write_fp8_per_head(k_new, v_new, slot_mapping, num_tokens,
                                                    static_cast<uint8_t *>(k_cache),
                                                    static_cast<uint8_t *>(v_cache), num_blocks,
                                                    num_kv_heads, head_dim, block_size, k_scales,
                                                    v_scales, err_flag, stream)
                      : paged_kv_write_fp8(k_new, v_new, slot_mapping, num_tokens,
                                           static_cast<uint8_t *>(k_cache),
                                           static_cast<uint8_t *>(v_cache), num_blocks,
                                           num_kv_heads, head_dim, block_size, k_scale, v_scale,
                                           err_flag, stream);
      return rc;
    }
    rc = paged_block_copy(static_cast<uint16_t *>(k_cache), static_cast<uint16_t *>(v_cache),
                          block_pairs, num_pairs, num_blocks, num_kv_heads, head_dim, block_size,
                          err_flag, stream);
    if (rc == PKV_OK)
      rc = paged_kv_write(k_new, v_new, slot_mapping, num_tokens,
                          static_cast<uint16_t *>(k_cache), static_cast<uint16_t *>(v_cache),
                          num_blocks, num_kv_heads, head_dim, block_size, err_flag, stream);
    return rc;
  }
  if (num_pairs > kStepMaxPairs) {  // the copies in a launch of their own, first
    rc = kv8 ? paged_block_copy_fp8(static_cast<uint8_t *>(k_cache),
                                    static_cast<uint8_t *>(v_cache), block_pairs, num_pairs,
                                    num_blocks, num_kv_heads, head_dim, block_size, err_flag,
                                    stream)
             : paged_block_copy(static_cast<uint16_t *>(k_cache),
                                static_cast<uint16_t *>(v_cache), block_pairs, num_pairs,
                                num_blocks, num_kv_heads, head_dim, block_size, err_flag, stream);
    if (rc != PKV_OK) return rc;
    num_pairs = 0;
  }

  StepIO io;
  io.k_new = reinterpret_cast<const uint4 *>(k_new);
  io.v_new = reinterpret_cast<const uint4 *>(v_new);
  io.slots = slot_mapping;
  io.num_tokens = num_tokens;
  io.pairs = block_pairs;
  io.num_pairs = num_pairs;
  io.k_cache = k_cache;
  io.v_cache = v_cache;
  io.heads = num_kv_heads;
  io.row_vecs = head_dim / 8;
  io.num_blocks = num_blocks;
  io.num_slots = (int64_t)num_blocks * kBlockSize;
  io.block_vecs = (int64_t)num_kv_heads * kBlockSize * head_dim * (kv8 ? 1 : 2) / 16;
  io.kv8 = kv8 ? 1 : 0;
  io.k_scale = k_scale;
  io.v_scale = v_scale;
  io.k_scales = k_scales;
  io.v_scales = v_scales;
  io.err = err_flag;
  const int sms = device_sm_count();
  io.pair_ctas = num_pairs > 0 ? std::min(num_pairs, sms) : 0;
  // Tokens per write CTA: about one 16-byte vector per thread; for an E4M3 cache, whose
  // V stores take four times the sectors, as few as lets every CTA of the prologue start
  // at once (one per SM: the copy path needs more than 64 registers a thread).
  io.win = step_window(num_kv_heads * (head_dim / 8));
  if (kv8 && num_tokens > 0) {
    const int room = std::max(1, sms - 1 - io.pair_ctas);
    io.win = std::min(io.win, std::max(1, (num_tokens + room - 1) / room));
  }
  io.write_ctas = num_tokens > 0 ? std::min((num_tokens + io.win - 1) / io.win, 4 * sms) : 0;
  int slots = 64;
  while (slots < 4 * num_pairs) slots *= 2;
  io.table_slots = slots;
  const size_t smem = num_pairs > 0 ? (size_t)slots * sizeof(int2) : 0;
  const int grid = 1 + io.pair_ctas + io.write_ctas;
  if (launch_pdl(step_prologue_kernel, dim3(grid), dim3(kStepThreads), smem, st, d.a, head_dim,
                 io) != cudaSuccess)
    return PKV_ERR_CUDA;
  return decode_launch_after_plan(d, st);
}

extern "C" {

int paged_decode_step(uint16_t *out, const uint16_t *q, uint16_t *k_cache, uint16_t *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                      int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, float scale, int partition_size,
                      int max_context_len, const uint16_t *k_new, const uint16_t *v_new,
                      const int64_t *slot_mapping, int num_tokens, const int32_t *block_pairs,
                      int num_pairs, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                      void *stream) {
  return step_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                   max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                   num_blocks, scale, partition_size, max_context_len, k_new, v_new,
                   slot_mapping, num_tokens, block_pairs, num_pairs, workspace, workspace_bytes,
                   err_flag, stream, false, 1.f, 1.f, nullptr, nullptr);
}

int paged_decode_step_fp8(uint16_t *out, const uint16_t *q, uint8_t *k_cache, uint8_t *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, float scale,
                          float k_scale, float v_scale, const float *k_scales,
                          const float *v_scales, int partition_size, int max_context_len,
                          const uint16_t *k_new, const uint16_t *v_new,
                          const int64_t *slot_mapping, int num_tokens,
                          const int32_t *block_pairs, int num_pairs, void *workspace,
                          size_t workspace_bytes, int32_t *err_flag, void *stream) {
  if (head_dim != 128 && head_dim != 64) return PKV_ERR_SHAPE;
  if ((k_scales == nullptr) != (v_scales == nullptr)) return PKV_ERR_NULL;
  if (k_scales == nullptr && (!(k_scale > 0.f) || !(v_scale > 0.f))) return PKV_ERR_SHAPE;
  // With per-head scales the kernels multiply each KV head's k_scale in themselves.
  const float ks = k_scales ? 1.f : k_scale, vs = v_scales ? 1.f : v_scale;
  return step_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                   max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                   num_blocks, scale, partition_size, max_context_len, k_new, v_new,
                   slot_mapping, num_tokens, block_pairs, num_pairs, workspace, workspace_bytes,
                   err_flag, stream, true, ks, vs, k_scales, v_scales);
}

}  // extern "C"
