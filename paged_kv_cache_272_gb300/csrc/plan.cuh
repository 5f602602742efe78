// The split-K plan of one decode-attention call, as a CTA-wide device routine: run by the
// plan kernel of paged_attention_decode, and by one CTA of the fused step prologue
// (paged_decode_step), where it overlaps the step's copy and write.
//
// From context_lens alone it
//  * validates every length (a negative one, or one beyond the block table or the
//    workspace, sets PKV_DEV_BAD_CONTEXT and counts as empty) and writes zeros to the
//    output of every empty sequence (no partition will write it);
//  * chooses the partition size P: part_tokens, or, when part_max > part_tokens, the
//    largest candidate <= part_max (part_tokens x 2^k, or with part_fine part_tokens x
//    1, 1.5, 2, 3, 4, 6, 8) not above (total context tokens x work items per partition)
//    / (part_div x the partition kernel's resident CTAs) -- each CTA then meets part_div
//    partitions' worth of work or more, so claiming still balances, while a large batch
//    gets fewer, longer partitions (fewer items, fewer partial results to merge); P goes
//    to *part_eff for the partition kernel;
//  * lists the partitions as records {s, t0, t1, np} ordered by size, largest first (a
//    counting sort over 32 bins of P / 32 tokens, rounded up to whole blocks: every
//    partition but a sequence's last has P tokens), so that claiming records in order
//    balances load;
//  * lists the merge units (sequence, group of 8 query heads, chunk of kChunk
//    partitions) of sequences with several partitions, multi-chunk sequences first (the
//    longest merges start first), and zeroes their second-level arrival counters;
//  * resets the claim counter and publishes the record and unit counts.
// Work that grows with one sequence's length (its records, units, counters, a zeroed
// output row) is spread over the lanes of the warp that owns the sequence, so a
// 131072-token sequence costs no more latency than a short one.
#pragma once

#include "attention.cuh"

namespace pkv {

constexpr unsigned kPlanFull = 0xffffffffu;

// Length of sequence s after validation (0 if invalid); raises the error bit if `flag`.
__device__ __forceinline__ int plan_len(const AttnArgs &a, int s, int cap, bool flag) {
  int c = a.context_lens[s];
  if (c < 0 || c > cap) {
    if (flag) flag_error(a.err, PKV_DEV_BAD_CONTEXT);
    c = 0;
  }
  return c;
}

// Lanes whose `count` is large hand their rows of work to the whole warp: for each such
// lane in turn, every lane runs fn(owner's payload, i) for i = lane, lane + 32, ... <
// count.  Lanes with small counts run their own loop.  All 32 lanes must call it.
template <typename F>
__device__ __forceinline__ void warp_spread(int count, int4 v, int lane, F fn) {
  const bool big = count > 8;
  if (!big)
    for (int i = 0; i < count; ++i) fn(v, i);
  unsigned todo = __ballot_sync(kPlanFull, big);
  while (todo) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1;
    const int n = __shfl_sync(kPlanFull, count, src);
    const int4 w = make_int4(__shfl_sync(kPlanFull, v.x, src), __shfl_sync(kPlanFull, v.y, src),
                             __shfl_sync(kPlanFull, v.z, src), __shfl_sync(kPlanFull, v.w, src));
    for (int i = lane; i < n; i += 32) fn(w, i);
  }
}

// Must be called by every thread of the CTA (blockDim.x a multiple of 32, at most 1024).
__device__ __forceinline__ void attn_plan_cta(const AttnArgs &a, int head_dim) {
  constexpr int kBins = 33;  // partitions of 1..32 blocks (bin 0 unused)
  __shared__ int hist[kBins];
  __shared__ int cursor[kBins];
  __shared__ int ucount[2], ucursor[2];  // merge units: [0] multi-chunk, [1] one chunk
  // Sequences with many full partitions: their records are written by the whole CTA.
  constexpr int kBigMax = 64;
  __shared__ int4 big[kBigMax];          // {s, first record, full partitions, partitions}
  __shared__ int nbig;
  const int tid = threadIdx.x, lane = tid & 31, nthr = blockDim.x;
  for (int i = tid; i < kBins; i += nthr) hist[i] = 0;
  if (tid < 2) ucount[tid] = 0;
  if (tid == 0) nbig = 0;
  __syncthreads();
  const int cap = min(a.max_blocks * kBlockSize, a.max_parts * a.part_tokens);
  // Pass 0 (automatic size only): the call's total context, then P.
  int P = a.part_tokens;
  if (a.part_max > P) {
    __shared__ unsigned long long total;
    if (tid == 0) total = 0;
    __syncthreads();
    unsigned long long mine = 0;
    for (int s = tid; s < a.num_seqs; s += nthr) mine += (unsigned)plan_len(a, s, cap, false);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(kPlanFull, mine, off);
    if (lane == 0 && mine) atomicAdd(&total, mine);
    __syncthreads();
    const unsigned long long budget = total * (unsigned)(a.num_kv_heads * a.sub_groups) /
                                      ((unsigned long long)a.part_div * (unsigned)a.slots);
    // candidates part_tokens x m / 2, m = 2, 3, 4, 6, 8, 12, 16 (fine) or 2, 4, 8, ...
    for (int k = 1;; ++k) {
      const int next = a.part_fine ? a.part_tokens / 2 * ((k & 1) ? 3 << (k >> 1) : 2 << (k >> 1))
                                   : a.part_tokens << k;
      if (next > a.part_max || (unsigned long long)next > budget) break;
      P = next;
    }
  }
  if (tid == 0) *a.part_eff = P;
  const int G8 = (a.num_q_heads + 7) / 8;
  // Bins of P / 32 tokens (whole blocks when P <= 512): bin(blocks) in 1..32.
  const int nbP = P / kBlockSize;
  auto bin_of = [&](int blocks) { return nbP <= 32 ? blocks : (blocks * 32 + nbP - 1) / nbP; };
  const int full_bin = bin_of(nbP);
  const int row_vecs = a.num_q_heads * head_dim / 8;  // 16-byte vectors of one output row
  // Every warp runs the same number of rounds, so the warp-wide steps see all lanes.
  const int rounds = (a.num_seqs + nthr - 1) / nthr;

  // Pass 1: counts.  Empty sequences' outputs are zeroed; multi-chunk sequences' arrival
  // counters are reset.
  for (int r = 0; r < rounds; ++r) {
    const int s = r * nthr + tid;
    const bool live = s < a.num_seqs;
    const int c = live ? plan_len(a, s, cap, true) : 0;
    const int n = (c + P - 1) / P;
    const int nch = (n + kChunk - 1) / kChunk;
    if (n > 1) atomicAdd(&ucount[nch > 1 ? 0 : 1], nch * G8);
    const int nfull = c / P, tail = c - nfull * P;
    if (nfull) atomicAdd(&hist[full_bin], nfull);
    if (tail) atomicAdd(&hist[bin_of((tail + kBlockSize - 1) / kBlockSize)], 1);
    const int4 me = make_int4(s, 0, 0, 0);
    warp_spread(live && n == 0 ? row_vecs : 0, me, lane, [&](int4 v, int i) {
      reinterpret_cast<uint4 *>(a.out + (size_t)v.x * a.num_q_heads * head_dim)[i] =
          make_uint4(0, 0, 0, 0);
    });
    warp_spread(nch > 1 ? a.num_q_heads : 0, me, lane, [&](int4 v, int h) {
      a.cnt_seq[(size_t)v.x * a.num_q_heads + h] = 0;
    });
  }
  __syncthreads();
  // Bin offsets, largest bin first (one warp: a suffix sum over 32 bins by shuffles).
  if (tid < 32) {
    const int b = 32 - lane;  // lane 0 holds bin 32
    const int v = hist[b];
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(kPlanFull, incl, off);
      if (lane >= off) incl += u;
    }
    cursor[b] = incl - v;
    if (lane == 31) {
      *a.num_items = incl;
      *a.work_next = 0;
      ucursor[0] = 0;
      ucursor[1] = ucount[0];
      *a.num_units = ucount[0] + ucount[1];
    }
  }
  __syncthreads();
  // Pass 2: records and units.
  for (int r = 0; r < rounds; ++r) {
    const int s = r * nthr + tid;
    const bool live = s < a.num_seqs;
    const int c = live ? plan_len(a, s, cap, false) : 0;
    const int n = (c + P - 1) / P;
    const int nfull = c / P, tail = c - nfull * P;
    const int pos = nfull ? atomicAdd(&cursor[full_bin], nfull) : 0;
    if (tail) {
      const int at = atomicAdd(&cursor[bin_of((tail + kBlockSize - 1) / kBlockSize)], 1);
      a.items[at] = make_int4(s, nfull * P, c, n);
    }
    // the full partitions of sequence s occupy records pos .. pos + nfull - 1; a long
    // list goes to the CTA-wide pass below (if there is room for it)
    bool mine = true;
    if (nfull > 2 * 32) {
      const int at = atomicAdd(&nbig, 1);
      if (at < kBigMax) {
        big[at] = make_int4(s, pos, nfull, n);
        mine = false;
      }
    }
    warp_spread(mine ? nfull : 0, make_int4(s, pos, n, 0), lane, [&](int4 v, int p) {
      a.items[v.y + p] = make_int4(v.x, p * P, (p + 1) * P, v.z);
    });
    // its merge units (chunk-major, 8-head groups inside a chunk)
    const int nch = n > 1 ? (n + kChunk - 1) / kChunk : 0;
    const int upos = nch ? atomicAdd(&ucursor[nch > 1 ? 0 : 1], nch * G8) : 0;
    warp_spread(nch * G8, make_int4(s, upos, n, 0), lane, [&](int4 v, int u) {
      a.units[v.y + u] = make_int4(v.x, u % G8, u / G8, v.z);
    });
  }
  __syncthreads();
  const int nb = min(nbig, kBigMax);
  for (int b = 0; b < nb; ++b) {
    const int4 v = big[b];
    for (int p = tid; p < v.z; p += nthr) a.items[v.y + p] = make_int4(v.x, p * P, (p + 1) * P, v.w);
  }
}

}  // namespace pkv
