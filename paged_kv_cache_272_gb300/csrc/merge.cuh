// The split-K merge (log-sum-exp weights), as the warp-level device routines of the merge
// kernel:
//   M = max_k lse_k,  o = sum_k 2^(lse_k - M) o_k / sum_k 2^(lse_k - M).
// A partition's result is its normalised output o_k = O_k / l_k and lse_k = m_k + log2 l_k
// (base 2: scores are kept in the log2 domain), so the merged output is the softmax over
// the union of the partitions' tokens ("System-level optimization", section 3.2: tile
// results combined through running max and sum; the combination rule itself is the
// split-K reduction of this implementation).
#pragma once

#include <math.h>

#include "attention.cuh"

namespace pkv {

// A warp merges n entries of one query head: their lse values are read 32 at a time (one
// per lane), their outputs eight at a time with all loads issued before use, and the
// running sum is rescaled when the maximum grows.  Reads bypass L1 (the entries were
// written by other CTAs).
template <int D>
__device__ __forceinline__ void warp_merge(const float *lse, const float *o, size_t stride, int n,
                                           int lane, float &m, float &L, float (&acc)[D / 32]) {
  constexpr int PER = D / 32;
  constexpr unsigned kAllLanes = 0xffffffffu;
  m = -INFINITY;
  L = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  // Eight outputs at a time, every load of a batch issued before any use.
  auto load8 = [&](int first, int cnt, float (&v)[8][PER]) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (first + u < cnt) {
        const float *src = o + (size_t)(first + u) * stride * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
          v[u][0] = t.x, v[u][1] = t.y, v[u][2] = t.z, v[u][3] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
          v[u][0] = t.x, v[u][1] = t.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < PER; ++e) v[u][e] = 0.f;
      }
    }
  };
  for (int k0 = 0; k0 < n; k0 += 32) {
    const int cnt = min(32, n - k0);
    const float x = lane < cnt ? __ldcg(lse + (size_t)(k0 + lane) * stride) : -INFINITY;
    // The first eight outputs do not depend on the weights: load them together with the
    // lse values (one round trip for sequences with at most eight partitions).
    float v[8][PER];
    load8(k0, k0 + cnt, v);
    float mb = x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(kAllLanes, mb, off));
    const float mn = fmaxf(m, mb);
    const float sc = exp2f(m - mn);
    m = mn;
    const float w = exp2f(x - mn);  // this lane's entry weight (0 past the end)
    float ws = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(kAllLanes, ws, off);
    L = fmaf(L, sc, ws);
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= sc;
    for (int k = 0; k < cnt; k += 8) {
      if (k > 0) load8(k0 + k, k0 + cnt, v);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float c = k + u < cnt ? __shfl_sync(kAllLanes, w, (k + u) & 31) : 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(c, v[u][e], acc[e]);
      }
    }
  }
}

// One merge work item `it` = (merge unit it / 8, query head it % 8 of the unit's group),
// done by one warp.  A sequence with one chunk (at most kChunk partitions) is finished
// here; one with several leaves a result per chunk and head, and the warp that completes
// the last chunk of a head (an arrival counter per sequence and head) merges that head's
// chunk results.
template <int D>
__device__ __forceinline__ void merge_item(const AttnArgs &a, int it, int lane) {
  constexpr int PER = D / 32;
  constexpr unsigned kAllLanes = 0xffffffffu;
  const int4 un = a.units[it >> 3];
  const int s = un.x, g8 = un.y, ch = un.z, np = un.w;
  const int h = g8 * 8 + (it & 7);
  if (h >= a.num_q_heads) return;
  const int nch = (np + kChunk - 1) / kChunk;
  const int p0 = ch * kChunk, n = min(kChunk, np - p0);
  float m, L, acc[PER];
  const size_t row = ((size_t)s * a.max_parts + p0) * a.num_q_heads + h;
  warp_merge<D>(a.part_lse + row, a.part_o + row * D, a.num_q_heads, n, lane, m, L, acc);
  float inv = 1.f / L;
  if (nch == 1) {
    uint16_t *o = a.out + ((size_t)s * a.num_q_heads + h) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = f32_to_bf16(acc[e] * inv);
    return;
  }
  const size_t crow = ((size_t)s * a.max_chunks + ch) * a.num_q_heads + h;
  float *co = a.chunk_o + crow * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) co[e] = acc[e] * inv;
  if (lane == 0) a.chunk_lse[crow] = m + log2f(L);
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(&a.cnt_seq[(size_t)s * a.num_q_heads + h], 1) == nch - 1;
  if (!__shfl_sync(kAllLanes, last, 0)) return;
  __threadfence();
  const size_t row2 = (size_t)s * a.max_chunks * a.num_q_heads + h;
  warp_merge<D>(a.chunk_lse + row2, a.chunk_o + row2 * D, a.num_q_heads, nch, lane, m, L, acc);
  inv = 1.f / L;
  uint16_t *o = a.out + ((size_t)s * a.num_q_heads + h) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) o[e] = f32_to_bf16(acc[e] * inv);
}

}  // namespace pkv
