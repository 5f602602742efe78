// Paged decode attention: plan, split-K partition kernel (CUDA-core variant), LSE merge,
// and the C entry points.
//
// What is computed ("System-level optimization: batching, PagedAttention and
// FlashAttention", section 3.1, the attention equation, and section 3.3, scale =
// head_dim^-1/2): for each sequence s and query head h,
//   out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s
// over the context_lens[s] tokens that block_tables[s] reaches ("Continuous batching
// and PagedAttention", section 3: logical block i -> physical block; 16-token blocks).
//
// How: the context is split into partitions of part_tokens tokens.  One work item is
// (sequence, partition, KV head, query sub-group); it streams the partition's K/V
// blocks once and serves every query head of the group from them, keeping a running
// maximum, a running sum and an unnormalised output (online softmax, fp32).  A
// sequence with one partition is written straight to `out`; otherwise each partition
// leaves (o_p / l_p, m_p + log2 l_p) and a second kernel merges them:
//   M = max_p lse_p,  out = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M).
// Scores are kept in the base-2 domain (q is pre-scaled by scale * log2 e).
#include <math.h>

#include <atomic>

#include "attention.cuh"
#include "merge.cuh"
#include "plan.cuh"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------------------------------
// Plan (one CTA of 1024 threads): see attn_plan_cta.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) attn_plan_kernel(const AttnArgs a, int head_dim) {
  pdl_trigger();
  pdl_wait();
  attn_plan_cta(a, head_dim);
}

// ------------------------------------------------------------------------------------
// Partition kernel, CUDA-core variant.
// Block = 4 warps.  Each warp takes every 4th 16-token block of the partition; a lane
// loads 16-byte chunks of the block's K and V rows (LPT lanes per row), forms partial
// dot products against the GM query heads, sums them over the row's lanes with
// shuffles, and keeps its own online-softmax state.  The 4 warp states are merged in
// shared memory at the end of the item.
// ------------------------------------------------------------------------------------
template <int D, int GM>
__global__ void __launch_bounds__(128) attn_fma_kernel(const AttnArgs a) {
  constexpr int LPT = D / 8;             // lanes per token row (one 16-byte chunk each)
  constexpr int TPI = 32 / LPT;          // rows one warp-wide load covers
  constexpr int NI = kBlockSize / TPI;   // loads per block per lane
  constexpr int NW = 4;
  __shared__ __align__(16) float q_s[GM][D];
  __shared__ float red_m[NW][GM], red_l[NW][GM];
  __shared__ __align__(16) float red_o[NW][GM][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tg = lane / LPT;
  const int dc = lane % LPT;
  pdl_trigger();
  pdl_wait();
  const int per_pair = a.num_kv_heads * a.sub_groups;
  const int total = *a.num_items * per_pair;
  const int part = *a.part_eff;
  // K/V rows are read once: evict them first, so partials and queries stay in L2
  const uint64_t pol = l2_evict_first_policy();
  const uint64_t keep = l2_evict_last_policy();

  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const int pair = w / per_pair;
    const int rem = w - pair * per_pair;
    const int g = rem / a.sub_groups;
    const int sub = rem - g * a.sub_groups;
    const int4 rec = a.items[pair];
    const int s = rec.x, t0 = rec.y, t1 = rec.z;
    const bool single = rec.w == 1;
    const int p = t0 / part;
    const int nblk = (t1 - t0 + kBlockSize - 1) / kBlockSize;
    const int h0 = g * a.group + sub * GM;
    const int gcnt = min(GM, a.group - sub * GM);

    for (int i = threadIdx.x; i < GM * D; i += blockDim.x) {
      const int j = i / D, d = i - j * D;
      q_s[j][d] = j < gcnt
                      ? bf16_to_f32(a.q[((size_t)s * a.num_q_heads + h0 + j) * D + d]) * a.scale_log2
                      : 0.f;
    }
    __syncthreads();

    float m[GM], l[GM], acc[GM][8];
#pragma unroll
    for (int j = 0; j < GM; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
    }

    const int32_t *bt = a.block_tables + (size_t)s * a.max_blocks + t0 / kBlockSize;
    for (int jb = warp; jb < nblk; jb += NW) {
      const int blk = bt[jb];
      if ((unsigned)blk >= (unsigned)a.num_blocks) {
        if (lane == 0) flag_error(a.err, PKV_DEV_BAD_BLOCK);
        continue;
      }
      const size_t base = ((size_t)blk * a.num_kv_heads + g) * (size_t)(kBlockSize * D);
      const uint4 *kp = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.k_cache) + base);
      const uint4 *vp = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.v_cache) + base);
      uint4 kr[NI], vr[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i) kr[i] = ld_stream_v4_hint(kp + i * 32 + lane, pol);
#pragma unroll
      for (int i = 0; i < NI; ++i) vr[i] = ld_stream_v4_hint(vp + i * 32 + lane, pol);
      const int tb = t0 + jb * kBlockSize + tg;  // token of load i: tb + i * TPI

      float sc[NI][GM];
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const float4 qa = *reinterpret_cast<const float4 *>(&q_s[j][dc * 8]);
        const float4 qb = *reinterpret_cast<const float4 *>(&q_s[j][dc * 8 + 4]);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          float x = qa.x * bf16_lo(kr[i].x);
          x = fmaf(qa.y, bf16_hi(kr[i].x), x);
          x = fmaf(qa.z, bf16_lo(kr[i].y), x);
          x = fmaf(qa.w, bf16_hi(kr[i].y), x);
          x = fmaf(qb.x, bf16_lo(kr[i].z), x);
          x = fmaf(qb.y, bf16_hi(kr[i].z), x);
          x = fmaf(qb.z, bf16_lo(kr[i].w), x);
          x = fmaf(qb.w, bf16_hi(kr[i].w), x);
          sc[i][j] = x;
        }
      }
#pragma unroll
      for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
        for (int i = 0; i < NI; ++i)
#pragma unroll
          for (int j = 0; j < GM; ++j) sc[i][j] += __shfl_xor_sync(kFull, sc[i][j], off);
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (tb + i * TPI >= t1)
#pragma unroll
          for (int j = 0; j < GM; ++j) sc[i][j] = -INFINITY;

#pragma unroll
      for (int j = 0; j < GM; ++j) {
        float bmax = sc[0][j];
#pragma unroll
        for (int i = 1; i < NI; ++i) bmax = fmaxf(bmax, sc[i][j]);
#pragma unroll
        for (int off = LPT; off < 32; off <<= 1)
          bmax = fmaxf(bmax, __shfl_xor_sync(kFull, bmax, off));
        const float mn = fmaxf(m[j], bmax);
        const float alpha = exp2f(m[j] - mn);
        m[j] = mn;
        l[j] *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] *= alpha;
      }
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const bool valid = tb + i * TPI < t1;
        float vf[8];
        vf[0] = bf16_lo(vr[i].x); vf[1] = bf16_hi(vr[i].x);
        vf[2] = bf16_lo(vr[i].y); vf[3] = bf16_hi(vr[i].y);
        vf[4] = bf16_lo(vr[i].z); vf[5] = bf16_hi(vr[i].z);
        vf[6] = bf16_lo(vr[i].w); vf[7] = bf16_hi(vr[i].w);
#pragma unroll
        for (int e = 0; e < 8; ++e) vf[e] = valid ? vf[e] : 0.f;  // rows past the end may hold anything
#pragma unroll
        for (int j = 0; j < GM; ++j) {
          const float pr = exp2f(sc[i][j] - m[j]);
          l[j] += pr;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(pr, vf[e], acc[j][e]);
        }
      }
    }

    // Sum over the warp's token groups (lanes that share a head_dim chunk).
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1)
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        l[j] += __shfl_xor_sync(kFull, l[j], off);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] += __shfl_xor_sync(kFull, acc[j][e], off);
      }
    if (lane == 0)
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        red_m[warp][j] = m[j];
        red_l[warp][j] = l[j];
      }
    if (tg == 0)
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        *reinterpret_cast<float4 *>(&red_o[warp][j][dc * 8]) =
            make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
        *reinterpret_cast<float4 *>(&red_o[warp][j][dc * 8 + 4]) =
            make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
      }
    __syncthreads();

    for (int i = threadIdx.x; i < GM * D; i += blockDim.x) {
      const int j = i / D, d = i - j * D;
      if (j >= gcnt) continue;
      float M = red_m[0][j];
#pragma unroll
      for (int ww = 1; ww < NW; ++ww) M = fmaxf(M, red_m[ww][j]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) {
        const float c = exp2f(red_m[ww][j] - M);
        L = fmaf(red_l[ww][j], c, L);
        O = fmaf(red_o[ww][j][d], c, O);
      }
      const int h = h0 + j;
      if (single) {
        a.out[((size_t)s * a.num_q_heads + h) * D + d] = f32_to_bf16(O / L);
      } else {  // partials stay in L2 for the merge kernel (evict-last)
        const size_t idx = ((size_t)s * a.max_parts + p) * a.num_q_heads + h;
        st_f32_hint(a.part_o + idx * D + d, O / L, keep);
        if (d == 0) st_f32_hint(a.part_lse + idx, M + log2f(L), keep);
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------
// Merge kernel: persistent and warp-granular, a work item is (merge unit, one of its 8
// query heads), so the warps of a CTA never wait for one another (see merge_item).
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnArgs a) {
  const int lane = threadIdx.x & 31;
  const int warps = (int)(gridDim.x * (blockDim.x >> 5));
  pdl_trigger();
  pdl_wait();
  const int nitems = *a.num_units * 8;
  for (int it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < nitems; it += warps)
    merge_item<D>(a, it, lane);
}

template <typename K>
int blocks_per_sm(K kernel, int threads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

template <int D, int GM>
int launch_fma_t(const AttnArgs &a, cudaStream_t st) {
  static std::atomic<int> occ_slots[kMaxDevices];
  const int occ = per_device_setup(occ_slots, [] { return blocks_per_sm(attn_fma_kernel<D, GM>, 128); });
  const int64_t upper = (int64_t)a.num_seqs * a.max_parts * a.num_kv_heads * a.sub_groups;
  int64_t grid = (int64_t)device_sm_count() * occ;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  return (int)launch_pdl(attn_fma_kernel<D, GM>, dim3((int)grid), dim3(128), 0, st, a);
}

int launch_merge(const AttnArgs &a, int head_dim, int64_t max_units, cudaStream_t st) {
  static std::atomic<int> occ128[kMaxDevices], occ64[kMaxDevices];
  const int occ = head_dim == 128
                      ? per_device_setup(occ128, [] { return blocks_per_sm(attn_merge_kernel<128>, 256); })
                      : per_device_setup(occ64, [] { return blocks_per_sm(attn_merge_kernel<64>, 256); });
  int64_t grid = (int64_t)device_sm_count() * occ;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  return (int)(head_dim == 128
                   ? launch_pdl(attn_merge_kernel<128>, dim3((int)grid), dim3(256), 0, st, a)
                   : launch_pdl(attn_merge_kernel<64>, dim3((int)grid), dim3(256), 0, st, a));
}

std::atomic<int> g_variant{PKV_ATTN_AUTO};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

AttnWorkspace attn_workspace_layout(int num_seqs, int num_q_heads, int head_dim, int max_parts) {
  AttnWorkspace w;
  size_t off = 0;
  const size_t S = (size_t)num_seqs, P = (size_t)max_parts, H = (size_t)num_q_heads;
  w.num_items_off = off;
  off = align256(off + sizeof(int32_t));
  w.work_next_off = off;
  off = align256(off + sizeof(int32_t));
  w.items_off = off;
  off = align256(off + S * P * sizeof(int4));
  w.lse_off = off;
  off = align256(off + S * P * H * sizeof(float));
  w.o_off = off;
  off = align256(off + S * P * H * (size_t)head_dim * sizeof(float));
  const size_t C = (P + kChunk - 1) / kChunk, G8 = (H + 7) / 8;
  w.units_off = off;
  off = align256(off + S * G8 * C * sizeof(int4));
  w.num_units_off = off;
  off = align256(off + sizeof(int32_t));
  w.cnt_seq_off = off;
  off = align256(off + S * H * sizeof(int32_t));
  w.chunk_lse_off = off;
  off = align256(off + S * C * H * sizeof(float));
  w.chunk_o_off = off;
  off = align256(off + S * C * H * (size_t)head_dim * sizeof(float));
  w.total = off;
  return w;
}

int launch_attn_fma(const AttnArgs &a, int head_dim, int width, cudaStream_t st) {
  if (head_dim == 128) {
    switch (width) {
      case 1: return launch_fma_t<128, 1>(a, st);
      case 2: return launch_fma_t<128, 2>(a, st);
      case 4: return launch_fma_t<128, 4>(a, st);
      default: return launch_fma_t<128, 8>(a, st);
    }
  }
  switch (width) {
    case 1: return launch_fma_t<64, 1>(a, st);
    case 2: return launch_fma_t<64, 2>(a, st);
    case 4: return launch_fma_t<64, 4>(a, st);
    default: return launch_fma_t<64, 8>(a, st);
  }
}

}  // namespace pkv

using namespace pkv;

namespace {
// partition_size <= 0: the workspace holds 512-token partitions and each call's plan
// picks 512, 1024 or 2048 tokens (see attn_plan_cta).
constexpr int kDefaultPartition = 512;
constexpr int kAutoPartitionMax = 4 * kDefaultPartition;
constexpr int kAutoPartitionMaxGqa = 8 * kDefaultPartition;

int max_parts_for(int max_context_len, int part) {
  const int mp = (max_context_len + part - 1) / part;
  return mp > 0 ? mp : 1;
}
}  // namespace

namespace pkv {

int decode_prepare(DecodeCall *d, uint16_t *out, const uint16_t *q, const void *k_cache,
                   const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                   int num_seqs, int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, int num_blocks, float scale, int partition_size,
                   int max_context_len, void *workspace, size_t workspace_bytes,
                   int32_t *err_flag, bool kv8, float k_scale, float v_scale,
                   const float *k_scales, const float *v_scales) {
  d->empty = true;
  if (block_size != kBlockSize) return PKV_ERR_BLOCK_SIZE;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_blocks <= 0 || max_context_len < 0 || num_q_heads % num_kv_heads != 0 ||
      (head_dim != 64 && head_dim != 128))
    return PKV_ERR_SHAPE;
  const bool auto_part = partition_size <= 0;
  const int part = auto_part ? kDefaultPartition : partition_size;
  if (part % kBlockSize != 0) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return PKV_ERR_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ALIGN;
  const int max_parts = max_parts_for(max_context_len, part);
  if ((int64_t)num_seqs * max_parts >= (int64_t)1 << 31) return PKV_ERR_SHAPE;
  const AttnWorkspace ws = attn_workspace_layout(num_seqs, num_q_heads, head_dim, max_parts);
  if (workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKV_ERR_ALIGN;

  char *wb = static_cast<char *>(workspace);
  AttnArgs &a = d->a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.max_blocks = max_blocks_per_seq;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.num_blocks = num_blocks;
  a.part_tokens = part;
  a.slots = device_sm_count() * 4;
  a.max_parts = max_parts;
  a.scale_log2 = (float)((double)scale * (kv8 ? (double)k_scale : 1.0) * 1.4426950408889634);
  a.v_scale = kv8 ? v_scale : 1.0f;
  a.kv8 = kv8 ? 1 : 0;
  a.k_scales = kv8 ? k_scales : nullptr;
  a.v_scales = kv8 ? v_scales : nullptr;
  a.num_items = reinterpret_cast<int32_t *>(wb + ws.num_items_off);
  a.part_eff = a.num_items + 1;  // same 256-byte section
  a.work_next = reinterpret_cast<int32_t *>(wb + ws.work_next_off);
  a.items = reinterpret_cast<int4 *>(wb + ws.items_off);
  a.part_lse = reinterpret_cast<float *>(wb + ws.lse_off);
  a.part_o = reinterpret_cast<float *>(wb + ws.o_off);
  a.max_chunks = (max_parts + kChunk - 1) / kChunk;
  a.units = reinterpret_cast<int4 *>(wb + ws.units_off);
  a.num_units = reinterpret_cast<int32_t *>(wb + ws.num_units_off);
  a.cnt_seq = reinterpret_cast<int32_t *>(wb + ws.cnt_seq_off);
  a.chunk_lse = reinterpret_cast<float *>(wb + ws.chunk_lse_off);
  a.chunk_o = reinterpret_cast<float *>(wb + ws.chunk_o_off);
  a.err = err_flag;

  const int variant = g_variant.load();
  // AUTO: the tensor-core variant once a KV head serves 4 or more query heads (the
  // CUDA-core dot products then cost more issue slots than the bytes they consume);
  // the CUDA-core variant for MHA and small groups, where it already streams at the
  // HBM roofline.  The TMA tensor map indexes rows with 32-bit coordinates.
  const bool tma_ok = (int64_t)num_blocks * num_kv_heads * kBlockSize < ((int64_t)1 << 31);
  const bool use_mma = kv8 || (tma_ok && (variant == PKV_ATTN_MMA ||
                                          (variant == PKV_ATTN_AUTO && a.group >= 4)));
  if (kv8 && !tma_ok) return PKV_ERR_SHAPE;
  const int width = a.group >= 8 ? 8 : (a.group >= 4 ? 4 : (a.group >= 2 ? 2 : 1));
  a.sub_groups = use_mma ? (a.group + 7) / 8 : (a.group + width - 1) / width;
  // Automatic size: the grouped (G >= 4) tensor-core path runs best with about three
  // partitions' worth of records per resident CTA, sizes 512 x {1, 1.5, 2, 3, 4, 6, 8}
  // (measured on GB300: GQA-8 B=256 1536 tokens, the long-context batch 4096); MHA and
  // small groups with four, in powers of two up to 2048 (MHA B=64: 1024).
  const bool gqa_mma = auto_part && use_mma && a.group >= 4;
  a.part_max = auto_part ? (gqa_mma ? kAutoPartitionMaxGqa : kAutoPartitionMax) : part;
  a.part_fine = gqa_mma ? 1 : 0;
  a.part_div = gqa_mma ? 3 : 4;
  d->head_dim = head_dim;
  d->use_mma = use_mma;
  d->width = width;
  d->empty = false;
  return PKV_OK;
}

int decode_launch_after_plan(const DecodeCall &d, cudaStream_t st) {
  const AttnArgs &a = d.a;
  const int rc = d.use_mma ? launch_attn_mma(a, d.head_dim, st)
                           : launch_attn_fma(a, d.head_dim, d.width, st);
  if (rc != 0) return PKV_ERR_CUDA;
  if (a.max_parts > 1) {
    const int64_t units = (int64_t)a.num_seqs * ((a.num_q_heads + 7) / 8) * a.max_chunks;
    if (launch_merge(a, d.head_dim, units, st) != 0) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace pkv

static int decode_impl(uint16_t *out, const uint16_t *q, const void *k_cache,
                       const void *v_cache, const int32_t *block_tables,
                       const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, float scale, int partition_size, int max_context_len,
                       void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream,
                       bool kv8, float k_scale, float v_scale, const float *k_scales = nullptr,
                       const float *v_scales = nullptr) {
  DecodeCall d;
  const int rc = decode_prepare(&d, out, q, k_cache, v_cache, block_tables, context_lens,
                                num_seqs, max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim,
                                block_size, num_blocks, scale, partition_size, max_context_len,
                                workspace, workspace_bytes, err_flag, kv8, k_scale, v_scale,
                                k_scales, v_scales);
  if (rc != PKV_OK || d.empty) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_pdl(attn_plan_kernel, dim3(1), dim3(1024), 0, st, d.a, head_dim) != cudaSuccess)
    return PKV_ERR_CUDA;
  return decode_launch_after_plan(d, st);
}

extern "C" {

size_t paged_attention_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                      int max_context_len, int partition_size) {
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
  const int part = partition_size > 0 ? partition_size : kDefaultPartition;
  return attn_workspace_layout(num_seqs, num_q_heads, head_dim,
                               max_parts_for(max_context_len, part))
      .total;
}

int paged_attention_set_variant(int variant) {
  if (variant != PKV_ATTN_AUTO && variant != PKV_ATTN_FMA && variant != PKV_ATTN_MMA)
    return PKV_ERR_ARG;
  return g_variant.exchange(variant);
}


int paged_attention_decode(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, float scale, int partition_size, int max_context_len,
                           void *workspace, size_t workspace_bytes, int32_t *err_flag,
                           void *stream) {
  return decode_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, partition_size, max_context_len, workspace,
                     workspace_bytes, err_flag, stream, false, 1.0f, 1.0f);
}

int paged_attention_decode_fp8(uint16_t *out, const uint16_t *q, const uint8_t *k_cache,
                               const uint8_t *v_cache, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs,
                               int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, float scale,
                               float k_scale, float v_scale, int partition_size,
                               int max_context_len, void *workspace, size_t workspace_bytes,
                               int32_t *err_flag, void *stream) {
  if (head_dim != 128 && head_dim != 64) return PKV_ERR_SHAPE;
  if (!(k_scale > 0.f) || !(v_scale > 0.f)) return PKV_ERR_SHAPE;
  return decode_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, partition_size, max_context_len, workspace,
                     workspace_bytes, err_flag, stream, true, k_scale, v_scale);
}

int paged_attention_decode_fp8_per_head(uint16_t *out, const uint16_t *q, const uint8_t *k_cache,
                                        const uint8_t *v_cache, const int32_t *block_tables,
                                        const int32_t *context_lens, int num_seqs,
                                        int max_blocks_per_seq, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int num_blocks, float scale, const float *k_scales,
                                        const float *v_scales, int partition_size,
                                        int max_context_len, void *workspace,
                                        size_t workspace_bytes, int32_t *err_flag, void *stream) {
  if (head_dim != 128 && head_dim != 64) return PKV_ERR_SHAPE;
  if (num_seqs > 0 && (!k_scales || !v_scales)) return PKV_ERR_NULL;
  // scale_log2 = scale * log2(e) here; the kernel multiplies in each KV head's k_scale.
  return decode_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, partition_size, max_context_len, workspace,
                     workspace_bytes, err_flag, stream, true, 1.f, 1.f, k_scales, v_scales);
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// Allocation-free decode attention.
//
// Some callers cannot call cudaMalloc at all: code that runs while a CUDA graph is
// being recorded by someone else, an embedding runtime whose memory is owned by its
// own pool, a real-time service that forbids allocation on the serving thread.  For
// them the split-K workspace lives in this fixed device array instead of a buffer
// the caller passes.  Every GPU that loads the library holds the array until the
// process exits.  All calls on a device share it and it keeps the last call's
// contents; the attention path overwrites every part of it it reads, so nothing needs
// clearing between calls.  Calls whose kernels overlap on the GPU race on it.
// ------------------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_noalloc_ptr[kMaxDevices];

// Device address of the array on the current device, looked up once per device.  In
// host code the array's name is only a host-side stand-in, never a device address.
int noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  void *p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PKV_OK;
}

}  // namespace

extern "C" int paged_attention_decode_noalloc(
    uint16_t *out, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, float scale, int partition_size, int max_context_len, int32_t *err_flag,
    void *stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0)
    return PKV_ERR_SHAPE;
  const size_t need = paged_attention_workspace_size(num_seqs, num_q_heads, head_dim,
                                                     max_context_len, partition_size);
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  // The array is chosen by the current device; a stream of another device would get
  // that device's kernels pointed at this device's array.
  int cur = -1, sdev = -1;
  if (cudaGetDevice(&cur) != cudaSuccess ||
      cudaStreamGetDevice((cudaStream_t)stream, &sdev) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (sdev != cur) return PKV_ERR_ARG;
  void *scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != PKV_OK) return rc;
  return paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim,
                                block_size, num_blocks, scale, partition_size, max_context_len,
                                scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, err_flag, stream);
}
