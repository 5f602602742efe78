// Partition kernel, tensor-core variant: the query-group contraction on mma.sync tiles,
// K/V tiles staged by TMA into per-warp shared-memory rings.
//
// Same arithmetic as the CUDA-core variant (softmax(scale q K^T) V per query head with
// an online max and sum in fp32, "System-level optimization: batching, PagedAttention
// and FlashAttention", sections 3.1 and 3.3), arranged for GB300:
//
//  * One CTA = one producer warp + NW consumer warps, several CTAs per SM, persistent:
//    the producer claims the plan's records (largest first) from a global counter and
//    announces them to the consumers through a small shared-memory ring, so CTAs that
//    drew lighter records take more of them.  Block jb of an item goes to consumer
//    warp jb % NW.
//  * The producer reads each block id from the block table ("Continuous batching and
//    PagedAttention", section 3: logical block -> physical block) and issues TMA tiled
//    copies (cp.async.bulk.tensor.2d, 128-byte swizzle) of the block's K and V head
//    tiles (16 rows x head_dim bf16) into the target warp's ring slot; completion is
//    signalled on the slot's "full" mbarrier with the byte count.  The consumer frees
//    the slot through its "empty" mbarrier.  Every wait is bounded.
//  * (E4M3 cache: K tiles by TMA as above, V tiles -- stored transposed, [d][16] -- by a
//    plain bulk copy; a ring stage holds two blocks, so a stage carries the bytes of one
//    bf16 block and one softmax update covers 32 tokens; codes convert to f16 in
//    registers, see the KV8 branches.)
//  * A consumer computes S^T[16 tokens x 8 heads] = K Q^T with mma.m16n8k16 (tokens are
//    the M dimension, the query group is N, head_dim is K), so a GQA-8 group fills the
//    tile exactly; Q^T fragments live in registers for the whole item.  The softmax
//    weights P (rounded to bf16) go from the accumulator layout to the B-operand layout
//    with movmatrix (an 8x8 transpose in registers), and O^T[head_dim x 8] += V^T P^T is
//    a second set of mma tiles whose A operand ldmatrix.trans reads straight from the
//    staged V tile.  The sum of the weights uses the same rounded values.
//  * At the end of an item each consumer warp writes its state (max, sum, O tiles) into
//    the last ring stage it consumed, which it keeps until the merge is done (no merge
//    buffer: the shared memory goes to more CTAs per SM); each warp then merges a slice
//    of head_dim across the NW states, and the item's result goes to `out` (one
//    partition) or to the split-K partials (merged by the LSE merge kernel).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attention.cuh"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// c += A(16x16, row) * B(16x8, col), f16 inputs, fp32 accumulate (E4M3 cache path).
__device__ __forceinline__ void mma16816_f16(float (&c)[4], uint32_t a0, uint32_t a1,
                                             uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void sts128(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__device__ __forceinline__ void lds128(uint32_t addr, float &a, float &b, float &c, float &d) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(a), "=f"(b), "=f"(c), "=f"(d)
               : "r"(addr)
               : "memory");
}

// Four E4M3 codes (lowest byte first) -> two f16x2 words (codes 0-1, codes 2-3), exactly:
// the 32-bit word is split into its two 16-bit halves in registers and each half
// converted by one cvt.rn.f16x2.e4m3x2.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

// 2^x by the MUFU ex2 instruction (relative error below 2^-22; subnormal results flush to
// zero: such weights are below 2^-126 of the running maximum's).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// Q^T as the B operand of S^T = K Q^T for one item: thread (gid, tig) holds
// q[h0 + gid][16 kk + 2 tig (+8) .. +1] as bf16 pairs (zero for heads past the group).
// For the E4M3 cache the head_dim index inside each 16-wide k-step is permuted so that a
// thread's four K elements are four consecutive bytes: logical k = 2 tig + j reads
// column 16 kk + 4 tig + j and k = 2 tig + 8 + j reads 16 kk + 4 tig + 2 + j.  Q uses
// the same permutation (a dot product does not depend on the order of its terms), in
// f16 (bf16 -> f16 is exact for |q| in [2^-14, 65504]; smaller magnitudes keep f16's
// subnormal precision).
template <int D>
__device__ __forceinline__ void load_q_frag_f16perm(uint32_t (&qb)[D / 16][2], const AttnArgs &a,
                                                    int item, int per_pair, int4 rec, int gid,
                                                    int tig, bool live) {
  const int rem = item % per_pair;
  const int g = rem / a.sub_groups;
  const int sub = rem - g * a.sub_groups;
  const int h0 = g * a.group + sub * 8;
  const bool on = live && gid < min(8, a.group - sub * 8);
  const uint2 *qrow =
      reinterpret_cast<const uint2 *>(a.q + ((size_t)rec.x * a.num_q_heads + h0 + gid) * D);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint2 w = on ? qrow[(16 * kk + 4 * tig) >> 2] : make_uint2(0u, 0u);
    qb[kk][0] = pack_f16(bf16_lo(w.x), bf16_hi(w.x));
    qb[kk][1] = pack_f16(bf16_lo(w.y), bf16_hi(w.y));
  }
}

template <int D>
__device__ __forceinline__ void load_q_frag(uint32_t (&qb)[D / 16][2], const AttnArgs &a,
                                            int item, int per_pair, int4 rec, int gid, int tig,
                                            bool live) {
  const int rem = item % per_pair;
  const int g = rem / a.sub_groups;
  const int sub = rem - g * a.sub_groups;
  const int h0 = g * a.group + sub * 8;
  const bool on = live && gid < min(8, a.group - sub * 8);
  const uint32_t *qrow =
      reinterpret_cast<const uint32_t *>(a.q + ((size_t)rec.x * a.num_q_heads + h0 + gid) * D);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    qb[kk][0] = on ? qrow[(16 * kk + 2 * tig) >> 1] : 0u;
    qb[kk][1] = on ? qrow[(16 * kk + 8 + 2 * tig) >> 1] : 0u;
  }
}

template <int D, int NW, int NS, bool KV8 = false>
struct MmaLayout {
  static constexpr int kTile = kBlockSize * D * (KV8 ? 1 : 2);  // one K (or V) head tile
  // Blocks per ring stage: two for the E4M3 cache, so that a stage carries as many bytes
  // (and a consumer step as many tokens per softmax update) as one bf16 block.
  static constexpr int kBps = KV8 ? 2 : 1;
  static constexpr int kStage = 2 * kTile * kBps;  // [K0 V0 (K1 V1)]
  static constexpr int kRing = 4;                    // item slots producer -> consumers
  static constexpr int kStagesBytes = NW * NS * kStage;
  // Item-end merge: each consumer warp leaves its state (float4 chunks [KSTEPS + 1][32
  // lanes]) in the last stage it consumed, so the merge needs no buffer of its own.
  static_assert((D / 16 + 1) * 32 * 16 <= kStage, "warp state must fit in one stage");
  // mbarriers (block full/empty, item full/empty), item records, then ints
  static constexpr int kCtlBytes =
      (2 * NW * NS + 2 * kRing) * 8 + (kRing + 1) * 16 + (kRing + 2 + NW * NS + NW) * 4 + 16;
  static constexpr int kSmem = 1024 + kStagesBytes + kCtlBytes;
};

template <int D, int NW, int NS, bool KV8>
__global__ void __launch_bounds__((NW + 1) * 32,
                                  NW == 1 ? 8 : (NW <= 2 ? 5 : (NW <= 3 ? 4 : (NW <= 4 ? 2 : 1))))
    attn_mma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv) {
  using L = MmaLayout<D, NW, NS, KV8>;
  constexpr int KSTEPS = D / 16;
  constexpr int HALVES = D / 64;
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned stage area (the swizzle pattern repeats every 1024 bytes).
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  unsigned char *base = smem_raw + (base_u32 - raw_u32);
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + L::kStagesBytes);
  int4 *ring_rec = reinterpret_cast<int4 *>(bars + 2 * NW * NS + 2 * L::kRing);  // [kRing]
  volatile int4 *cons_rec = ring_rec + L::kRing;
  int *ring_item = reinterpret_cast<int *>(ring_rec + L::kRing + 1);         // [kRing]
  volatile int *cons_item = ring_item + L::kRing;
  volatile int *abort_flag = cons_item + 1;
  int *valid = const_cast<int *>(abort_flag) + 1;                            // [NW][NS]
  volatile uint32_t *state_at = reinterpret_cast<volatile uint32_t *>(valid + NW * NS);  // [NW]
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + NW * NS * 8;
  const uint32_t ifull0 = empty0 + NW * NS * 8, iempty0 = ifull0 + L::kRing * 8;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < L::kRing; ++i) {
      mbar_init(ifull0 + 8 * i, 1);
      mbar_init(iempty0 + 8 * i, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // the plan's records (and the step's cache writes) are complete

  const int per_pair = a.num_kv_heads * a.sub_groups;
  const int total = *a.num_items * per_pair;
  const int part = *a.part_eff;  // the plan's partition size

  if (warp == NW) {
    // ------------------------------- producer -------------------------------------
    // Items are claimed from the plan's list (largest first) through a global counter,
    // one item ahead, and announced to the consumers through a small ring of item
    // slots.  Lane w < NW feeds consumer warp w: stage js of an item (blocks
    // kBps js .. kBps js + kBps - 1) goes to lane js % NW, so the lanes issue their
    // copies side by side.  Lane w counts the stages it handed to warp w (ring slot =
    // count % NS, phase = count / NS).
    constexpr int BPS = L::kBps;
    // K/V tiles are read once: evict them first, so partials and queries stay in L2
    const uint64_t pol = l2_evict_first_policy();
    int cnt = 0;               // stages handed to warp `lane` so far
    int pslot = 0, pphase = 0;  // = cnt % NS, (cnt / NS) & 1, kept incrementally
    bool stop = false;
    auto claim = [&]() -> int {
      int it = 0;
      if (lane == 0) it = atomicAdd(a.work_next, 1);
      return __shfl_sync(kFull, it, 0);
    };
    auto first_chunk = [&](int it, int4 r) -> int {  // first block-table entries, one per lane
      if (it >= total) return 0;
      const int nb = (r.z - r.y + kBlockSize - 1) / kBlockSize;
      return lane < nb ? a.block_tables[(size_t)r.x * a.max_blocks + r.y / kBlockSize + lane] : 0;
    };
    auto publish = [&](int k, int it, int4 r) -> bool {
      int ok = 1;
      if (lane == 0) {
        const int slot = k % L::kRing;
        ok = mbar_wait(iempty0 + 8 * slot, ((k / L::kRing) & 1) ^ 1, abort_flag, a.err);
        if (ok) {
          ring_item[slot] = it;
          ring_rec[slot] = r;
          mbar_arrive(ifull0 + 8 * slot);
        }
      }
      return __shfl_sync(kFull, ok, 0) != 0;
    };
    int cur = claim();
    int4 rec = cur < total ? a.items[cur / per_pair] : make_int4(0, 0, 0, 0);
    int chunk0 = first_chunk(cur, rec);
    stop = !publish(0, cur, rec);
    for (int k = 0; cur < total && !stop; ++k) {
      const int nxt = claim();
      const int4 rec_n = nxt < total ? a.items[nxt / per_pair] : rec;
      const int g = (cur % per_pair) / a.sub_groups;
      const int nblk = (rec.z - rec.y + kBlockSize - 1) / kBlockSize;
      const int32_t *bt = a.block_tables + (size_t)rec.x * a.max_blocks + rec.y / kBlockSize;
      // Block ids come 32 lanes at a time, in chunks of CH (a multiple of NW * BPS) so
      // that the blocks of stage js = (c + r) / BPS + lane always land on warp js % NW.
      constexpr int CH = (32 / (NW * BPS)) * NW * BPS;
      for (int c = 0; c < nblk && !stop; c += CH) {
        const int blk_lane = c == 0 ? chunk0 : (c + lane < nblk ? bt[c + lane] : 0);
        const int n = min(CH, nblk - c);
        for (int r = 0; r < n; r += NW * BPS) {
          int bj[BPS];
#pragma unroll
          for (int j = 0; j < BPS; ++j)
            bj[j] = __shfl_sync(kFull, blk_lane, (r + BPS * lane + j) & 31);
          int ok = 1;
          if (lane < NW && r + BPS * lane < n) {
            const int slot = pslot;
            const uint32_t fb = full0 + 8 * (lane * NS + slot);
            ok = mbar_spin_wait(empty0 + 8 * (lane * NS + slot), pphase ^ 1, abort_flag, a.err);
            if (ok) {
              // bit j: block j of the stage exists and its id is inside the pool
              int vbits = 0;
#pragma unroll
              for (int j = 0; j < BPS; ++j) {
                if (r + BPS * lane + j >= n) continue;
                if ((unsigned)bj[j] >= (unsigned)a.num_blocks)
                  flag_error(a.err, PKV_DEV_BAD_BLOCK);
                else
                  vbits |= 1 << j;
              }
              valid[lane * NS + slot] = vbits;
              if (vbits == 0) {
                mbar_arrive(fb);
              } else {
                mbar_arrive_expect_tx(fb, __popc(vbits) * 2 * L::kTile);
#pragma unroll
                for (int j = 0; j < BPS; ++j) {
                  if (!((vbits >> j) & 1)) continue;
                  const uint32_t dst =
                      base_u32 + (uint32_t)((lane * NS + slot) * L::kStage + j * 2 * L::kTile);
                  const int y = (bj[j] * a.num_kv_heads + g) * kBlockSize;
                  if constexpr (KV8) {
                    // K: one [16][128 B] swizzled box; V (stored [d][16]): 2 KB contiguous
                    tma_load_2d_hint(dst, &tk, 0, y, fb, pol);
                    bulk_load_hint(dst + L::kTile,
                                   static_cast<const uint8_t *>(a.v_cache) + (size_t)y * D,
                                   L::kTile, fb, pol);
                  } else {
#pragma unroll
                    for (int h = 0; h < HALVES; ++h) {
                      tma_load_2d_hint(dst + h * 2048, &tk, h * 64, y, fb, pol);
                      tma_load_2d_hint(dst + L::kTile + h * 2048, &tv, h * 64, y, fb, pol);
                    }
                  }
                }
              }
              ++cnt;
              if (++pslot == NS) {
                pslot = 0;
                pphase ^= 1;
              }
            }
          }
          if (!__all_sync(kFull, ok)) {
            stop = true;
            break;
          }
        }
      }
      const int chunk0_n = first_chunk(nxt, rec_n);
      if (!stop) stop = !publish(k + 1, nxt, rec_n);
      cur = nxt;
      rec = rec_n;
      chunk0 = chunk0_n;
    }
    // Wait for every copy still in flight before the CTA may exit.
    if (lane < NW) {
      for (int i = max(0, cnt - NS); i < cnt; ++i)
        mbar_drain(full0 + 8 * (lane * NS + i % NS), (i / NS) & 1);
    }
    return;
  }

  // --------------------------------- consumers --------------------------------------
  // Thread 0 takes item k from the ring and leaves it in cons_item / cons_rec; a
  // consumer-wide barrier then hands it to every consumer thread, so all consumer
  // warps follow the same item sequence (and the same barriers) even after a timeout.
  auto fetch = [&](int k) {
    const int slot = k % L::kRing;
    if (mbar_wait(ifull0 + 8 * slot, (k / L::kRing) & 1, abort_flag, a.err)) {
      *cons_item = ring_item[slot];
      const int4 r = ring_rec[slot];
      cons_rec->x = r.x;
      cons_rec->y = r.y;
      cons_rec->z = r.z;
      cons_rec->w = r.w;
      mbar_arrive(iempty0 + 8 * slot);
    } else {
      *cons_item = total;  // give up: behave as if the list had ended
    }
  };
  const int gid = lane >> 2, tig = lane & 3;
  const uint64_t keep = l2_evict_last_policy();  // for the split-K partials
  int cslot = 0, cphase = 0;  // ring slot and phase of this warp's next block
  // Per-thread shared-memory offsets inside a stage (the swizzle folded in once; a k-step
  // then only flips the 16-byte chunk bits 4..6, which a stage base never sets).
  const int tokA8 = 4 * (gid >> 1) + (gid & 1), tokB8 = tokA8 + 2;  // E4M3 token order
  // E4M3 K rows are D bytes: head_dim 128 with the 128-byte swizzle (16-byte chunk ^=
  // row & 7), head_dim 64 with the 64-byte swizzle (chunk ^= (row >> 1) & 3).
  // E4M3 fragments come from ldmatrix.x4 (b16 view of the codes: a thread receives 4
  // bytes of one 16-byte row segment, the 4 codes its f16 fragment needs).  K: lane l
  // addresses row token (l >> 3) & 1 ? tokB : tokA of row-group l & 7, k-step + (l >> 4);
  // V (transposed, [d][16] without swizzle): row d = 16 (l >> 4) + 8 ((l >> 3) & 1) + (l & 7).
  const int lm = lane >> 3, lr = lane & 7;
  const int ltok = 4 * (lr >> 1) + (lr & 1) + ((lm & 1) ? 2 : 0);
  const uint32_t krow8 = (uint32_t)(ltok * D);  // D bytes per E4M3 K row
  const uint32_t kkey8 = D == 128 ? (uint32_t)(ltok & 7) : (uint32_t)((ltok >> 1) & 3);
  const uint32_t kstep8 = (uint32_t)(lm >> 1);
  const uint32_t vrow8 = (uint32_t)((16 * (lm >> 1) + 8 * (lm & 1) + lr) * 16);
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row (bf16 K tile)
  const uint32_t koff16 = (uint32_t)(lrow * 128 + ((((lane >> 4) & 1) ^ (lrow & 7)) << 4));
  if (threadIdx.x == 0) fetch(0);
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
  int cur = *cons_item;
  int4 rec = make_int4(cons_rec->x, cons_rec->y, cons_rec->z, cons_rec->w);
  uint32_t qb[KSTEPS][2];
  if constexpr (KV8)
    load_q_frag_f16perm<D>(qb, a, cur < total ? cur : 0, per_pair, rec, gid, tig, cur < total);
  else
    load_q_frag<D>(qb, a, cur < total ? cur : 0, per_pair, rec, gid, tig, cur < total);
  asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");  // cons_* read by all
  for (int k = 0; cur < total; ++k) {
    const int rem = cur % per_pair;
    const int g = rem / a.sub_groups;
    const int sub = rem - g * a.sub_groups;
    const int s = rec.x, t0 = rec.y, t1 = rec.z;
    const int nblk = (t1 - t0 + kBlockSize - 1) / kBlockSize;
    const int h0 = g * a.group + sub * 8;
    const int gcnt = min(8, a.group - sub * 8);
    float sl2 = a.scale_log2, vsc = a.v_scale;  // per-cache values (1 for v_scale of bf16)
    if constexpr (KV8) {
      if (a.k_scales != nullptr) {  // E4M3 scales of this KV head
        const float ks = __ldg(a.k_scales + g), vs = __ldg(a.v_scales + g);
        if (lane == 0 && (!(ks > 0.f) || !(vs > 0.f))) flag_error(a.err, PKV_DEV_BAD_SCALE);
        sl2 *= ks;
        vsc = vs;
      }
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[KSTEPS][4];
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

    const int nstage = (nblk + L::kBps - 1) / L::kBps;
    int held = -1;  // ring slot this warp keeps until the item's merge is done
    for (int jb = warp; jb < nstage; jb += NW) {
      const int slot = cslot;
      const uint32_t par = cphase;
      if (++cslot == NS) {
        cslot = 0;
        cphase ^= 1;
      }
      const uint32_t fb = full0 + 8 * (warp * NS + slot);
      int ok = mbar_wait(fb, par, abort_flag, a.err);
      ok = __all_sync(kFull, ok);
      if (!ok) continue;  // aborted: keep the item/barrier sequence, skip the work (the
                          // slot is not released: the producer has stopped)
      const uint32_t kst = base_u32 + (uint32_t)((warp * NS + slot) * L::kStage);
      if constexpr (KV8) {
        // Two blocks per stage (2 jb, 2 jb + 1); a block that is absent (past the end of
        // the item) or whose id was rejected counts as having no valid token.
        const int vb = valid[warp * NS + slot];
        int nv[2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          nv[j] = ((vb >> j) & 1) ? max(0, min(kBlockSize, t1 - (t0 + (2 * jb + j) * kBlockSize)))
                                  : 0;
        if (nv[0] | nv[1]) {
          // S^T = K Q^T per block (rows: tokens tokA8, tokB8; columns: heads 2 tig, +1).
          // Tile row m of S^T holds token tokA8 (m = gid) / tokB8 (m = gid + 8), a token
          // order in which the P.V operand's four k-slots of a thread are four
          // consecutive tokens (the transposed V codes of one head_dim row).
          float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (nv[j] == 0) continue;
            const uint32_t kj = kst + (uint32_t)(j * 2 * L::kTile);
#pragma unroll
            for (int kk = 0; kk < KSTEPS; kk += 2) {
              uint32_t w[4];  // (tokA, kk), (tokB, kk), (tokA, kk + 1), (tokB, kk + 1)
              ldsm_x4(kj + krow8 + ((((uint32_t)kk + kstep8) ^ kkey8) << 4), w[0], w[1], w[2],
                      w[3]);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(w[2 * h], a0, a2);
                e4m3x4_to_f16x2x2(w[2 * h + 1], a1, a3);
                mma16816_f16(sc[j], a0, a1, a2, a3, qb[kk + h][0], qb[kk + h][1]);
              }
            }
          }
          float x[2][4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int i = 0; i < 4; ++i) x[j][i] = sc[j][i] * sl2;
            if (tokA8 >= nv[j]) x[j][0] = x[j][1] = -INFINITY;
            if (tokB8 >= nv[j]) x[j][2] = x[j][3] = -INFINITY;
          }
          float mx0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
          float mx1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
          }
          const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
          const float al0 = ex2_ftz(m0 - n0), al1 = ex2_ftz(m1 - n1);
          m0 = n0;
          m1 = n1;
          uint32_t p01[2], p23[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            p01[j] = pack_f16(ex2_ftz(x[j][0] - m0), ex2_ftz(x[j][1] - m1));
            p23[j] = pack_f16(ex2_ftz(x[j][2] - m0), ex2_ftz(x[j][3] - m1));
          }
          // the sum of the weights uses the rounded (f16) values that multiply V
          l0 = fmaf(l0, al0, (f16_lo(p01[0]) + f16_lo(p23[0])) + (f16_lo(p01[1]) + f16_lo(p23[1])));
          l1 = fmaf(l1, al1, (f16_hi(p01[0]) + f16_hi(p23[0])) + (f16_hi(p01[1]) + f16_hi(p23[1])));
          {
            // acc[mt][0, 1] and acc[mt][2, 3] are (head 2 tig, head 2 tig + 1) pairs
            const uint64_t al = f32x2(al0, al1);
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
              f32x2_split(mul_f32x2(f32x2(acc[mt][0], acc[mt][1]), al), acc[mt][0], acc[mt][1]);
              f32x2_split(mul_f32x2(f32x2(acc[mt][2], acc[mt][3]), al), acc[mt][2], acc[mt][3]);
            }
          }
          // O^T += V^T P^T per block, P^T as the B operand (movmatrix), V^T[d][token]
          // fragments straight from the transposed codes: head_dim rows 16 mt + gid (+8),
          // tokens 4 tig .. 4 tig + 3 = k-slots 2 tig, +1, 2 tig + 8, +9.  Codes of tokens
          // past the end of the context are masked to +0.
          auto pv8 = [&](uint32_t vst, uint32_t b0, uint32_t b1, uint32_t vmask) {
#pragma unroll
            for (int mt = 0; mt < KSTEPS; mt += 2) {
              uint32_t w[4];  // d rows (16 mt + gid, + 8) of m-tiles mt and mt + 1
              ldsm_x4(vst + (uint32_t)(mt * 256) + vrow8, w[0], w[1], w[2], w[3]);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(w[2 * h] & vmask, a0, a2);
                e4m3x4_to_f16x2x2(w[2 * h + 1] & vmask, a1, a3);
                mma16816_f16(acc[mt + h], a0, a1, a2, a3, b0, b1);
              }
            }
          };
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (nv[j] == 0) continue;
            const uint32_t b0 = movmatrix_t(p01[j]), b1 = movmatrix_t(p23[j]);
            const uint32_t vst = kst + (uint32_t)(j * 2 * L::kTile + L::kTile);
            if (nv[j] == kBlockSize) {
              pv8(vst, b0, b1, 0xffffffffu);  // a full block: no mask (the AND folds away)
            } else {
              uint32_t vmask = 0u;
#pragma unroll
              for (int b = 0; b < 4; ++b)
                if (4 * tig + b < nv[j]) vmask |= 0xffu << (8 * b);
              pv8(vst, b0, b1, vmask);
            }
          }
        }
      } else {
        const int nvalid = min(kBlockSize, t1 - (t0 + jb * kBlockSize));
        const uint32_t vst = kst + L::kTile;
        if (valid[warp * NS + slot]) {
          if (nvalid < kBlockSize) {
            // Rows past the end of the context may hold anything (even NaN): zero them in
            // V so that their zero weights contribute exactly nothing.
            unsigned char *vrow = base + (vst - base_u32);
            {
              const int nz = (kBlockSize - nvalid) * (D / 8);
              for (int i = lane; i < nz; i += 32) {
                const int row = nvalid + i / (D / 8), ch = i % (D / 8);
                *reinterpret_cast<uint4 *>(vrow + (ch >> 3) * 2048 + row * 128 + (ch & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
            }
            __syncwarp();
          }
          // S^T = K Q^T  (rows: tokens gid, gid + 8; columns: heads 2 tig, 2 tig + 1)
          float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            // column 16 kk + 8 (lane >> 4): half kk / 4, chunk (2 kk + (lane >> 4)) & 7
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kst + (uint32_t)((kk >> 2) * 2048) + (koff16 ^ (uint32_t)(((2 * kk) & 7) << 4)),
                    a0, a1, a2, a3);
            mma16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
          }
          float x0 = sc[0] * a.scale_log2, x1 = sc[1] * a.scale_log2;
          float x2 = sc[2] * a.scale_log2, x3 = sc[3] * a.scale_log2;
          if (gid >= nvalid) x0 = x1 = -INFINITY;
          if (gid + 8 >= nvalid) x2 = x3 = -INFINITY;
          float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
          }
          const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
          const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
          m0 = n0;
          m1 = n1;
          const uint32_t p01 = pack_bf16(exp2f(x0 - m0), exp2f(x1 - m1));
          const uint32_t p23 = pack_bf16(exp2f(x2 - m0), exp2f(x3 - m1));
          l0 = fmaf(l0, al0, bf16_lo(p01) + bf16_lo(p23));
          l1 = fmaf(l1, al1, bf16_hi(p01) + bf16_hi(p23));
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            acc[mt][0] *= al0;
            acc[mt][1] *= al1;
            acc[mt][2] *= al0;
            acc[mt][3] *= al1;
          }
          // P^T as the B operand of O^T += V^T P^T.
          const uint32_t b0 = movmatrix_t(p01), b1 = movmatrix_t(p23);
          const int j4 = lane >> 3;
          const int tok = (lane & 7) + ((j4 >> 1) << 3);
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vst + tile_off(tok, 16 * mt + ((j4 & 1) << 3)), a0, a1, a2, a3);
            mma16816(acc[mt], a0, a1, a2, a3, b0, b1);
          }
          if (nvalid < kBlockSize)  // generic writes above, async-proxy writes next
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
      __syncwarp();
      if (jb + NW < nstage) {
        if (lane == 0) mbar_arrive(empty0 + 8 * (warp * NS + slot));
      } else {
        held = (int)slot;  // the warp's last stage of the item: kept for its merge state
      }
    }

    // ---- merge the NW warp states of this item; take the next item meanwhile ----
    // Each warp that consumed a stage of the item keeps its last stage and writes its
    // state there -- per lane the accumulator tile acc[mt][0..3] as float4 chunk mt and
    // (m0, m1, l0, l1) as chunk KSTEPS, chunk-major (chunk c of lane i at 512 c + 16 i),
    // so a warp's 16-byte accesses hit distinct banks -- and publishes the stage address.
    // Warp w then merges m-tiles w, w + NW, ... of every warp's state and writes that
    // slice of the item's output; the held stages are released after a second barrier.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, off);
      l1 += __shfl_xor_sync(kFull, l1, off);
    }
    const uint32_t held_at =
        held >= 0 ? base_u32 + (uint32_t)((warp * NS + held) * L::kStage) : ~0u;
    if (held >= 0) {
      const uint32_t at = held_at + (uint32_t)lane * 16u;
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt)
        sts128(at + (uint32_t)(mt * 512), acc[mt][0], acc[mt][1], acc[mt][2], acc[mt][3]);
      sts128(at + (uint32_t)(KSTEPS * 512), m0, m1, l0, l1);
    }
    if (lane == 0) state_at[warp] = held_at;
    if (threadIdx.x == 0) fetch(k + 1);
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
    const int nxt = *cons_item;
    const int4 rec_n = make_int4(cons_rec->x, cons_rec->y, cons_rec->z, cons_rec->w);
    uint32_t qn[KSTEPS][2];
    if constexpr (KV8)
      load_q_frag_f16perm<D>(qn, a, nxt < total ? nxt : 0, per_pair, rec_n, gid, tig, nxt < total);
    else
      load_q_frag<D>(qn, a, nxt < total ? nxt : 0, per_pair, rec_n, gid, tig, nxt < total);
    if (warp < KSTEPS) {
      // Weights of the warp states for this lane's two heads (2 tig, 2 tig + 1).
      uint32_t src[NW];
      float wm0[NW], wm1[NW], wl0[NW], wl1[NW];
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        src[w] = state_at[w];
        wm0[w] = wm1[w] = -INFINITY;
        wl0[w] = wl1[w] = 0.f;
        if (src[w] != ~0u) {
          src[w] += (uint32_t)lane * 16u;
          lds128(src[w] + (uint32_t)(KSTEPS * 512), wm0[w], wm1[w], wl0[w], wl1[w]);
          M0 = fmaxf(M0, wm0[w]);
          M1 = fmaxf(M1, wm1[w]);
        }
      }
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        wm0[w] = src[w] != ~0u ? exp2f(wm0[w] - M0) : 0.f;  // now the weights
        wm1[w] = src[w] != ~0u ? exp2f(wm1[w] - M1) : 0.f;
        L0 = fmaf(wl0[w], wm0[w], L0);
        L1 = fmaf(wl1[w], wm1[w], L1);
      }
      const float f0 = vsc / L0, f1 = vsc / L1;
      const bool single = rec.w == 1;
      const int p = t0 / part;
      const int hA = 2 * tig, hB = 2 * tig + 1;  // heads of this lane, within the item
      const size_t rowA = single ? ((size_t)s * a.num_q_heads + h0 + hA)
                                 : (((size_t)s * a.max_parts + p) * a.num_q_heads + h0 + hA);
      for (int mt = warp; mt < KSTEPS; mt += NW) {
        float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          if (src[w] == ~0u) continue;
          float v0, v1, v2, v3;
          lds128(src[w] + (uint32_t)(mt * 512), v0, v1, v2, v3);
          o[0] = fmaf(v0, wm0[w], o[0]);
          o[1] = fmaf(v1, wm1[w], o[1]);
          o[2] = fmaf(v2, wm0[w], o[2]);
          o[3] = fmaf(v3, wm1[w], o[3]);
        }
        // o[0]: (head hA, d0), o[1]: (hB, d0), o[2]: (hA, d0 + 8), o[3]: (hB, d0 + 8)
        const int d0 = 16 * mt + gid;
        if (single) {
          uint16_t *oa = a.out + rowA * D + d0;
          if (hA < gcnt) {
            oa[0] = f32_to_bf16(o[0] * f0);
            oa[8] = f32_to_bf16(o[2] * f0);
          }
          if (hB < gcnt) {
            oa[D] = f32_to_bf16(o[1] * f1);
            oa[D + 8] = f32_to_bf16(o[3] * f1);
          }
        } else {
          // partials stay in L2 for the merge kernel (evict-last)
          float *oa = a.part_o + rowA * D + d0;
          if (hA < gcnt) {
            st_f32_hint(oa, o[0] * f0, keep);
            st_f32_hint(oa + 8, o[2] * f0, keep);
          }
          if (hB < gcnt) {
            st_f32_hint(oa + D, o[1] * f1, keep);
            st_f32_hint(oa + D + 8, o[3] * f1, keep);
          }
        }
      }
      if (!single && warp == 0 && gid == 0) {
        if (hA < gcnt) st_f32_hint(a.part_lse + rowA, M0 + log2f(L0), keep);
        if (hB < gcnt) st_f32_hint(a.part_lse + rowA + 1, M1 + log2f(L1), keep);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
    if (held >= 0) {
      // generic writes into the stage above, async-proxy writes into it next
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * (warp * NS + held));
    }
    cur = nxt;
    rec = rec_n;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qb[kk][0] = qn[kk][0];
      qb[kk][1] = qn[kk][1];
    }
  }
}

// ------------------------------------------------------------------------------------
// Host side: tensor maps (cached) and launch.
// ------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The cache viewed as a 2-D tensor [num_blocks * Hkv * 16 rows][head_dim], boxes of
// 16 rows x 128 bytes (64 bf16 columns or 128 E4M3 codes) with the 128-byte swizzle;
// rows of only 64 bytes (E4M3, head_dim 64) are one box of 16 x 64 bytes with the
// 64-byte swizzle.  elem = 2 (bf16) or 1 (E4M3 codes).
bool encode_kv_map(CUtensorMap *m, const void *base, uint64_t rows, int D, int elem) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool narrow = D * elem < 128;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * elem};
  cuuint32_t box[2] = {(cuuint32_t)(narrow ? D : 128 / elem), (cuuint32_t)kBlockSize};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MapCache {
  struct Entry {
    const void *base;
    uint64_t rows;
    int D, elem;
    CUtensorMap map;
  };
  std::mutex mu;
  Entry e[8];
  int n = 0, next = 0;
  bool get(const void *base, uint64_t rows, int D, int elem, CUtensorMap *out) {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < n; ++i)
      if (e[i].base == base && e[i].rows == rows && e[i].D == D && e[i].elem == elem) {
        *out = e[i].map;
        return true;
      }
    CUtensorMap m;
    if (!encode_kv_map(&m, base, rows, D, elem)) return false;
    Entry &slot = e[next];
    next = (next + 1) % 8;
    if (n < 8) ++n;
    slot.base = base;
    slot.rows = rows;
    slot.D = D;
    slot.elem = elem;
    slot.map = m;
    *out = m;
    return true;
  }
};
MapCache g_maps;

template <int D, int NW, int NS, bool KV8 = false>
int launch_mma_t(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                 cudaStream_t st) {
  using L = MmaLayout<D, NW, NS, KV8>;
  // CTAs per SM (after opting the kernel into its shared memory on this device)
  static std::atomic<int> occ_slots[kMaxDevices];
  const int occ = per_device_setup(occ_slots, [] {
    const cudaError_t e = cudaFuncSetAttribute(
        attn_mma_kernel<D, NW, NS, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return -(int)e;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_mma_kernel<D, NW, NS, KV8>,
                                                      (NW + 1) * 32, L::kSmem) != cudaSuccess ||
        n < 1)
      n = 1;
    return n;
  });
  if (occ <= 0) return -occ;
  const int64_t upper = (int64_t)a.num_seqs * a.max_parts * a.num_kv_heads * a.sub_groups;
  int64_t grid = (int64_t)device_sm_count() * occ;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  return (int)launch_pdl(attn_mma_kernel<D, NW, NS, KV8>, dim3((int)grid), dim3((NW + 1) * 32),
                         (size_t)L::kSmem, st, a, tk, tv);
}

// Ring shape (consumer warps x stages per warp), overridable for tuning through the
// PKV_MMA_RING environment variable; -1 = the path's default.
int ring_choice() {
  static const int choice = [] {  // read once (thread-safe static initialisation)
    static const char *names[] = {"3x2", "8x2", "4x4", "4x3", "2x2", "2x3", "4x2", "2x4", "3x3",
                                  "1x4", "1x6"};
    const char *v = std::getenv("PKV_MMA_RING");
    int c = -1;
    for (int i = 0; v && i < (int)(sizeof(names) / sizeof(names[0])); ++i)
      if (std::strcmp(v, names[i]) == 0) c = i;
    return c;
  }();
  return choice;
}

template <bool KV8>
int launch_mma_ring(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                    cudaStream_t st) {
  // Defaults measured on GB300: bf16 (one 8 KB block per stage) 3 consumer warps x 2
  // stages, 4 CTAs per SM; E4M3 (two blocks, 8 KB, per stage) 2 x 3 (with the automatic
  // split-K size: 0.844 / 0.985 of the copy peak on the GQA-8 / long-context batches
  // against 0.834 / 0.971 for 2 x 2 in the same call).
  int c = ring_choice();
  if (c < 0) c = KV8 ? 5 : 0;
  switch (c) {
    case 1: return launch_mma_t<128, 8, 2, KV8>(a, tk, tv, st);
    case 2: return launch_mma_t<128, 4, 4, KV8>(a, tk, tv, st);
    case 3: return launch_mma_t<128, 4, 3, KV8>(a, tk, tv, st);
    case 4: return launch_mma_t<128, 2, 2, KV8>(a, tk, tv, st);
    case 5: return launch_mma_t<128, 2, 3, KV8>(a, tk, tv, st);
    case 6: return launch_mma_t<128, 4, 2, KV8>(a, tk, tv, st);
    case 7: return launch_mma_t<128, 2, 4, KV8>(a, tk, tv, st);
    case 8: return launch_mma_t<128, 3, 3, KV8>(a, tk, tv, st);
    case 9: return launch_mma_t<128, 1, 4, KV8>(a, tk, tv, st);
    case 10: return launch_mma_t<128, 1, 6, KV8>(a, tk, tv, st);
    default: return launch_mma_t<128, 3, 2, KV8>(a, tk, tv, st);
  }
}

}  // namespace

bool kv_tensor_map(CUtensorMap *out, const void *base, uint64_t rows, int D, int elem) {
  return g_maps.get(base, rows, D, elem, out);
}

int launch_attn_mma(const AttnArgs &a, int head_dim, cudaStream_t st) {
  const uint64_t rows = (uint64_t)a.num_blocks * a.num_kv_heads * kBlockSize;
  if (rows >= (1ull << 31)) return (int)cudaErrorInvalidValue;
  const int elem = a.kv8 ? 1 : 2;
  CUtensorMap tk, tv;
  if (!kv_tensor_map(&tk, a.k_cache, rows, head_dim, elem) ||
      !kv_tensor_map(&tv, a.v_cache, rows, head_dim, elem))
    return (int)cudaErrorInvalidValue;
  if (a.kv8) {
    if (head_dim == 64) return launch_mma_t<64, 4, 4, true>(a, tk, tv, st);
    if (head_dim != 128) return (int)cudaErrorInvalidValue;
    return launch_mma_ring<true>(a, tk, tv, st);
  }
  if (head_dim == 64) return launch_mma_t<64, 4, 4>(a, tk, tv, st);
  return launch_mma_ring<false>(a, tk, tv, st);
}

}  // namespace pkv
