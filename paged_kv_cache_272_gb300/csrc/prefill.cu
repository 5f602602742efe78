// Chunked-prefill attention over the paged cache, on tensor cores.
//
// A chunked prefill feeds a long prompt to the model a chunk of tokens per iteration,
// so that it does not stall the decoding requests batched with it ("Continuous
// batching and PagedAttention", section 2, continuous batching: chunked prefill is the
// first remedy listed).  Each new token attends causally ("System-level optimization",
// section 3.3, is_causal=True) over the sequence's paged cache: the token at position p
// sees tokens 0..p ("Continuous batching and PagedAttention", section 3: logical block
// -> physical block through the block table).  Its K/V are already in the cache
// (written by paged_kv_write for the chunk's slots).
//
// Many query rows share each K/V row here (L tokens x G query heads per KV head), so the
// two products are real matrix products and run as mma.sync tiles:
//  * One CTA = 4 warps owns 64 rows of one (sequence, KV head); row r is query token
//    r / G of the chunk and query head g G + r % G, so a GQA group's heads sit in
//    consecutive rows and share every K/V tile.  Each warp keeps its 16 rows of Q as
//    A fragments in registers for the whole key loop.
//  * Keys come in tiles of 64 (four 16-token blocks).  Lanes 0-3 of warp 0 each read
//    one block id from the block table and issue TMA tiled copies
//    (cp.async.bulk.tensor.2d, 128-byte swizzle) of that block's K and V head tiles
//    into a ring of stages; "full" mbarriers carry the byte counts, "empty" mbarriers
//    (one arrival per warp) free a stage for the next copy.  Every wait is bounded.
//  * S = Q K^T (16 rows x 64 keys per warp) with K fragments read by ldmatrix; scores
//    are scaled into the log2 domain, keys past a row's position are masked, and the
//    online softmax (running max and sum per row, fp32) rescales the output.  The
//    weights, rounded to bf16, are re-used in registers as the A fragments of
//    O += P V, whose V fragments ldmatrix.trans reads from the staged tile.  The row
//    sums use the same rounded weights.
//  * Row tiles are launched latest-first, so the CTAs with the longest key ranges start
//    first.
#include <cuda.h>
#include <math.h>

#include <climits>

#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kRows = 64;                        // (token, head) rows per CTA
constexpr int kKeys = 64;                        // keys per staged tile
constexpr int kTileBlocks = kKeys / kBlockSize;  // blocks per staged tile (= producer lanes)
constexpr int kWarps = kRows / 16;
constexpr unsigned kAll = 0xffffffffu;

struct PrefillArgs {
  uint16_t *out;                  // [T][Hq][D] bf16
  const uint16_t *q;              // [T][Hq][D] bf16
  const int32_t *block_tables;    // [S][MB]
  const int32_t *context_lens;    // [S] tokens after the step (chunk included)
  const int32_t *query_start;     // [S+1] first row of each sequence's chunk
  int num_seqs, num_tokens, max_blocks, num_q_heads, num_kv_heads, group, num_blocks;
  int max_query_len;              // host bound of the chunk lengths
  int row_tiles;                  // ceil(max_query_len * group / kRows)
  float scale_log2;               // scale * log2(e)
  int32_t *err;
};

template <int D, int NST>
struct PrefillLayout {
  static constexpr int kBlk = kBlockSize * D * 2;  // one block's K (or V) head tile, bytes
  static constexpr int kHalf = kTileBlocks * kBlk; // K (or V) part of a stage
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kSmem = 1024 + NST * kStage + 2 * NST * 8 + 16;
};

template <int D, int NST>
__global__ void __launch_bounds__(kWarps * 32, 2)
    prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv) {
  using Lay = PrefillLayout<D, NST>;
  constexpr int KSTEPS = D / 16, HALVES = D / 64, NT = kKeys / 8, DT = D / 8;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // the swizzle repeats every 1024 bytes
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + (base - raw) + NST * Lay::kStage);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * NST);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * NST;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int s = blockIdx.z, g = blockIdx.y;
  const int tile = a.row_tiles - 1 - (int)blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(full0 + 8 * i, kTileBlocks);
      mbar_init(empty0 + 8 * i, kWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_trigger();
  pdl_wait();

  // The sequence's chunk: rows query_start[s] .. query_start[s+1]-1, the last L of its
  // ctx tokens.  Every test below is uniform over the CTA.
  const int q0 = a.query_start[s], q1 = a.query_start[s + 1];
  const int ctx = a.context_lens[s];
  const int L = q1 - q0;
  if (q0 < 0 || L < 0 || q1 > a.num_tokens || L > a.max_query_len || L > ctx ||
      ctx > a.max_blocks * kBlockSize) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) flag_error(a.err, PKV_DEV_BAD_CONTEXT);
    return;
  }
  const int G = a.group;
  const int rows = L * G;
  const int r0 = tile * kRows;
  if (r0 >= rows) return;
  const int first_pos = ctx - L;                 // position of the chunk's first token
  const int r_last = min(r0 + kRows, rows) - 1;
  const int kv_end = first_pos + r_last / G + 1; // keys any row of this CTA sees
  const int nkt = (kv_end + kKeys - 1) / kKeys;
  __syncthreads();                               // barrier initialisation visible

  // This thread's rows (a: gid, b: gid + 8 of the warp's 16).  A row past the chunk
  // takes the last row's position and a zero query; it is computed but not stored.
  const int ra = r0 + warp * 16 + gid, rb = ra + 8;
  const bool va = ra < rows, vb = rb < rows;
  const int pos_a = first_pos + (va ? ra : r_last) / G;
  const int pos_b = first_pos + (vb ? rb : r_last) / G;
  const int warp_pos_lo = first_pos + min(r0 + warp * 16, r_last) / G;

  uint32_t qa[KSTEPS][4];
  {
    const uint32_t *qpa = reinterpret_cast<const uint32_t *>(
        a.q + ((size_t)(q0 + ra / G) * a.num_q_heads + g * G + ra % G) * D);
    const uint32_t *qpb = reinterpret_cast<const uint32_t *>(
        a.q + ((size_t)(q0 + rb / G) * a.num_q_heads + g * G + rb % G) * D);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qa[kk][0] = va ? qpa[8 * kk + tig] : 0u;
      qa[kk][1] = vb ? qpb[8 * kk + tig] : 0u;
      qa[kk][2] = va ? qpa[8 * kk + 4 + tig] : 0u;
      qa[kk][3] = vb ? qpb[8 * kk + 4 + tig] : 0u;
    }
  }

  // Producer step (warp 0, lanes 0..3): lane b stages block b of key tile kt.
  const int32_t *table = a.block_tables + (size_t)s * a.max_blocks;
  auto issue = [&](int kt) {
    const int st = kt % NST;
    const int tok = kt * kKeys + lane * kBlockSize;
    int blk = -1;
    if (tok < kv_end) {
      blk = table[tok / kBlockSize];
      if (blk < 0 || blk >= a.num_blocks) {
        flag_error(a.err, PKV_DEV_BAD_BLOCK);
        blk = -1;
      }
    }
    const uint32_t bar = full0 + 8 * st;
    mbar_arrive_expect_tx(bar, blk >= 0 ? 2u * Lay::kBlk : 0u);
    if (blk >= 0) {
      const int row = (blk * a.num_kv_heads + g) * kBlockSize;
      const uint32_t dk = base + st * Lay::kStage + lane * Lay::kBlk;
#pragma unroll
      for (int h = 0; h < HALVES; ++h) {
        tma_load_2d(dk + h * 2048, &tk, h * 64, row, bar);
        tma_load_2d(dk + Lay::kHalf + h * 2048, &tv, h * 64, row, bar);
      }
    }
  };
  int issued = 0;  // meaningful in warp 0
  if (warp == 0) {
    issued = min(NST, nkt);
    if (lane < kTileBlocks)
      for (int kt = 0; kt < issued; ++kt) issue(kt);
  }

  float o[DT][4];
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  for (int kt = 0; kt < nkt; ++kt) {
    const int st = kt % NST;
    const uint32_t ph = (uint32_t)(kt / NST) & 1u;
    if (!mbar_wait(full0 + 8 * st, ph, abort_flag, a.err)) break;
    const uint32_t ks = base + st * Lay::kStage, vs = ks + Lay::kHalf;
    const int t0 = kt * kKeys;

    if (t0 + kKeys > kv_end) {
      // Last tile: V rows at or past kv_end (the tail of the last block, blocks not
      // staged) are set to zero so that their zero weights contribute exactly nothing.
      // Each warp clears them for itself (all write the same zeros), so no CTA barrier
      // is needed; no copy reuses this stage afterwards.
      const int z0 = kv_end - t0;
      const int nchunks = (kKeys - z0) * HALVES * 8;  // 16-byte chunks
      for (int i = lane; i < nchunks; i += 32) {
        const int r = z0 + i / (HALVES * 8), rem = i % (HALVES * 8);
        const uint32_t addr = vs + (r >> 4) * Lay::kBlk + (rem >> 3) * 2048 + (r & 15) * 128 +
                              (rem & 7) * 16;
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
      }
      __syncwarp();
    }

    // S = Q K^T for this warp's 16 rows x 64 keys.
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const int key = nt * 8 + (lane & 7);
      const uint32_t kblk = ks + (key >> 4) * Lay::kBlk;
      const int m = lane >> 3;
#pragma unroll
      for (int kp = 0; kp < KSTEPS / 2; ++kp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kblk + tile_off(key & 15, 16 * (2 * kp + (m >> 1)) + 8 * (m & 1)), b0, b1, b2,
                b3);
        mma16816(sc[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
        mma16816(sc[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2],
                 qa[2 * kp + 1][3], b2, b3);
      }
    }

    // Scale, causal mask, running max.
    const bool need_mask = t0 + kKeys - 1 > warp_pos_lo;  // uniform over the warp
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = t0 + nt * 8 + 2 * tig + j;
        float xa = sc[nt][j] * a.scale_log2, xb = sc[nt][2 + j] * a.scale_log2;
        if (need_mask) {
          if (key > pos_a) xa = -INFINITY;
          if (key > pos_b) xb = -INFINITY;
        }
        sc[nt][j] = xa;
        sc[nt][2 + j] = xb;
        mx_a = fmaxf(mx_a, xa);
        mx_b = fmaxf(mx_b, xb);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kAll, mx_a, off));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kAll, mx_b, off));
    }
    // Key 0 is visible to every row, so the running max is finite after the first tile.
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float ca = exp2f(m_a - mn_a), cb = exp2f(m_b - mn_b);
    m_a = mn_a;
    m_b = mn_b;

    // Weights -> bf16 A fragments of P V (accumulator layout = A layout, 16 keys per step).
    uint32_t pa[kKeys / 16][4];
    float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t lo = pack_bf16(exp2f(sc[nt][0] - mn_a), exp2f(sc[nt][1] - mn_a));
      const uint32_t hi = pack_bf16(exp2f(sc[nt][2] - mn_b), exp2f(sc[nt][3] - mn_b));
      ps_a += bf16_lo(lo) + bf16_hi(lo);
      ps_b += bf16_lo(hi) + bf16_hi(hi);
      pa[nt >> 1][(nt & 1) * 2] = lo;
      pa[nt >> 1][(nt & 1) * 2 + 1] = hi;
    }
    l_a = l_a * ca + ps_a;
    l_b = l_b * cb + ps_b;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      o[dt][0] *= ca;
      o[dt][1] *= ca;
      o[dt][2] *= cb;
      o[dt][3] *= cb;
    }

    // O += P V; 16 keys (one block) per k-step.
#pragma unroll
    for (int j = 0; j < kKeys / 16; ++j) {
      const int m = lane >> 3;
      const uint32_t vrow = vs + j * Lay::kBlk;
      const int r = 8 * (m & 1) + (lane & 7);
#pragma unroll
      for (int dp = 0; dp < DT / 2; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vrow + tile_off(r, 8 * (2 * dp + (m >> 1))), b0, b1, b2, b3);
        mma16816(o[2 * dp], pa[j][0], pa[j][1], pa[j][2], pa[j][3], b0, b1);
        mma16816(o[2 * dp + 1], pa[j][0], pa[j][1], pa[j][2], pa[j][3], b2, b3);
      }
    }

    // Release the stage; warp 0 refills it with tile kt + NST once every warp is done.
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    if (warp == 0 && kt + NST < nkt) {
      if (!mbar_wait(empty0 + 8 * st, ph, abort_flag, a.err)) break;
      if (lane < kTileBlocks) issue(kt + NST);
      ++issued;
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // A wait gave up: let the copies still in flight land before the CTA exits.
    if (warp == 0 && lane == 0)
      for (int kt = max(0, issued - NST); kt < issued; ++kt)
        mbar_drain(full0 + 8 * (kt % NST), (uint32_t)(kt / NST) & 1u);
    return;
  }

#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_a += __shfl_xor_sync(kAll, l_a, off);
    l_b += __shfl_xor_sync(kAll, l_b, off);
  }
  const float ia = 1.f / l_a, ib = 1.f / l_b;
  if (va) {
    uint32_t *oa = reinterpret_cast<uint32_t *>(
        a.out + ((size_t)(q0 + ra / G) * a.num_q_heads + g * G + ra % G) * D);
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) oa[4 * dt + tig] = pack_bf16(o[dt][0] * ia, o[dt][1] * ia);
  }
  if (vb) {
    uint32_t *ob = reinterpret_cast<uint32_t *>(
        a.out + ((size_t)(q0 + rb / G) * a.num_q_heads + g * G + rb % G) * D);
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) ob[4 * dt + tig] = pack_bf16(o[dt][2] * ib, o[dt][3] * ib);
  }
}

template <int D, int NST>
int launch_prefill_t(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                     cudaStream_t st) {
  using Lay = PrefillLayout<D, NST>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        prefill_kernel<D, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmem);
    if (e != cudaSuccess) return (int)e;
    attr_set = true;
  }
  return (int)launch_pdl(prefill_kernel<D, NST>,
                         dim3((unsigned)a.row_tiles, (unsigned)a.num_kv_heads,
                              (unsigned)a.num_seqs),
                         dim3(kWarps * 32), (size_t)Lay::kSmem, st, a, tk, tv);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int paged_attention_prefill(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                                       const uint16_t *v_cache, const int32_t *block_tables,
                                       const int32_t *context_lens, const int32_t *query_start,
                                       int num_seqs, int num_tokens, int max_blocks_per_seq,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, float scale,
                                       int max_query_len, int32_t *err_flag, void *stream) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return PKV_ERR_NULL;
  if (block_size != kBlockSize) return PKV_ERR_BLOCK_SIZE;
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || max_blocks_per_seq <= 0 ||
      num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      num_q_heads % num_kv_heads != 0 || (head_dim != 64 && head_dim != 128) ||
      num_seqs > 65535 || num_kv_heads > 65535 || !(scale > 0.f))
    return PKV_ERR_SHAPE;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ALIGN;
  const int group = num_q_heads / num_kv_heads;
  const int64_t tiles = ((int64_t)max_query_len * group + kRows - 1) / kRows;
  const uint64_t cache_rows = (uint64_t)num_blocks * num_kv_heads * kBlockSize;
  if (tiles > INT_MAX || cache_rows >= (1ull << 31)) return PKV_ERR_SHAPE;
  if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PKV_OK;

  PrefillArgs a;
  a.out = out;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.query_start = query_start;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_blocks = max_blocks_per_seq;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.num_blocks = num_blocks;
  a.max_query_len = max_query_len;
  a.row_tiles = (int)tiles;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.err = err_flag;

  CUtensorMap tk, tv;
  if (!kv_tensor_map(&tk, k_cache, cache_rows, head_dim, 2) ||
      !kv_tensor_map(&tv, v_cache, cache_rows, head_dim, 2))
    return PKV_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rc = head_dim == 128 ? launch_prefill_t<128, 3>(a, tk, tv, st)
                                 : launch_prefill_t<64, 4>(a, tk, tv, st);
  return rc == 0 ? PKV_OK : PKV_ERR_CUDA;
}
