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

#include <atomic>
#include <climits>
#include <cstdlib>
#include <cstring>

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
  static std::atomic<int> ready[kMaxDevices];  // the kernel's shared-memory opt-in, per device
  const int r = per_device_setup(ready, [] {
    const cudaError_t e = cudaFuncSetAttribute(
        prefill_kernel<D, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmem);
    return e == cudaSuccess ? 1 : -(int)e;
  });
  if (r <= 0) return -r;
  return (int)launch_pdl(prefill_kernel<D, NST>,
                         dim3((unsigned)a.row_tiles, (unsigned)a.num_kv_heads,
                              (unsigned)a.num_seqs),
                         dim3(kWarps * 32), (size_t)Lay::kSmem, st, a, tk, tv);
}


// ------------------------------------------------------------------------------------
// tcgen05 variant (head_dim 64 and 128): the same arithmetic on the 5th-generation tensor
// cores.  One CTA = 128 (token, head) rows of one (sequence, KV head), eight warps:
//  * warps 0-3 ("softmax"): thread t owns row t -- TMEM lane t of the S and O
//    accumulators and row t of the Q tile in shared memory.  They stage Q, read each
//    S tile from TMEM (tcgen05.ld), mask, keep the running max and sum (the sum in fp32
//    from the unrounded weights; packed f32x2 arithmetic), write the bf16 weights P over
//    the tile's S columns in TMEM (tcgen05.st; or to shared memory), rescale O in TMEM
//    when the running max grows by more than 8 in the log2 domain (the sum and O always
//    share one reference, so a stale reference only needs to keep the weights below
//    2^8), and finally normalise O.
//  * warp 4 ("S", one elected lane): S_j = Q K_j^T (M 128, N 64, K 128) into one of two
//    TMEM S buffers by tcgen05.mma from shared-memory descriptors, once K_j has landed
//    and the buffer is free; tcgen05.commit signals S ready and the K slot free.
//  * warp 7 ("P V", one elected lane): O += P_j V_j (M 128, N 128, K 64) into the TMEM
//    O accumulator once P_j and V_j are ready; commits O ready, the V slot free and
//    (P in TMEM) the S buffer free.  A tcgen05.mma takes about 70 cycles to issue from
//    one thread (an S product's eight take longer than they take to run), so the two
//    kinds of product are issued by different warps and neither waits behind the other.
//  * warps 5 and 6 ("tma"): lanes 0-3 load the four K (warp 5) or V (warp 6) blocks of
//    each 64-key tile into their own two-slot ring (TMA tiled copies as in the mma.sync
//    variant), reading the block ids one tile ahead.
// Shared-memory tiles use the 128-byte swizzle that TMA writes: Q [head_dim / 64 halves]
// [128 rows][128 B], P [128 rows][64 keys x 2 B], K and V tiles [head_dim / 64 halves]
// [64 keys][128 B] per ring slot.  Q, K (both K-major) and P (K-major) enter as canonical
// SW128 operands (8-row groups 1024 B apart); V enters as the MN-major operand of
// O += P V (64-column chunks 8192 B apart, 8-key groups 1024 B apart).  TMEM: S buffers
// at columns 0 and 64, O at columns 128 .. 128 + head_dim - 1 (256 allocated).  At
// head_dim 64 a score product is M 128 x N 64 x K 64 and O has 64 columns; the rest is
// the same.

constexpr int kTcRows = 128;
constexpr int kTcWarps = 8;
constexpr uint32_t kTmemCols = 256;

// Shared memory is requested 1024-byte aligned, so that two CTAs fit on one SM (2 x 112
// KB at head_dim 128; 2 x 78 KB at head_dim 64, where the tiles need 64 KB, so that a
// third CTA does not wait for TMEM); a CTA whose window is not aligned reports an error
// and exits
// without touching it.  K and V tiles live in separate two-slot rings: a K slot is
// released as soon as its scores are computed, a V slot once its P V product is done,
// so the next K tiles load while the current softmax runs.
template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;             // 64-column halves of head_dim
  static constexpr int kQHalf = kTcRows * 128;       // 16 KB: 128 rows x 64 dims
  static constexpr int kKHalf = kKeys * 128;         // 8 KB: 64 keys x 64 dims
  static constexpr int kQ = 0;                       // D 128: 32 KB, D 64: 16 KB
  static constexpr int kP = kHalves * kQHalf;        // 16 KB
  static constexpr int kSlot = kHalves * kKHalf;     // one K or V tile
  static constexpr int kK = kP + 16384;              // 2 slots
  static constexpr int kV = kK + 2 * kSlot;          // 2 slots
  static constexpr int kBars = kV + 2 * kSlot;
  static constexpr int kNumBars = 18;                // K full/empty x2, V full/empty x2,
                                                     // S full/free x2, P full x2, O done,
                                                     // final, P V done x2
  static constexpr int kSmem = kBars + kNumBars * 8 + 16;
  // Requested per CTA: at least 78 KB, so that no more than two CTAs share an SM (each
  // holds 256 TMEM columns; a third would wait in its allocation).
  static constexpr int kSmemLaunch = kSmem > 78 * 1024 ? kSmem : 78 * 1024;
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator, M x N.
__host__ __device__ constexpr uint32_t bf16_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with the A operand (M x K: one row per TMEM lane, two 16-bit elements per
// 32-bit column, the lower k in the low half) read from tensor memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 2^x by the MUFU ex2 instruction (subnormal results flush to zero: such weights are
// below 2^-126 of the row maximum's).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (one instruction).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}

template <int D, bool PT>
__global__ void __launch_bounds__(kTcWarps * 32, 2)
    prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv) {
  using Lay = TcLayout<D>;
  constexpr int H = Lay::kHalves;
  extern __shared__ __align__(1024) unsigned char smem_tc[];
  const uint32_t base = smem_u32(smem_tc);
  if (base & 1023u) {  // the swizzled tiles need a 1024-byte aligned window
    if (threadIdx.x == 0) flag_error(a.err, PKV_DEV_LAYOUT);
    return;
  }
  unsigned char *gbase = smem_tc;
  const uint32_t sQ = base + Lay::kQ, sP = base + Lay::kP;
  const uint32_t sK = base + Lay::kK, sV = base + Lay::kV;
  const uint32_t k_full = base + Lay::kBars, k_empty = k_full + 16;
  const uint32_t v_full = k_empty + 16, v_empty = v_full + 16;
  const uint32_t s_full = v_empty + 16, s_free = s_full + 16, p_full = s_free + 16;
  const uint32_t o_done = p_full + 16, fin = o_done + 8, pv_done = fin + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + Lay::kBars + Lay::kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, g = blockIdx.y;
  const int tile = a.row_tiles - 1 - (int)blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full + 8 * i, kTileBlocks);
      mbar_init(k_empty + 8 * i, 1);
      mbar_init(v_full + 8 * i, kTileBlocks);
      mbar_init(v_empty + 8 * i, 1);
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_free + 8 * i, 4);
      mbar_init(p_full + 8 * i, 4);
      mbar_init(pv_done + 8 * i, 1);
    }
    mbar_init(o_done, 1);
    mbar_init(fin, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_trigger();
  pdl_wait();

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
  const int r0 = tile * kTcRows;
  if (r0 >= rows) return;
  const int first_pos = ctx - L;
  const int r_last = min(r0 + kTcRows, rows) - 1;
  const int kv_end = first_pos + r_last / G + 1;
  const int nkt = (kv_end + kKeys - 1) / kKeys;

  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;  // S buffers at columns 0 and 64, O after

  if (warp < 4) {
    // ---------------- softmax warps: thread t owns row t ----------------
    const int t = threadIdx.x;
    const int r = r0 + t;
    const bool valid = r < rows;
    const int pos = first_pos + (valid ? r : r_last) / G;
    const int warp_pos_lo = first_pos + min(r0 + warp * 32, r_last) / G;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint16_t *orow = a.out + ((size_t)(q0 + r / G) * a.num_q_heads + g * G + r % G) * D;
    {
      const uint4 *qrow = reinterpret_cast<const uint4 *>(
          a.q + ((size_t)(q0 + r / G) * a.num_q_heads + g * G + r % G) * D);
#pragma unroll
      for (int c = 0; c < 8 * H; ++c) {
        const uint4 v = valid ? qrow[c] : make_uint4(0u, 0u, 0u, 0u);
        st_shared_v4(sQ + (c >> 3) * Lay::kQHalf + t * 128 + (((c & 7) ^ (t & 7)) << 4), v.x,
                     v.y, v.z, v.w);
      }
    }
    fence_proxy_async();
    named_bar_sync(1, 160);

    float m = -INFINITY, l = 0.f;
    int o_seen = -1;  // last P V product whose completion this thread has observed
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int sb = j & 1;
      const int t0 = j * kKeys;
      if (!mbar_wait(s_full + 8 * sb, (uint32_t)(j >> 1) & 1u, abort_flag, a.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x[64];
      {
        uint32_t (&x0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[0]);
        uint32_t (&x1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[32]);
        tmem_ld32(tS + 64 * sb + lane_base, x0);
        tmem_ld32(tS + 64 * sb + 32 + lane_base, x1);
        tmem_wait_ld();
      }
      if (!PT) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free + 8 * sb);
      }

      // Raw scores; keys past the row's position become -inf (diagonal tiles only).  The
      // max is taken on raw scores (scale > 0), the weights are 2^(scale s - m) by one
      // packed FFMA per two scores and one ex2 each.
      // (Eight independent three-input max chains and four packed sum chains keep the
      // reductions short.)
      const bool need_mask = t0 + kKeys - 1 > warp_pos_lo;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (t0 + c > pos) x[c] = __float_as_uint(-INFINITY);
      }
      float mxv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mxv[c] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 2)
        mxv[(c >> 1) & 7] =
            max3f(mxv[(c >> 1) & 7], __uint_as_float(x[c]), __uint_as_float(x[c + 1]));
      float mx = max3f(max3f(mxv[0], mxv[1], mxv[2]), max3f(mxv[3], mxv[4], mxv[5]),
                       fmaxf(mxv[6], mxv[7]));
      mx *= a.scale_log2;
      if (j == 0) {
        m = mx;  // key 0 is visible to every row
      } else {
        const bool need = mx > m + 8.f;
        if (__any_sync(kAll, need)) {
          if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
          o_seen = j - 1;
          tc_fence_after();
          const float mn = need ? mx : m;
          const float corr = fast_exp2(m - mn);
          m = mn;
          l *= corr;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * cc + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(tO + 32 * cc + lane_base, o);
          }
          tmem_wait_st();
        }
      }
      uint32_t pk[32];
      uint64_t ps2[4];
      const uint64_t sl2 = f32x2(a.scale_log2, a.scale_log2), nm2 = f32x2(-m, -m);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float e0, e1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])),
                              sl2, nm2),
                    e0, e1);
        const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
        const uint64_t pp = f32x2(p0, p1);
        ps2[c & 3] = c < 4 ? pp : add_f32x2(ps2[c & 3], pp);
        pk[c] = pack_bf16(p0, p1);
      }
      {
        float s0, s1;
        f32x2_split(add_f32x2(add_f32x2(ps2[0], ps2[1]), add_f32x2(ps2[2], ps2[3])), s0, s1);
        l += s0 + s1;
      }
      // The P tile is free once the previous P V product has completed.
      if (!PT && j >= 1 && o_seen < j - 1) {
        if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        o_seen = j - 1;
      }
      if (t0 + kKeys > kv_end) {
        // Last tile: V rows at or past kv_end (tail of the last block, blocks not staged)
        // are set to zero so that their zero weights contribute exactly nothing.
        if (!mbar_wait(v_full + 8 * (j & 1), (uint32_t)(j >> 1) & 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        const uint32_t vst = sV + (j & 1) * Lay::kSlot;
        const int z0 = kv_end - t0;
        for (int i = t; i < (kKeys - z0) * 8 * H; i += 128) {
          const int row = z0 + i / (8 * H), rem = i % (8 * H);
          st_shared_v4(vst + (rem >> 3) * Lay::kKHalf + row * 128 + (rem & 7) * 16, 0u, 0u, 0u,
                       0u);
        }
      }
      if (PT) {
        // P overwrites the first 32 columns of this tile's S buffer (already read).
        if (t0 + kKeys > kv_end) fence_proxy_async();  // the zeroed V rows
        tmem_st32(tS + 64 * sb + lane_base, pk);
        tmem_wait_st();
      } else {
        const uint32_t prow = sP + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(prow + ((c ^ (t & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                       pk[4 * c + 3]);
        fence_proxy_async();
      }
      tc_fence_before();
      __syncwarp();
      // Two P barriers (by tile parity): without the P-tile wait above (P in tensor
      // memory) the softmax may finish tile j + 1 before the P V warp has seen tile j.
      if (lane == 0) mbar_arrive(p_full + 8 * sb);
    }
    // Every product has completed once the P V warp's final commit fires.
    if (ok && !mbar_wait(fin, 0u, abort_flag, a.err)) ok = false;
    if (ok && !*abort_flag) {
      tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc + lane_base, o);
        tmem_wait_ld();
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * cc);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(
                pack_bf16(__uint_as_float(o[8 * e]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv));
        }
      }
    }
    tc_fence_before();
  } else if (warp == 4) {
    // ---------------- S warp: lane 0 issues the score products ----------------
    // S_j goes into TMEM buffer j & 1 once K_j has landed and that buffer is free (tile
    // j - 2's scores were read and, with P in tensor memory, its P V product -- which
    // reads P from that buffer -- is done).  The P V products are issued by warp 7, so
    // neither kind of product waits behind the other's issue.
    named_bar_sync(1, 160);
    tc_fence_after();
    constexpr uint32_t idS = bf16_idesc(kTcRows, kKeys, false);
    int js = 0;
    for (; js < nkt; ++js) {
      const int sb = js & 1;
      int ok = 1;
      if (lane == 0)
        ok = mbar_spin_wait(k_full + 8 * sb, (uint32_t)(js >> 1) & 1u, abort_flag, a.err) &&
             (js < 2 || mbar_spin_wait((PT ? pv_done : s_free) + 8 * sb,
                                       (uint32_t)((js - 2) >> 1) & 1u, abort_flag, a.err));
      if (!__shfl_sync(kAll, ok, 0)) break;
      tc_fence_after();
      const uint32_t kst = sK + sb * Lay::kSlot;
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma(tS + 64 * sb,
                 sw128_desc(sQ + (kk >> 2) * Lay::kQHalf + (kk & 3) * 32, 16, 1024),
                 sw128_desc(kst + (kk >> 2) * Lay::kKHalf + (kk & 3) * 32, 16, 1024), idS,
                 kk > 0 ? 1u : 0u);
        tc_commit(s_full + 8 * sb);
        tc_commit(k_empty + 8 * sb);
      }
      __syncwarp();
    }
    // The score products this thread issued have completed once the last one's commit
    // fires (a commit tracks every earlier product of its thread).
    if (lane == 0 && js > 0) mbar_drain(s_full + 8 * ((js - 1) & 1), (uint32_t)((js - 1) >> 1) & 1u);
    __syncwarp();
    tc_fence_before();
  } else if (warp == 7) {
    // ---------------- P V warp: lane 0 issues O += P_j V_j ----------------
    tc_fence_after();
    constexpr uint32_t idO = bf16_idesc(kTcRows, D, true);
    for (int jp = 0; jp < nkt; ++jp) {
      int ok = 1;
      if (lane == 0)
        ok = mbar_spin_wait(p_full + 8 * (jp & 1), (uint32_t)(jp >> 1) & 1u, abort_flag, a.err) &&
             mbar_spin_wait(v_full + 8 * (jp & 1), (uint32_t)(jp >> 1) & 1u, abort_flag, a.err);
      if (!__shfl_sync(kAll, ok, 0)) break;
      tc_fence_after();
      const uint32_t vst = sV + (jp & 1) * Lay::kSlot;
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k) {
          if (PT)
            tc_mma_ts(tO, tS + 64 * (jp & 1) + 8 * k,
                      sw128_desc(vst + 2048 * k, Lay::kKHalf, 1024), idO,
                      (jp > 0 || k > 0) ? 1u : 0u);
          else
            tc_mma(tO, sw128_desc(sP + 32 * k, 16, 1024),
                   sw128_desc(vst + 2048 * k, Lay::kKHalf, 1024), idO,
                   (jp > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(o_done);
        tc_commit(v_empty + 8 * (jp & 1));
        if (PT) tc_commit(pv_done + 8 * (jp & 1));
      }
      __syncwarp();
    }
    // Every P V product has completed once `fin` fires; the score products before them
    // had to (each P V reads the softmax of its scores).
    if (lane == 0) tc_commit(fin);
    __syncwarp();
    mbar_drain(fin, 0);
    tc_fence_before();
  } else {
    // ---------------- producer warps: warp 5 stages K, warp 6 V; lane b block b ----------------
    const int32_t *table = a.block_tables + (size_t)s * a.max_blocks;
    const bool is_v = warp == 6;
    const uint32_t full = is_v ? v_full : k_full, empty = is_v ? v_empty : k_empty;
    const uint32_t ring = is_v ? sV : sK;
    const CUtensorMap *map = is_v ? &tv : &tk;
    int issued = 0;
    if (lane < kTileBlocks) {
      // block ids are read one tile ahead, so their latency overlaps the slot waits
      int next = lane * kBlockSize < kv_end ? table[lane] : INT_MIN;
      for (int j = 0; j < nkt; ++j) {
        const int slot = j & 1;
        int blk = next;
        const int tok_n = (j + 1) * kKeys + lane * kBlockSize;
        next = (j + 1 < nkt && tok_n < kv_end) ? table[tok_n / kBlockSize] : INT_MIN;
        if (j >= 2 &&
            !mbar_wait(empty + 8 * slot, (uint32_t)((j - 2) >> 1) & 1u, abort_flag, a.err))
          break;
        if (blk != INT_MIN && (blk < 0 || blk >= a.num_blocks)) {
          flag_error(a.err, PKV_DEV_BAD_BLOCK);
          blk = INT_MIN;
        }
        const uint32_t bar = full + 8 * slot;
        // one head tile: H boxes of 16 rows x 64 columns
        mbar_arrive_expect_tx(bar, blk != INT_MIN ? 2048u * H : 0u);
        if (blk != INT_MIN) {
          const int row = (blk * a.num_kv_heads + g) * kBlockSize;
          const uint32_t dst = ring + slot * Lay::kSlot + lane * 2048;
#pragma unroll
          for (int h = 0; h < H; ++h) tma_load_2d(dst + h * Lay::kKHalf, map, 64 * h, row, bar);
        }
        issued = j + 1;
      }
    }
    __syncwarp();
    // If a wait gave up, let the copies still in flight land before the CTA exits.
    if (lane == 0 && *abort_flag)
      for (int j = max(0, issued - 2); j < issued; ++j)
        mbar_drain(full + 8 * (j & 1), (uint32_t)(j >> 1) & 1u);
  }

  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------------------------
// Separate-P variant (PKV_PREFILL_TC_SEP): the same CTA, warps and rings as the kernel
// above, with another TMEM layout (256 columns): one S buffer at columns 0..63, P (bf16
// pairs) at 64..95, the first 64 head-dim columns of Q at 96..127 and O at 128.  S is
// free again as soon as the softmax has read it into registers, so the next score
// product is issued while the softmax of this tile runs (it no longer waits for the
// P V product that read P out of S's columns), and P's one buffer is free once the
// previous P V product has completed -- well before the softmax needs it again.  The
// score products take their A operand for head-dim columns 0..63 from TMEM (only the K
// tile is read from shared memory there) and for 64..127 from shared memory.
// Shared memory: Q's head-dim columns 64..127 (D 128 only), then NS-slot K and V rings.
template <int D, int NS>
struct SepLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kTcRows * 128;           // 16 KB: 128 rows x 64 dims
  static constexpr int kKHalf = kKeys * 128;             // 8 KB: 64 keys x 64 dims
  static constexpr int kSlot = kHalves * kKHalf;         // one K or V tile
  static constexpr int kQ = 0;
  static constexpr int kK = (kHalves - 1) * kQHalf;
  static constexpr int kV = kK + NS * kSlot;
  static constexpr int kBars = kV + NS * kSlot;
  static constexpr int kNumBars = 4 * NS + 5;  // K/V full and empty [NS]; S full, S free,
                                               // P full, O done, final
  static constexpr int kSmem = kBars + kNumBars * 8 + 16;
  // at least 78 KB, so that no more than two CTAs share an SM (256 TMEM columns each)
  static constexpr int kSmemLaunch = kSmem > 78 * 1024 ? kSmem : 78 * 1024;
};

template <int D, int NS>
__global__ void __launch_bounds__(kTcWarps * 32, 2)
    prefill_tcs_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv) {
  using Lay = SepLayout<D, NS>;
  constexpr int H = Lay::kHalves;
  extern __shared__ __align__(1024) unsigned char smem_tc[];
  const uint32_t base = smem_u32(smem_tc);
  if (base & 1023u) {  // the swizzled tiles need a 1024-byte aligned window
    if (threadIdx.x == 0) flag_error(a.err, PKV_DEV_LAYOUT);
    return;
  }
  const uint32_t sQ = base + Lay::kQ;
  const uint32_t sK = base + Lay::kK, sV = base + Lay::kV;
  const uint32_t k_full = base + Lay::kBars, k_empty = k_full + 8 * NS;
  const uint32_t v_full = k_empty + 8 * NS, v_empty = v_full + 8 * NS;
  const uint32_t s_full = v_empty + 8 * NS, s_free = s_full + 8, p_full = s_free + 8;
  const uint32_t o_done = p_full + 8, fin = o_done + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_tc + Lay::kBars + Lay::kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, g = blockIdx.y;
  const int tile = a.row_tiles - 1 - (int)blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(k_full + 8 * i, kTileBlocks);
      mbar_init(k_empty + 8 * i, 1);
      mbar_init(v_full + 8 * i, kTileBlocks);
      mbar_init(v_empty + 8 * i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(fin, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_trigger();
  pdl_wait();

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
  const int r0 = tile * kTcRows;
  if (r0 >= rows) return;
  const int first_pos = ctx - L;
  const int r_last = min(r0 + kTcRows, rows) - 1;
  const int kv_end = first_pos + r_last / G + 1;
  const int nkt = (kv_end + kKeys - 1) / kKeys;

  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tP = tmem + 64, tQ = tmem + 96, tO = tmem + 128;

  if (warp < 4) {
    // ---------------- softmax warps: thread t owns row t ----------------
    const int t = threadIdx.x;
    const int r = r0 + t;
    const bool valid = r < rows;
    const int pos = first_pos + (valid ? r : r_last) / G;
    const int warp_pos_lo = first_pos + min(r0 + warp * 32, r_last) / G;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint16_t *orow = a.out + ((size_t)(q0 + r / G) * a.num_q_heads + g * G + r % G) * D;
    {
      // Q: head-dim columns 0..63 into TMEM (row t = lane t of this warp's quarter, two
      // bf16 per column, the lower column in the low half), 64..127 into shared memory.
      const uint4 *qrow = reinterpret_cast<const uint4 *>(
          a.q + ((size_t)(q0 + r / G) * a.num_q_heads + g * G + r % G) * D);
      uint32_t qt[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = valid ? qrow[c] : make_uint4(0u, 0u, 0u, 0u);
        qt[4 * c] = v.x, qt[4 * c + 1] = v.y, qt[4 * c + 2] = v.z, qt[4 * c + 3] = v.w;
      }
      tmem_st32(tQ + lane_base, qt);
#pragma unroll
      for (int c = 8; c < 8 * H; ++c) {
        const uint4 v = valid ? qrow[c] : make_uint4(0u, 0u, 0u, 0u);
        st_shared_v4(sQ + t * 128 + (((c & 7) ^ (t & 7)) << 4),
                     v.x, v.y, v.z, v.w);
      }
      tmem_wait_st();
    }
    fence_proxy_async();
    tc_fence_before();
    named_bar_sync(1, 160);

    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int t0 = j * kKeys;
      if (!mbar_wait(s_full, (uint32_t)j & 1u, abort_flag, a.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x[64];
      {
        uint32_t (&x0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[0]);
        uint32_t (&x1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[32]);
        tmem_ld32(tS + lane_base, x0);
        tmem_ld32(tS + 32 + lane_base, x1);
        tmem_wait_ld();
      }
      // S has been read: the next score product may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);

      // Raw scores; keys past the row's position become -inf (diagonal tiles only).
      const bool need_mask = t0 + kKeys - 1 > warp_pos_lo;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (t0 + c > pos) x[c] = __float_as_uint(-INFINITY);
      }
      float mxv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mxv[c] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 2)
        mxv[(c >> 1) & 7] =
            max3f(mxv[(c >> 1) & 7], __uint_as_float(x[c]), __uint_as_float(x[c + 1]));
      float mx = max3f(max3f(mxv[0], mxv[1], mxv[2]), max3f(mxv[3], mxv[4], mxv[5]),
                       fmaxf(mxv[6], mxv[7]));
      mx *= a.scale_log2;
      bool p_free = j == 0;  // P's buffer: free once P V j - 1 has completed
      if (j == 0) {
        m = mx;  // key 0 is visible to every row
      } else {
        const bool need = mx > m + 8.f;
        if (__any_sync(kAll, need)) {
          if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
          p_free = true;
          tc_fence_after();
          const float mn = need ? mx : m;
          const float corr = fast_exp2(m - mn);
          m = mn;
          l *= corr;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * cc + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(tO + 32 * cc + lane_base, o);
          }
          tmem_wait_st();
        }
      }
      uint32_t pk[32];
      uint64_t ps2[4];
      const uint64_t sl2 = f32x2(a.scale_log2, a.scale_log2), nm2 = f32x2(-m, -m);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float e0, e1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])),
                              sl2, nm2),
                    e0, e1);
        const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
        const uint64_t pp = f32x2(p0, p1);
        ps2[c & 3] = c < 4 ? pp : add_f32x2(ps2[c & 3], pp);
        pk[c] = pack_bf16(p0, p1);
      }
      {
        float s0, s1;
        f32x2_split(add_f32x2(add_f32x2(ps2[0], ps2[1]), add_f32x2(ps2[2], ps2[3])), s0, s1);
        l += s0 + s1;
      }
      if (t0 + kKeys > kv_end) {
        // Last tile: V rows at or past kv_end (tail of the last block, blocks not staged)
        // are set to zero so that their zero weights contribute exactly nothing.
        if (!mbar_wait(v_full + 8 * (j % NS), (uint32_t)(j / NS) & 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        const uint32_t vst = sV + (j % NS) * Lay::kSlot;
        const int z0 = kv_end - t0;
        for (int i = t; i < (kKeys - z0) * 8 * H; i += 128) {
          const int row = z0 + i / (8 * H), rem = i % (8 * H);
          st_shared_v4(vst + (rem >> 3) * Lay::kKHalf + row * 128 + (rem & 7) * 16, 0u, 0u, 0u,
                       0u);
        }
        fence_proxy_async();
      }
      if (!p_free) {
        if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tP + lane_base, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // Every product has completed once the P V warp's final commit fires.
    if (ok && !mbar_wait(fin, 0u, abort_flag, a.err)) ok = false;
    if (ok && !*abort_flag) {
      tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc + lane_base, o);
        tmem_wait_ld();
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * cc);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(
                pack_bf16(__uint_as_float(o[8 * e]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv));
        }
      }
    }
    tc_fence_before();
  } else if (warp == 4) {
    // ---------------- S warp: lane 0 issues S_j = Q K_j^T ----------------
    named_bar_sync(1, 160);
    tc_fence_after();
    constexpr uint32_t idS = bf16_idesc(kTcRows, kKeys, false);
    int js = 0;
    for (; js < nkt; ++js) {
      const int sb = js % NS;
      int ok = 1;
      if (lane == 0)
        ok = mbar_spin_wait(k_full + 8 * sb, (uint32_t)(js / NS) & 1u, abort_flag, a.err) &&
             (js < 1 || mbar_spin_wait(s_free, (uint32_t)(js - 1) & 1u, abort_flag, a.err));
      if (!__shfl_sync(kAll, ok, 0)) break;
      tc_fence_after();
      const uint32_t kst = sK + sb * Lay::kSlot;
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t bdesc = sw128_desc(kst + (kk >> 2) * Lay::kKHalf + (kk & 3) * 32, 16, 1024);
          if (kk < 4)  // head-dim columns 0..63: Q from TMEM
            tc_mma_ts(tS, tQ + 8 * kk, bdesc, idS, kk > 0 ? 1u : 0u);
          else
            tc_mma(tS, sw128_desc(sQ + (kk & 3) * 32, 16, 1024),
                   bdesc, idS, 1u);
        }
        tc_commit(s_full);
        tc_commit(k_empty + 8 * sb);
      }
      __syncwarp();
    }
    if (lane == 0 && js > 0) mbar_drain(s_full, (uint32_t)(js - 1) & 1u);
    __syncwarp();
    tc_fence_before();
  } else if (warp == 7) {
    // ---------------- P V warp: lane 0 issues O += P_j V_j ----------------
    tc_fence_after();
    constexpr uint32_t idO = bf16_idesc(kTcRows, D, true);
    for (int jp = 0; jp < nkt; ++jp) {
      int ok = 1;
      if (lane == 0)
        ok = mbar_spin_wait(p_full, (uint32_t)jp & 1u, abort_flag, a.err) &&
             mbar_spin_wait(v_full + 8 * (jp % NS), (uint32_t)(jp / NS) & 1u, abort_flag, a.err);
      if (!__shfl_sync(kAll, ok, 0)) break;
      tc_fence_after();
      const uint32_t vst = sV + (jp % NS) * Lay::kSlot;
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k)
          tc_mma_ts(tO, tP + 8 * k, sw128_desc(vst + 2048 * k, Lay::kKHalf, 1024), idO,
                    (jp > 0 || k > 0) ? 1u : 0u);
        tc_commit(o_done);
        tc_commit(v_empty + 8 * (jp % NS));
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(fin);
    __syncwarp();
    mbar_drain(fin, 0);
    tc_fence_before();
  } else {
    // ---------------- producer warps: warp 5 stages K, warp 6 V; lane b block b ----------------
    const int32_t *table = a.block_tables + (size_t)s * a.max_blocks;
    const bool is_v = warp == 6;
    const uint32_t full = is_v ? v_full : k_full, empty = is_v ? v_empty : k_empty;
    const uint32_t ring = is_v ? sV : sK;
    const CUtensorMap *map = is_v ? &tv : &tk;
    int issued = 0;
    if (lane < kTileBlocks) {
      int next = lane * kBlockSize < kv_end ? table[lane] : INT_MIN;
      for (int j = 0; j < nkt; ++j) {
        const int slot = j % NS;
        int blk = next;
        const int tok_n = (j + 1) * kKeys + lane * kBlockSize;
        next = (j + 1 < nkt && tok_n < kv_end) ? table[tok_n / kBlockSize] : INT_MIN;
        if (j >= NS &&
            !mbar_wait(empty + 8 * slot, (uint32_t)((j - NS) / NS) & 1u, abort_flag, a.err))
          break;
        if (blk != INT_MIN && (blk < 0 || blk >= a.num_blocks)) {
          flag_error(a.err, PKV_DEV_BAD_BLOCK);
          blk = INT_MIN;
        }
        const uint32_t bar = full + 8 * slot;
        mbar_arrive_expect_tx(bar, blk != INT_MIN ? 2048u * H : 0u);
        if (blk != INT_MIN) {
          const int row = (blk * a.num_kv_heads + g) * kBlockSize;
          const uint32_t dst = ring + slot * Lay::kSlot + lane * 2048;
#pragma unroll
          for (int h = 0; h < H; ++h) tma_load_2d(dst + h * Lay::kKHalf, map, 64 * h, row, bar);
        }
        issued = j + 1;
      }
    }
    __syncwarp();
    if (lane == 0 && *abort_flag)
      for (int j = max(0, issued - NS); j < issued; ++j)
        mbar_drain(full + 8 * (j % NS), (uint32_t)(j / NS) & 1u);
  }

  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

template <int D, int NS>
int launch_prefill_tcs_t(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                         cudaStream_t st) {
  using Lay = SepLayout<D, NS>;
  static std::atomic<int> ready[kMaxDevices];  // shared-memory opt-in and carve-out, per device
  const int r = per_device_setup(ready, [] {
    cudaError_t e = cudaFuncSetAttribute(
        prefill_tcs_kernel<D, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemLaunch);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_tcs_kernel<D, NS>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    return e == cudaSuccess ? 1 : -(int)e;
  });
  if (r <= 0) return -r;
  return (int)launch_pdl(prefill_tcs_kernel<D, NS>,
                         dim3((unsigned)a.row_tiles, (unsigned)a.num_kv_heads,
                              (unsigned)a.num_seqs),
                         dim3(kTcWarps * 32), (size_t)Lay::kSmemLaunch, st, a, tk, tv);
}

// K/V ring depth of the separate-P kernel: 3 slots each (the shared memory the P tile
// and Q's first half used in the kernel above), overridable for tuning through
// PKV_PREFILL_SEP_STAGES (2 or 3).  Measured on chunked-prefill config 2 / 3: 2 slots
// 1212-1237 / 1044 TFLOP/s, 3 slots 1219-1220 / 1123.
int launch_prefill_sep(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                       int head_dim, cudaStream_t st) {
  static const int stages = [] {  // read once (thread-safe static initialisation)
    const char *v = std::getenv("PKV_PREFILL_SEP_STAGES");
    return v && std::atoi(v) == 2 ? 2 : 3;
  }();
  if (head_dim == 64)
    return stages == 3 ? launch_prefill_tcs_t<64, 3>(a, tk, tv, st)
                       : launch_prefill_tcs_t<64, 2>(a, tk, tv, st);
  return stages == 3 ? launch_prefill_tcs_t<128, 3>(a, tk, tv, st)
                     : launch_prefill_tcs_t<128, 2>(a, tk, tv, st);
}

template <int D, bool PT>
int launch_prefill_tc_t(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                        cudaStream_t st) {
  using Lay = TcLayout<D>;
  static std::atomic<int> ready[kMaxDevices];  // shared-memory opt-in and carve-out, per device
  const int r = per_device_setup(ready, [] {
    cudaError_t e = cudaFuncSetAttribute(
        prefill_tc_kernel<D, PT>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemLaunch);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_tc_kernel<D, PT>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    return e == cudaSuccess ? 1 : -(int)e;
  });
  if (r <= 0) return -r;
  return (int)launch_pdl(prefill_tc_kernel<D, PT>,
                         dim3((unsigned)a.row_tiles, (unsigned)a.num_kv_heads,
                              (unsigned)a.num_seqs),
                         dim3(kTcWarps * 32), (size_t)Lay::kSmemLaunch, st, a, tk, tv);
}

// ------------------------------------------------------------------------------------
// Two-tile variant (PKV_PREFILL_TC_PAIR).  The tensor core reads its shared-memory
// operands at about 128 bytes per cycle per SM (probes: an M 128 x N 64 x K 16 product
// with both operands in shared memory, 6 KB, takes 48 cycles; N 128, 8 KB, 64), and the
// TMA writes of the K/V tiles share that bandwidth.  In the kernel above two CTAs per SM
// each stage their own copy of every K and V tile: per 64-key tile and CTA the score
// products read 48 KB (Q 32 KB + K 16 KB), the P V products 16 KB (V) and the copies
// write 32 KB, i.e. about 1500 cycles of shared-memory traffic per 1024 cycles of tensor
// work on the SM.  Here one CTA per SM holds two consecutive 128-row query tiles of one
// (sequence, KV head) as two independent chains -- each with its own Q tile, two S
// buffers and O accumulator in TMEM (columns 256 c .. 256 c + 255, all 512 allocated)
// and its own softmax, score and P V warps -- that share every K and V tile: the copies
// write half as much per query row (≈ 1250 cycles per 1024).
//  * warps 0-3 / 4-7: softmax of chain 0 / 1 (thread t owns row t of its tile);
//  * warps 8 / 9: score products of chain 0 / 1; warps 10 / 11: P V products;
//  * warps 12 / 13: K / V copies into NS-slot rings (lane b: block b of the tile).
// A K (V) slot is free once both chains' score (P V) products on it are done (two
// arrivals).  Chain 1 may need a tile more than chain 0 (its rows see later keys);
// a chain that does not use a staged tile waits for it to land and then only adds its
// arrival, so neither chain can run ahead of the copies.  P sits over its S columns in
// TMEM (as in the kernel above).
constexpr int kPairWarps = 14;

template <int D, int NS>
struct PairLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kTcRows * 128;         // 16 KB: 128 rows x 64 dims
  static constexpr int kKHalf = kKeys * 128;           // 8 KB: 64 keys x 64 dims
  static constexpr int kQChain = kHalves * kQHalf;     // one chain's Q tile
  static constexpr int kSlot = kHalves * kKHalf;       // one K or V tile
  static constexpr int kK = 2 * kQChain;
  static constexpr int kV = kK + NS * kSlot;
  static constexpr int kBars = kV + NS * kSlot;
  // k_full, k_empty, v_full, v_empty [NS]; per chain: s_full[2], p_full[2], pv_done[2],
  // o_done, fin
  static constexpr int kNumBars = 4 * NS + 2 * 8;
  static constexpr int kSmem = kBars + kNumBars * 8 + 16;
  // more than half an SM's shared memory: one CTA per SM (it holds all 512 TMEM columns)
  static constexpr int kSmemLaunch = kSmem > 120 * 1024 ? kSmem : 120 * 1024;
};

template <int D, int NS>
__global__ void __launch_bounds__(kPairWarps * 32, 1)
    prefill_tc_pair_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tk,
                           const __grid_constant__ CUtensorMap tv) {
  using Lay = PairLayout<D, NS>;
  constexpr int H = Lay::kHalves;
  extern __shared__ __align__(1024) unsigned char smem_tc[];
  const uint32_t base = smem_u32(smem_tc);
  if (base & 1023u) {  // the swizzled tiles need a 1024-byte aligned window
    if (threadIdx.x == 0) flag_error(a.err, PKV_DEV_LAYOUT);
    return;
  }
  const uint32_t sK = base + Lay::kK, sV = base + Lay::kV;
  const uint32_t bars = base + Lay::kBars;
  const uint32_t k_full = bars, k_empty = bars + 8 * NS, v_full = bars + 16 * NS,
                 v_empty = bars + 24 * NS;
  auto chain_bar = [&](int c, int k) { return bars + 32 * NS + 64 * c + 8 * k; };
  // per chain c: s_full = chain_bar(c, 0..1), p_full (2..3), pv_done (4..5), o_done (6),
  // fin (7)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_tc + Lay::kBars + Lay::kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, g = blockIdx.y;
  const int pair = (a.row_tiles + 1) / 2 - 1 - (int)blockIdx.x;  // latest rows first

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(k_full + 8 * i, kTileBlocks);
      mbar_init(k_empty + 8 * i, 2);
      mbar_init(v_full + 8 * i, kTileBlocks);
      mbar_init(v_empty + 8 * i, 2);
    }
    for (int c = 0; c < 2; ++c) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(chain_bar(c, i), 1);
        mbar_init(chain_bar(c, 2 + i), 4);
        mbar_init(chain_bar(c, 4 + i), 1);
      }
      mbar_init(chain_bar(c, 6), 1);
      mbar_init(chain_bar(c, 7), 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_trigger();
  pdl_wait();

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
  const int first_pos = ctx - L;
  // Chain c's rows start at r0 + 128 c; its keys end at kv_end_c (tiles: nkt_c).
  const int r0 = 2 * pair * kTcRows;
  if (r0 >= rows) return;  // no row of this pair exists
  auto keys_end = [&](int rs) { return first_pos + (min(rs + kTcRows, rows) - 1) / G + 1; };
  const int kv_end0 = keys_end(r0);
  const bool has1 = r0 + kTcRows < rows;
  const int kv_end = has1 ? keys_end(r0 + kTcRows) : kv_end0;  // the CTA's last key + 1
  const int nkt0 = (kv_end0 + kKeys - 1) / kKeys;
  const int nkt = (kv_end + kKeys - 1) / kKeys;
  auto chain_tiles = [&](int c) { return c == 0 ? nkt0 : (has1 ? nkt : 0); };

  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ---------------- softmax warps: chain c, thread t owns row t of its tile ----------
    const int c = warp >> 2, t = threadIdx.x & 127, wq = warp & 3;
    const int nk = chain_tiles(c);
    const uint32_t tS = tmem + 256 * c, tO = tS + 128;
    const uint32_t sQ = base + c * Lay::kQChain;
    const uint32_t s_full = chain_bar(c, 0), p_full = chain_bar(c, 2), o_done = chain_bar(c, 6),
                   fin = chain_bar(c, 7);
    if (nk > 0) {
      const int rc0 = r0 + c * kTcRows;
      const int r = rc0 + t;
      const bool valid = r < rows;
      const int r_last = min(rc0 + kTcRows, rows) - 1;
      const int pos = first_pos + (valid ? r : r_last) / G;
      const int warp_pos_lo = first_pos + min(rc0 + wq * 32, r_last) / G;
      const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
      uint16_t *orow = a.out + ((size_t)(q0 + r / G) * a.num_q_heads + g * G + r % G) * D;
      {
        const uint4 *qrow = reinterpret_cast<const uint4 *>(
            a.q + ((size_t)(q0 + r / G) * a.num_q_heads + g * G + r % G) * D);
#pragma unroll
        for (int cc = 0; cc < 8 * H; ++cc) {
          const uint4 v = valid ? qrow[cc] : make_uint4(0u, 0u, 0u, 0u);
          st_shared_v4(sQ + (cc >> 3) * Lay::kQHalf + t * 128 + (((cc & 7) ^ (t & 7)) << 4),
                       v.x, v.y, v.z, v.w);
        }
      }
      fence_proxy_async();
      named_bar_sync(1 + c, 160);

      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nk; ++j) {
        const int sb = j & 1;
        const int t0 = j * kKeys;
        if (!mbar_wait(s_full + 8 * sb, (uint32_t)(j >> 1) & 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t x[64];
        {
          uint32_t (&x0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[0]);
          uint32_t (&x1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[32]);
          tmem_ld32(tS + 64 * sb + lane_base, x0);
          tmem_ld32(tS + 64 * sb + 32 + lane_base, x1);
          tmem_wait_ld();
        }
        // Raw scores; keys past the row's position become -inf (diagonal tiles only).
        const bool need_mask = t0 + kKeys - 1 > warp_pos_lo;
        if (need_mask) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (t0 + cc > pos) x[cc] = __float_as_uint(-INFINITY);
        }
        float mxv[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) mxv[cc] = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 2)
          mxv[(cc >> 1) & 7] =
              max3f(mxv[(cc >> 1) & 7], __uint_as_float(x[cc]), __uint_as_float(x[cc + 1]));
        float mx = max3f(max3f(mxv[0], mxv[1], mxv[2]), max3f(mxv[3], mxv[4], mxv[5]),
                         fmaxf(mxv[6], mxv[7]));
        mx *= a.scale_log2;
        if (j == 0) {
          m = mx;  // key 0 is visible to every row
        } else {
          const bool need = mx > m + 8.f;
          if (__any_sync(kAll, need)) {
            if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, a.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float mn = need ? mx : m;
            const float corr = fast_exp2(m - mn);
            m = mn;
            l *= corr;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(tO + 32 * cc + lane_base, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
              tmem_st32(tO + 32 * cc + lane_base, o);
            }
            tmem_wait_st();
          }
        }
        uint32_t pk[32];
        uint64_t ps2[4];
        const uint64_t sl2 = f32x2(a.scale_log2, a.scale_log2), nm2 = f32x2(-m, -m);
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) {
          float e0, e1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(x[2 * cc]), __uint_as_float(x[2 * cc + 1])),
                                sl2, nm2),
                      e0, e1);
          const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
          const uint64_t pp = f32x2(p0, p1);
          ps2[cc & 3] = cc < 4 ? pp : add_f32x2(ps2[cc & 3], pp);
          pk[cc] = pack_bf16(p0, p1);
        }
        {
          float s0, s1;
          f32x2_split(add_f32x2(add_f32x2(ps2[0], ps2[1]), add_f32x2(ps2[2], ps2[3])), s0, s1);
          l += s0 + s1;
        }
        if (t0 + kKeys > kv_end) {
          // The CTA's last tile: V rows at or past kv_end (tail of the last block, blocks
          // not staged) are set to zero so that their zero weights add exactly nothing.
          // Both chains may zero them (the same values) before their own P V product.
          const int slot = j % NS;
          if (!mbar_wait(v_full + 8 * slot, (uint32_t)(j / NS) & 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t vst = sV + slot * Lay::kSlot;
          const int z0 = kv_end - t0;
          for (int i = t; i < (kKeys - z0) * 8 * H; i += 128) {
            const int row = z0 + i / (8 * H), rem = i % (8 * H);
            st_shared_v4(vst + (rem >> 3) * Lay::kKHalf + row * 128 + (rem & 7) * 16, 0u, 0u,
                         0u, 0u);
          }
          fence_proxy_async();
        }
        // P overwrites the first 32 columns of this tile's S buffer (already read).
        tmem_st32(tS + 64 * sb + lane_base, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + 8 * sb);
      }
      // Every product of this chain has completed once its P V warp's final commit fires.
      if (ok && !mbar_wait(fin, 0u, abort_flag, a.err)) ok = false;
      if (ok && !*abort_flag) {
        tc_fence_after();
        const float inv = 1.f / l;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * cc + lane_base, o);
          tmem_wait_ld();
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * cc);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(
                  pack_bf16(__uint_as_float(o[8 * e]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                  pack_bf16(__uint_as_float(o[8 * e + 2]) * inv,
                            __uint_as_float(o[8 * e + 3]) * inv),
                  pack_bf16(__uint_as_float(o[8 * e + 4]) * inv,
                            __uint_as_float(o[8 * e + 5]) * inv),
                  pack_bf16(__uint_as_float(o[8 * e + 6]) * inv,
                            __uint_as_float(o[8 * e + 7]) * inv));
          }
        }
      }
    }
    tc_fence_before();
  } else if (warp < 10) {
    // ---------------- score warps: lane 0 issues S_j = Q_c K_j^T ----------------
    const int c = warp - 8;
    const int nk = chain_tiles(c);
    const uint32_t tS = tmem + 256 * c, sQ = base + c * Lay::kQChain;
    const uint32_t s_full = chain_bar(c, 0), pv_done = chain_bar(c, 4);
    if (nk > 0) named_bar_sync(1 + c, 160);
    tc_fence_after();
    constexpr uint32_t idS = bf16_idesc(kTcRows, kKeys, false);
    int js = 0;
    for (; js < nkt; ++js) {
      const int sb = js & 1, slot = js % NS;
      int ok = 1;
      if (lane == 0)
        ok = mbar_spin_wait(k_full + 8 * slot, (uint32_t)(js / NS) & 1u, abort_flag, a.err) &&
             (js >= nk || js < 2 ||
              mbar_spin_wait(pv_done + 8 * sb, (uint32_t)((js - 2) >> 1) & 1u, abort_flag,
                             a.err));
      if (!__shfl_sync(kAll, ok, 0)) break;
      tc_fence_after();
      const uint32_t kst = sK + slot * Lay::kSlot;
      if (lane == 0) {
        if (js < nk) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma(tS + 64 * sb,
                   sw128_desc(sQ + (kk >> 2) * Lay::kQHalf + (kk & 3) * 32, 16, 1024),
                   sw128_desc(kst + (kk >> 2) * Lay::kKHalf + (kk & 3) * 32, 16, 1024), idS,
                   kk > 0 ? 1u : 0u);
          tc_commit(s_full + 8 * sb);
          tc_commit(k_empty + 8 * slot);
        } else {
          mbar_arrive(k_empty + 8 * slot);  // a tile only the other chain reads
        }
      }
      __syncwarp();
    }
    // The score products this thread issued have completed once the last one's commit
    // fires (a commit tracks every earlier product of its thread).
    const int last = min(js, nk) - 1;
    if (lane == 0 && last >= 0) mbar_drain(s_full + 8 * (last & 1), (uint32_t)(last >> 1) & 1u);
    __syncwarp();
    tc_fence_before();
  } else if (warp < 12) {
    // ---------------- P V warps: lane 0 issues O_c += P_j V_j ----------------
    const int c = warp - 10;
    const int nk = chain_tiles(c);
    const uint32_t tS = tmem + 256 * c, tO = tS + 128;
    const uint32_t p_full = chain_bar(c, 2), pv_done = chain_bar(c, 4), o_done = chain_bar(c, 6),
                   fin = chain_bar(c, 7);
    tc_fence_after();
    constexpr uint32_t idO = bf16_idesc(kTcRows, D, true);
    for (int jp = 0; jp < nkt; ++jp) {
      const int slot = jp % NS;
      int ok = 1;
      if (lane == 0)
        ok = (jp >= nk || mbar_spin_wait(p_full + 8 * (jp & 1), (uint32_t)(jp >> 1) & 1u,
                                          abort_flag, a.err)) &&
             mbar_spin_wait(v_full + 8 * slot, (uint32_t)(jp / NS) & 1u, abort_flag, a.err);
      if (!__shfl_sync(kAll, ok, 0)) break;
      tc_fence_after();
      const uint32_t vst = sV + slot * Lay::kSlot;
      if (lane == 0) {
        if (jp < nk) {
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k)
            tc_mma_ts(tO, tS + 64 * (jp & 1) + 8 * k,
                      sw128_desc(vst + 2048 * k, Lay::kKHalf, 1024), idO,
                      (jp > 0 || k > 0) ? 1u : 0u);
          tc_commit(o_done);
          tc_commit(v_empty + 8 * slot);
          tc_commit(pv_done + 8 * (jp & 1));
        } else {
          mbar_arrive(v_empty + 8 * slot);  // a tile only the other chain reads
        }
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(fin);
    __syncwarp();
    mbar_drain(fin, 0);
    tc_fence_before();
  } else {
    // ---------------- copy warps: warp 12 stages K, warp 13 V; lane b block b ------------
    const int32_t *table = a.block_tables + (size_t)s * a.max_blocks;
    const bool is_v = warp == 13;
    const uint32_t full = is_v ? v_full : k_full, empty = is_v ? v_empty : k_empty;
    const uint32_t ring = is_v ? sV : sK;
    const CUtensorMap *map = is_v ? &tv : &tk;
    int issued = 0;
    if (lane < kTileBlocks) {
      // block ids are read one tile ahead, so their latency overlaps the slot waits
      int next = lane * kBlockSize < kv_end ? table[lane] : INT_MIN;
      for (int j = 0; j < nkt; ++j) {
        const int slot = j % NS;
        int blk = next;
        const int tok_n = (j + 1) * kKeys + lane * kBlockSize;
        next = (j + 1 < nkt && tok_n < kv_end) ? table[tok_n / kBlockSize] : INT_MIN;
        if (j >= NS &&
            !mbar_wait(empty + 8 * slot, (uint32_t)((j - NS) / NS) & 1u, abort_flag, a.err))
          break;
        if (blk != INT_MIN && (blk < 0 || blk >= a.num_blocks)) {
          flag_error(a.err, PKV_DEV_BAD_BLOCK);
          blk = INT_MIN;
        }
        const uint32_t bar = full + 8 * slot;
        mbar_arrive_expect_tx(bar, blk != INT_MIN ? 2048u * H : 0u);
        if (blk != INT_MIN) {
          const int row = (blk * a.num_kv_heads + g) * kBlockSize;
          const uint32_t dst = ring + slot * Lay::kSlot + lane * 2048;
#pragma unroll
          for (int h = 0; h < H; ++h) tma_load_2d(dst + h * Lay::kKHalf, map, 64 * h, row, bar);
        }
        issued = j + 1;
      }
    }
    __syncwarp();
    // If a wait gave up, let the copies still in flight land before the CTA exits.
    if (lane == 0 && *abort_flag)
      for (int j = max(0, issued - NS); j < issued; ++j)
        mbar_drain(full + 8 * (j % NS), (uint32_t)(j / NS) & 1u);
  }

  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                 : "memory");
  }
}

template <int D, int NS>
int launch_prefill_pair_t(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t st) {
  using Lay = PairLayout<D, NS>;
  static std::atomic<int> ready[kMaxDevices];  // shared-memory opt-in, per device
  const int r = per_device_setup(ready, [] {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_pair_kernel<D, NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kSmemLaunch);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_tc_pair_kernel<D, NS>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    return e == cudaSuccess ? 1 : -(int)e;
  });
  if (r <= 0) return -r;
  return (int)launch_pdl(prefill_tc_pair_kernel<D, NS>,
                         dim3((unsigned)((a.row_tiles + 1) / 2), (unsigned)a.num_kv_heads,
                              (unsigned)a.num_seqs),
                         dim3(kPairWarps * 32), (size_t)Lay::kSmemLaunch, st, a, tk, tv);
}

// K/V ring depth, overridable for tuning through PKV_PREFILL_PAIR_STAGES (2, 3 or 4).
int pair_stages() {
  static const int n = [] {  // read once (thread-safe static initialisation)
    const char *v = std::getenv("PKV_PREFILL_PAIR_STAGES");
    const int k = v ? std::atoi(v) : 2;
    return k >= 2 && k <= 4 ? k : 2;
  }();
  return n;
}

int launch_prefill_pair(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                        int head_dim, cudaStream_t st) {
  switch (pair_stages()) {
    case 3: return head_dim == 64 ? launch_prefill_pair_t<64, 3>(a, tk, tv, st)
                                  : launch_prefill_pair_t<128, 3>(a, tk, tv, st);
    case 4: return head_dim == 64 ? launch_prefill_pair_t<64, 4>(a, tk, tv, st)
                                  : launch_prefill_pair_t<128, 4>(a, tk, tv, st);
    default: return head_dim == 64 ? launch_prefill_pair_t<64, 2>(a, tk, tv, st)
                                   : launch_prefill_pair_t<128, 2>(a, tk, tv, st);
  }
}

// ------------------------------------------------------------------------------------
// SM-pair variant (PKV_PREFILL_TC_2SM, head_dim 128): a cluster of two CTAs on two SMs
// runs one chain over 256 query rows -- CTA rank r holds rows 128 r .. 128 r + 127 of the
// pair: its own Q tile, softmax warps, S buffers and O accumulator in its TMEM -- and
// rank 0 issues every product as tcgen05.mma.cta_group::2 (M = 256): one instruction
// drives both SMs' tensor pipes, each reading its own A rows (Q, or P from its TMEM) and
// its half of B from its own shared memory at the same offsets.  So each SM stages half
// of every tile: the 32 keys 32 r .. 32 r + 31 of a K tile (score products, N = 64) and
// the head-dim columns 64 r .. 64 r + 63 of a V tile (P V products, N = 128).  Per SM and
// 64-key tile that halves the copies and the B operand reads, and halves the product
// instructions an SM issues.  Two clusters share each pair of SMs (256 TMEM columns per
// CTA).
//  * warps 0-3 (both ranks): softmax of the CTA's 128 rows, as in the one-tile kernel;
//    rank 1 signals its Q and each P to rank 0's barriers (remote mbarrier arrivals).
//  * warp 4: rank 0 issues the score products; rank 1 forwards its K copies' completion
//    to rank 0.  warp 7: rank 0 issues the P V products; rank 1 forwards its V copies'.
//  * warps 5 / 6: this CTA's halves of the K / V tiles (TMA), into NS-slot rings.
// Completion of the products (tcgen05.commit ... multicast) arrives at both CTAs'
// barriers (S ready, K / V slot free, O updated, P V done, final).  Every wait is bounded;
// both CTAs leave through one cluster barrier before the pair releases its tensor memory.
constexpr int kPairCtaWarps = 8;

template <int NS>
struct Sm2Layout {
  static constexpr int kQHalf = kTcRows * 128;  // 16 KB: 128 rows x 64 dims
  static constexpr int kKPart = 32 * 128;       // 4 KB: 32 keys x 64 dims
  static constexpr int kKSlot = 2 * kKPart;     // this CTA's 32 keys, both dim halves
  static constexpr int kVSlot = kKeys * 128;    // 8 KB: 64 keys x this CTA's 64 dims
  static constexpr int kQ = 0;
  static constexpr int kK = 2 * kQHalf;
  static constexpr int kV = kK + NS * kKSlot;
  static constexpr int kBars = kV + NS * kVSlot;
  // k_full, k_empty, kp_full, v_full, v_empty, vp_full [NS]; s_full[2], p_full[2],
  // pv_done[2], o_done, fin, q_full
  static constexpr int kNumBars = 6 * NS + 9;
  static constexpr int kSmem = kBars + kNumBars * 8 + 16;
  // at least 78 KB, so that no more than two CTAs share an SM (256 TMEM columns each)
  static constexpr int kSmemLaunch = kSmem > 78 * 1024 ? kSmem : 78 * 1024;
};

__device__ __forceinline__ bool mbar_test_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_spin_wait for a barrier that the peer CTA also arrives on (acquire at cluster
// scope, pairing with the peer's release): same give-up rules.
__device__ inline bool mbar_spin_wait_cl(uint32_t bar, uint32_t parity, volatile int *abort,
                                         int32_t *err, long long limit = kWaitCycles) {
  if (mbar_test_wait_cl(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_wait_cl(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > limit) {
        *abort = 1;
        flag_error(err, PKV_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// One arrival on the barrier at the same shared-memory offset in CTA `rank` of the
// cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}

__device__ __forceinline__ void tc2_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc2_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Completion of this thread's earlier products arrives at the barrier at offset `bar`
// in both CTAs of the pair.
__device__ __forceinline__ void tc2_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

template <int NS>
__global__ void __launch_bounds__(kPairCtaWarps * 32, 2)
    prefill_tc2sm_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv) {
  constexpr int D = 128;
  using Lay = Sm2Layout<NS>;
  extern __shared__ __align__(1024) unsigned char smem_tc[];
  const uint32_t base = smem_u32(smem_tc);
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  // The swizzled tiles need a 1024-byte aligned window; both CTAs run the same code, so
  // a misaligned window is misaligned in both and both leave here.
  if (base & 1023u) {
    if (threadIdx.x == 0) flag_error(a.err, PKV_DEV_LAYOUT);
    return;
  }
  const uint32_t sQ = base + Lay::kQ, sK = base + Lay::kK, sV = base + Lay::kV;
  const uint32_t bars = base + Lay::kBars;
  const uint32_t k_full = bars, k_empty = bars + 8 * NS, kp_full = bars + 16 * NS,
                 v_full = bars + 24 * NS, v_empty = bars + 32 * NS, vp_full = bars + 40 * NS;
  const uint32_t s_full = bars + 48 * NS, p_full = s_full + 16, pv_done = p_full + 16,
                 o_done = pv_done + 16, fin = o_done + 8, q_full = fin + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_tc + Lay::kBars + Lay::kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, g = blockIdx.y;
  const int pair = (a.row_tiles + 1) / 2 - 1 - (int)(blockIdx.x >> 1);  // latest rows first

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(k_full + 8 * i, 2);        // two producer lanes: this CTA's two K blocks
      mbar_init(k_empty + 8 * i, 1);
      mbar_init(kp_full + 8 * i, 1);       // rank 1's forwarded K completion (rank 0 only)
      mbar_init(v_full + 8 * i, kTileBlocks);
      mbar_init(v_empty + 8 * i, 1);
      mbar_init(vp_full + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(p_full + 8 * i, 8);        // four softmax warps of each CTA (rank 0's copy)
      mbar_init(pv_done + 8 * i, 1);
    }
    mbar_init(o_done, 1);
    mbar_init(fin, 1);
    mbar_init(q_full, 8);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_trigger();
  pdl_wait();

  // Both CTAs of a pair read the same sequence and rows, so they leave (or stay) together.
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
  const int rp = pair * 2 * kTcRows;  // the pair's first row
  if (rp >= rows) return;
  const int first_pos = ctx - L;
  const int kv_end = first_pos + (min(rp + 2 * kTcRows, rows) - 1) / G + 1;  // pair's last key + 1
  const int nkt = (kv_end + kKeys - 1) / kKeys;

  // Every barrier of both CTAs is initialised before either CTA arrives on the other's.
  cluster_sync_all();
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;  // S buffers at columns 0 and 64, O after

  if (warp < 4) {
    // ---------------- softmax warps: thread t owns row t of this CTA ----------------
    const int t = threadIdx.x;
    const int r0 = rp + (int)rank * kTcRows;
    const int r = r0 + t;
    const bool valid = r < rows;
    const int r_clamp = min(r, rows - 1);
    const int pos = first_pos + r_clamp / G;
    const int warp_pos_lo = first_pos + min(r0 + warp * 32, rows - 1) / G;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint16_t *orow = a.out + ((size_t)(q0 + r_clamp / G) * a.num_q_heads + g * G + r_clamp % G) * D;
    {
      const uint4 *qrow = reinterpret_cast<const uint4 *>(
          a.q + ((size_t)(q0 + r_clamp / G) * a.num_q_heads + g * G + r_clamp % G) * D);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 v = valid ? qrow[c] : make_uint4(0u, 0u, 0u, 0u);
        st_shared_v4(sQ + (c >> 3) * Lay::kQHalf + t * 128 + (((c & 7) ^ (t & 7)) << 4), v.x,
                     v.y, v.z, v.w);
      }
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive_cta(q_full, 0);  // this CTA's Q is staged

    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int sb = j & 1;
      const int t0 = j * kKeys;
      if (!mbar_wait(s_full + 8 * sb, (uint32_t)(j >> 1) & 1u, abort_flag, a.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x[64];
      {
        uint32_t (&x0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[0]);
        uint32_t (&x1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&x[32]);
        tmem_ld32(tS + 64 * sb + lane_base, x0);
        tmem_ld32(tS + 64 * sb + 32 + lane_base, x1);
        tmem_wait_ld();
      }
      // Keys past the row's position become -inf (diagonal tiles only; rows past the
      // chunk take the last row's position, their outputs are not stored).
      const bool need_mask = t0 + kKeys - 1 > warp_pos_lo;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (t0 + c > pos) x[c] = __float_as_uint(-INFINITY);
      }
      float mxv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mxv[c] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 2)
        mxv[(c >> 1) & 7] =
            max3f(mxv[(c >> 1) & 7], __uint_as_float(x[c]), __uint_as_float(x[c + 1]));
      float mx = max3f(max3f(mxv[0], mxv[1], mxv[2]), max3f(mxv[3], mxv[4], mxv[5]),
                       fmaxf(mxv[6], mxv[7]));
      mx *= a.scale_log2;
      if (j == 0) {
        m = mx;  // key 0 is visible to every row
      } else {
        const bool need = mx > m + 8.f;
        if (__any_sync(kAll, need)) {
          if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float mn = need ? mx : m;
          const float corr = fast_exp2(m - mn);
          m = mn;
          l *= corr;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * cc + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(tO + 32 * cc + lane_base, o);
          }
          tmem_wait_st();
        }
      }
      uint32_t pk[32];
      uint64_t ps2[4];
      const uint64_t sl2 = f32x2(a.scale_log2, a.scale_log2), nm2 = f32x2(-m, -m);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float e0, e1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])),
                              sl2, nm2),
                    e0, e1);
        const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
        const uint64_t pp = f32x2(p0, p1);
        ps2[c & 3] = c < 4 ? pp : add_f32x2(ps2[c & 3], pp);
        pk[c] = pack_bf16(p0, p1);
      }
      {
        float s0, s1;
        f32x2_split(add_f32x2(add_f32x2(ps2[0], ps2[1]), add_f32x2(ps2[2], ps2[3])), s0, s1);
        l += s0 + s1;
      }
      if (t0 + kKeys > kv_end) {
        // Last tile: this CTA's V columns in rows at or past kv_end (tail of the last
        // block, blocks not staged) are set to zero, so that zero weights add nothing.
        const int slot = j % NS;
        if (!mbar_wait(v_full + 8 * slot, (uint32_t)(j / NS) & 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        const uint32_t vst = sV + slot * Lay::kVSlot;
        const int z0 = kv_end - t0;
        for (int i = t; i < (kKeys - z0) * 8; i += 128) {
          const int row = z0 + i / 8, rem = i % 8;
          st_shared_v4(vst + row * 128 + rem * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async();
      }
      // P overwrites the first 32 columns of this tile's S buffer (already read).
      tmem_st32(tS + 64 * sb + lane_base, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(p_full + 8 * sb, 0);
    }
    // Every product has completed once rank 0's final commit fires.
    if (ok && !mbar_wait(fin, 0u, abort_flag, a.err)) ok = false;
    if (ok && !*abort_flag) {
      tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc + lane_base, o);
        tmem_wait_ld();
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * cc);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(
                pack_bf16(__uint_as_float(o[8 * e]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv),
                pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv));
        }
      }
    }
    tc_fence_before();
  } else if (warp == 4 || warp == 7) {
    const bool is_pv = warp == 7;
    if (rank == 1) {
      // ---------------- rank 1: forward this CTA's K (warp 4) / V (warp 7) copies ------
      const uint32_t full = is_pv ? v_full : k_full, fwd = is_pv ? vp_full : kp_full;
      if (lane == 0)
        for (int j = 0; j < nkt; ++j) {
          if (!mbar_wait(full + 8 * (j % NS), (uint32_t)(j / NS) & 1u, abort_flag, a.err)) break;
          mbar_arrive_cta(fwd + 8 * (j % NS), 0);
        }
      __syncwarp();
    } else if (!is_pv) {
      // ---------------- rank 0, warp 4: S_j = Q K_j^T for both CTAs' rows ----------------
      tc_fence_after();
      constexpr uint32_t idS = bf16_idesc(2 * kTcRows, kKeys, false);
      int ok = 1;
      if (lane == 0) ok = mbar_spin_wait_cl(q_full, 0u, abort_flag, a.err);
      int js = 0;
      if (__shfl_sync(kAll, ok, 0))
        for (; js < nkt; ++js) {
          const int sb = js & 1, slot = js % NS;
          if (lane == 0)
            ok = mbar_spin_wait(k_full + 8 * slot, (uint32_t)(js / NS) & 1u, abort_flag, a.err) &&
                 mbar_spin_wait_cl(kp_full + 8 * slot, (uint32_t)(js / NS) & 1u, abort_flag,
                                   a.err) &&
                 (js < 2 || mbar_spin_wait(pv_done + 8 * sb, (uint32_t)((js - 2) >> 1) & 1u,
                                           abort_flag, a.err));
          if (!__shfl_sync(kAll, ok, 0)) break;
          tc_fence_after();
          const uint32_t kst = sK + slot * Lay::kKSlot;
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc2_mma(tS + 64 * sb,
                      sw128_desc(sQ + (kk >> 2) * Lay::kQHalf + (kk & 3) * 32, 16, 1024),
                      sw128_desc(kst + (kk >> 2) * Lay::kKPart + (kk & 3) * 32, 16, 1024), idS,
                      kk > 0 ? 1u : 0u);
            tc2_commit(s_full + 8 * sb);
            tc2_commit(k_empty + 8 * slot);
          }
          __syncwarp();
        }
      // the products this thread issued have completed once its last commit fires
      if (lane == 0 && js > 0) mbar_drain(s_full + 8 * ((js - 1) & 1), (uint32_t)((js - 1) >> 1) & 1u);
      __syncwarp();
      tc_fence_before();
    } else {
      // ---------------- rank 0, warp 7: O += P_j V_j for both CTAs' rows ----------------
      tc_fence_after();
      constexpr uint32_t idO = bf16_idesc(2 * kTcRows, D, true);
      for (int jp = 0; jp < nkt; ++jp) {
        const int slot = jp % NS;
        int ok = 1;
        if (lane == 0)
          ok = mbar_spin_wait_cl(p_full + 8 * (jp & 1), (uint32_t)(jp >> 1) & 1u, abort_flag,
                                 a.err) &&
               mbar_spin_wait(v_full + 8 * slot, (uint32_t)(jp / NS) & 1u, abort_flag, a.err) &&
               mbar_spin_wait_cl(vp_full + 8 * slot, (uint32_t)(jp / NS) & 1u, abort_flag, a.err);
        if (!__shfl_sync(kAll, ok, 0)) break;
        tc_fence_after();
        const uint32_t vst = sV + slot * Lay::kVSlot;
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k)
            tc2_mma_ts(tO, tS + 64 * (jp & 1) + 8 * k, sw128_desc(vst + 2048 * k, 8192, 1024),
                       idO, (jp > 0 || k > 0) ? 1u : 0u);
          tc2_commit(o_done);
          tc2_commit(v_empty + 8 * slot);
          tc2_commit(pv_done + 8 * (jp & 1));
        }
        __syncwarp();
      }
      if (lane == 0) tc2_commit(fin);
      __syncwarp();
      mbar_drain(fin, 0);
      tc_fence_before();
    }
  } else {
    // ---------------- copy warps: warp 5 K (this CTA's 32 keys), warp 6 V (its 64 dims) --
    const int32_t *table = a.block_tables + (size_t)s * a.max_blocks;
    const bool is_v = warp == 6;
    const uint32_t full = is_v ? v_full : k_full, empty = is_v ? v_empty : k_empty;
    const int nlanes = is_v ? kTileBlocks : 2;
    // K: lane b copies block 2 rank + b of the tile (both dim halves); V: lane b copies
    // block b (the CTA's dim half)
    const int blk_in_tile = is_v ? lane : 2 * (int)rank + lane;
    const CUtensorMap *map = is_v ? &tv : &tk;
    int issued = 0;
    if (lane < nlanes) {
      int next = blk_in_tile * kBlockSize < kv_end ? table[blk_in_tile] : INT_MIN;
      for (int j = 0; j < nkt; ++j) {
        const int slot = j % NS;
        int blk = next;
        const int tok_n = (j + 1) * kKeys + blk_in_tile * kBlockSize;
        next = (j + 1 < nkt && tok_n < kv_end) ? table[tok_n / kBlockSize] : INT_MIN;
        if (j >= NS &&
            !mbar_wait(empty + 8 * slot, (uint32_t)((j - NS) / NS) & 1u, abort_flag, a.err))
          break;
        if (blk != INT_MIN && (blk < 0 || blk >= a.num_blocks)) {
          flag_error(a.err, PKV_DEV_BAD_BLOCK);
          blk = INT_MIN;
        }
        const uint32_t bar = full + 8 * slot;
        mbar_arrive_expect_tx(bar, blk != INT_MIN ? (is_v ? 2048u : 4096u) : 0u);
        if (blk != INT_MIN) {
          const int row = (blk * a.num_kv_heads + g) * kBlockSize;
          if (is_v) {
            tma_load_2d(sV + slot * Lay::kVSlot + lane * 2048, map, 64 * (int)rank, row, bar);
          } else {
            const uint32_t dst = sK + slot * Lay::kKSlot + lane * 2048;
            tma_load_2d(dst, map, 0, row, bar);
            tma_load_2d(dst + Lay::kKPart, map, 64, row, bar);
          }
        }
        issued = j + 1;
      }
    }
    __syncwarp();
    // If a wait gave up, let the copies still in flight land before the CTA exits.
    if (lane == 0 && *abort_flag)
      for (int j = max(0, issued - NS); j < issued; ++j)
        mbar_drain(full + 8 * (j % NS), (uint32_t)(j / NS) & 1u);
  }

  __syncthreads();
  // Neither CTA releases the pair's tensor memory, or exits, while the other may still
  // read it or arrive on its barriers.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

template <int NS>
int launch_prefill_2sm_t(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                         cudaStream_t st) {
  using Lay = Sm2Layout<NS>;
  static std::atomic<int> ready[kMaxDevices];  // shared-memory opt-in, per device
  const int r = per_device_setup(ready, [] {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc2sm_kernel<NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kSmemLaunch);
    return e == cudaSuccess ? 1 : -(int)e;
  });
  if (r <= 0) return -r;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * ((a.row_tiles + 1) / 2)), (unsigned)a.num_kv_heads,
                     (unsigned)a.num_seqs);
  cfg.blockDim = dim3(kPairCtaWarps * 32);
  cfg.dynamicSmemBytes = (size_t)Lay::kSmemLaunch;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return (int)cudaLaunchKernelEx(&cfg, prefill_tc2sm_kernel<NS>, a, tk, tv);
}

// P kept in tensor memory by default (the A operand of P V read from TMEM: no shared-
// memory traffic for P, 6% faster on GB300); PKV_PREFILL_P=smem selects the variant that
// stages P in shared memory.
int launch_prefill_tc(const PrefillArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                      int head_dim, cudaStream_t st) {
  static const bool p_in_tmem = [] {  // read once (thread-safe static initialisation)
    const char *v = std::getenv("PKV_PREFILL_P");
    return !(v && std::strcmp(v, "smem") == 0);
  }();
  if (head_dim == 64)
    return p_in_tmem ? launch_prefill_tc_t<64, true>(a, tk, tv, st)
                     : launch_prefill_tc_t<64, false>(a, tk, tv, st);
  return p_in_tmem ? launch_prefill_tc_t<128, true>(a, tk, tv, st)
                   : launch_prefill_tc_t<128, false>(a, tk, tv, st);
}

std::atomic<int> g_prefill_variant{PKV_PREFILL_AUTO};

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
  const int variant = g_prefill_variant.load();
  const bool tc = variant != PKV_PREFILL_MMA;
  const bool pair = variant == PKV_PREFILL_TC_PAIR;
  const bool sm2 = variant == PKV_PREFILL_TC_2SM && head_dim == 128;
  // AUTO: the separate-P tcgen05 kernel (the fastest measured, head_dim 64 and 128)
  const bool sep = variant == PKV_PREFILL_TC_SEP || variant == PKV_PREFILL_AUTO;
  const int rows_per_cta = tc ? kTcRows : kRows;
  const int64_t tiles = ((int64_t)max_query_len * group + rows_per_cta - 1) / rows_per_cta;
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
  const int rc = sep    ? launch_prefill_sep(a, tk, tv, head_dim, st)
                 : sm2  ? launch_prefill_2sm_t<3>(a, tk, tv, st)
                 : pair ? launch_prefill_pair(a, tk, tv, head_dim, st)
                 : tc   ? launch_prefill_tc(a, tk, tv, head_dim, st)
                 : head_dim == 128 ? launch_prefill_t<128, 3>(a, tk, tv, st)
                                   : launch_prefill_t<64, 4>(a, tk, tv, st);
  return rc == 0 ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int paged_attention_prefill_set_variant(int variant) {
  if (variant != PKV_PREFILL_AUTO && variant != PKV_PREFILL_MMA && variant != PKV_PREFILL_TC &&
      variant != PKV_PREFILL_TC_PAIR && variant != PKV_PREFILL_TC_2SM &&
      variant != PKV_PREFILL_TC_SEP)
    return PKV_ERR_ARG;
  return g_prefill_variant.exchange(variant);
}
