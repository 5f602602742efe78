// Row movers of the paged KV write, shared by the write kernels and the fused decode-step
// prologue.  One call moves one 16-byte vector (8 bf16 elements) of one (token, KV head)
// row of k_new / v_new into the row's slot of the cache: a plain copy for a bf16 cache
// (bit-exact), or the E4M3 quantisation for an E4M3 cache.
#pragma once

#include <cuda_fp8.h>

#include "pkv_common.cuh"

namespace pkv {

// bf16 cache [NB][Hkv][16][D]: vector e of row (t, h) -> row (slot / 16, h, slot % 16).
__device__ __forceinline__ void put_row_vec_bf16(const uint4 *__restrict__ k_new,
                                                 const uint4 *__restrict__ v_new, int64_t i,
                                                 int64_t slot, int h, int e, int heads,
                                                 int row_vecs, uint4 *__restrict__ k_cache,
                                                 uint4 *__restrict__ v_cache) {
  const int64_t block = slot >> 4, offset = slot & 15;
  const int64_t dst = ((block * heads + h) * kBlockSize + offset) * row_vecs + e;
  k_cache[dst] = k_new[i];
  v_cache[dst] = v_new[i];
}

// E4M3 code of x / scale: the division rounded to nearest in fp32, then the hardware
// conversion (round to nearest even, finite saturation).  Four elements per call.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float scale) {
  const float2 lo = make_float2(__fdiv_rn(bf16_lo(w0), scale), __fdiv_rn(bf16_hi(w0), scale));
  const float2 hi = make_float2(__fdiv_rn(bf16_lo(w1), scale), __fdiv_rn(bf16_hi(w1), scale));
  const uint32_t a = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
  const uint32_t b = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
  return (a & 0xffffu) | (b << 16);
}

// E4M3 cache: K codes [NB][Hkv][16][D], V codes transposed within a block,
// [NB][Hkv][D][16], so each V code is a byte of its own head-dim row.  Scales:
// k_scales / v_scales per KV head when non-null (a scale that is not > 0 sets
// PKV_DEV_BAD_SCALE and the vector is skipped), else k_scale / v_scale.
// When row_vecs is a power of two up to 32 (head_dim 64, 128, ...), the row_vecs vectors
// of one (token, KV head) row must be handled by row_vecs consecutive lanes of one warp
// (lane & (row_vecs - 1) == e), all calling together: they trade V codes through
// shuffles so that in each of eight rounds lane e stores the code of head-dim row
// row_vecs * round + e -- the group's stores of a round cover row_vecs consecutive rows,
// two per 32-byte sector, half the sectors of storing each lane's own eight codes.
// Other head dims store each lane's own eight codes.
__device__ __forceinline__ void put_row_vec_e4m3(const uint4 *__restrict__ k_new,
                                                 const uint4 *__restrict__ v_new, int64_t i,
                                                 int64_t slot, int h, int e, int heads,
                                                 int row_vecs, uint2 *__restrict__ k_cache,
                                                 uint8_t *__restrict__ v_cache, float k_scale,
                                                 float v_scale, const float *k_scales,
                                                 const float *v_scales, int32_t *err) {
  float ks = k_scale, vs = v_scale;
  if (k_scales != nullptr) {  // one scale per KV head
    ks = __ldg(k_scales + h);
    vs = __ldg(v_scales + h);
    if (!(ks > 0.f) || !(vs > 0.f)) {
      flag_error(err, PKV_DEV_BAD_SCALE);
      return;
    }
  }
  const int64_t dst = (((slot >> 4) * heads + h) * kBlockSize + (slot & 15)) * row_vecs + e;
  const uint4 kv = k_new[i], vv = v_new[i];
  k_cache[dst] = make_uint2(quant4(kv.x, kv.y, ks), quant4(kv.z, kv.w, ks));
  // codes of head-dim rows 8e .. 8e + 3 (v0) and 8e + 4 .. 8e + 7 (v1), lowest byte first
  const uint32_t v0 = quant4(vv.x, vv.y, vs), v1 = quant4(vv.z, vv.w, vs);
  const int D = row_vecs * 8;
  uint8_t *vblk = v_cache + ((slot >> 4) * heads + h) * (int64_t)D * kBlockSize + (slot & 15);
  if ((row_vecs & (row_vecs - 1)) == 0 && row_vecs <= 32) {
    const int gbase = (int)(threadIdx.x & 31) & ~(row_vecs - 1);
    const unsigned gmask = (row_vecs == 32 ? 0xffffffffu : ((1u << row_vecs) - 1u)) << gbase;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int d = row_vecs * k + e;  // the row this lane stores in round k
      const uint32_t w0 = __shfl_sync(gmask, v0, gbase + (d >> 3));
      const uint32_t w1 = __shfl_sync(gmask, v1, gbase + (d >> 3));
      vblk[(int64_t)d * kBlockSize] = (uint8_t)(((d & 4) ? w1 : w0) >> (8 * (d & 3)));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      vblk[(int64_t)(8 * e + j) * kBlockSize] = (uint8_t)(v0 >> (8 * j));
      vblk[(int64_t)(8 * e + 4 + j) * kBlockSize] = (uint8_t)(v1 >> (8 * j));
    }
  }
}

}  // namespace pkv
