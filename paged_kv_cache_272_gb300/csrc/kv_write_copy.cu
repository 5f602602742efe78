// Paged KV write (slot_mapping scatter) and copy-on-write block copy.
//
// Both are pure byte movement in 16-byte vectors: no float conversion, so they are
// bit-exact by construction.  Sources: "Inference optimization", section "KV cache"
// (append only the new token's K/V) and "Continuous batching and PagedAttention",
// section 3 (copy-on-write of a shared block when a request diverges).
#include <cstring>

#include "kv_rows.cuh"
#include "pkv_common.cuh"

namespace pkv {
namespace {

// One thread moves one 16-byte vector of K and the matching vector of V.
// Thread index i enumerates (token t, KV head h, vector e) with e fastest, which is
// also the layout of k_new/v_new, so reads are fully coalesced; each (t, h) row of
// head_dim bf16 lands as one contiguous row in the cache.
__global__ void kv_write_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                const int64_t *__restrict__ slots, int64_t total, int row_vecs,
                                int heads, int64_t num_slots, uint4 *__restrict__ k_cache,
                                uint4 *__restrict__ v_cache, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t row = i / row_vecs;  // t * heads + h
    const int e = (int)(i - row * row_vecs);
    const int64_t t = row / heads;
    const int h = (int)(row - t * heads);
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      flag_error(err, PKV_DEV_BAD_SLOT);
      continue;
    }
    put_row_vec_bf16(k_new, v_new, i, slot, h, e, heads, row_vecs, k_cache, v_cache);
  }
}

// E4M3 write: thread i handles 8 consecutive elements of one (token, KV head) row (see
// put_row_vec_e4m3: the block size and the grid stride are multiples of row_vecs, so a
// row's vectors fall on consecutive lanes, and a row's lanes skip or stay together).
__global__ void kv_write_fp8_kernel(const uint4 *__restrict__ k_new,
                                    const uint4 *__restrict__ v_new,
                                    const int64_t *__restrict__ slots, int64_t total, int row_vecs,
                                    int heads, int64_t num_slots, uint2 *__restrict__ k_cache,
                                    uint8_t *__restrict__ v_cache, float k_scale, float v_scale,
                                    const float *__restrict__ k_scales,
                                    const float *__restrict__ v_scales, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t row = i / row_vecs;  // t * heads + h
    const int e = (int)(i - row * row_vecs);
    const int64_t t = row / heads;
    const int h = (int)(row - t * heads);
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      flag_error(err, PKV_DEV_BAD_SLOT);
      continue;
    }
    put_row_vec_e4m3(k_new, v_new, i, slot, h, e, heads, row_vecs, k_cache, v_cache, k_scale,
                     v_scale, k_scales, v_scales, err);
  }
}

// Thread index i enumerates (pair p, vector e of the block) with e fastest; a block is
// num_kv_heads * 16 * head_dim bf16 contiguous bytes in both caches.
__global__ void block_copy_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                  const int32_t *__restrict__ pairs, int64_t total,
                                  int64_t block_vecs, int num_blocks, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t p = i / block_vecs;
    const int64_t e = i - p * block_vecs;
    const int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if ((unsigned)src >= (unsigned)num_blocks || (unsigned)dst >= (unsigned)num_blocks) {
      if (e == 0) flag_error(err, PKV_DEV_BAD_BLOCK);
      continue;
    }
    const uint4 kv = k_cache[(int64_t)src * block_vecs + e];
    const uint4 vv = v_cache[(int64_t)src * block_vecs + e];
    k_cache[(int64_t)dst * block_vecs + e] = kv;
    v_cache[(int64_t)dst * block_vecs + e] = vv;
  }
}

int grid_for(int64_t total, int threads) {
  const int64_t want = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 16;  // grid-stride beyond this
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

int device_sm_count() {
  static std::atomic<int> slots[kMaxDevices];
  return per_device_setup(slots, [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    return n;
  });
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int paged_kv_version(void) { return PKV_ABI_VERSION; }

const char *paged_kv_strerror(int code) {
  switch (code) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_SHAPE: return "a size is out of range or head_dim is unsupported";
    case PKV_ERR_BLOCK_SIZE: return "block_size must be 16";
    case PKV_ERR_ALIGN: return "a bf16 buffer is not 16-byte aligned";
    case PKV_ERR_WORKSPACE: return "workspace is smaller than paged_attention_workspace_size";
    case PKV_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case PKV_ERR_OOM: return "block pool has no free block";
    case PKV_ERR_UNKNOWN_SEQ: return "unknown sequence id";
    case PKV_ERR_DUP_SEQ: return "sequence id already in use";
    case PKV_ERR_REFCOUNT: return "block refcount underflow";
    case PKV_ERR_ARG: return "bad argument";
    default: return "unknown error code";
  }
}

int paged_kv_write(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slot_mapping,
                   int num_tokens, uint16_t *k_cache, uint16_t *v_cache, int num_blocks,
                   int num_kv_heads, int head_dim, int block_size, int32_t *err_flag,
                   void *stream) {
  if (block_size != kBlockSize) return PKV_ERR_BLOCK_SIZE;
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 8 != 0)
    return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ALIGN;
  const int row_vecs = head_dim / 8;
  const int64_t total = (int64_t)num_tokens * num_kv_heads * row_vecs;
  const int threads = 256;
  const cudaError_t e = launch_pdl(
      kv_write_kernel, dim3(grid_for(total, threads)), dim3(threads), 0, (cudaStream_t)stream,
      reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
      slot_mapping, total, row_vecs, num_kv_heads, (int64_t)num_blocks * kBlockSize,
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), err_flag);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int paged_block_copy(uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_pairs,
                     int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                     int block_size, int32_t *err_flag, void *stream) {
  if (block_size != kBlockSize) return PKV_ERR_BLOCK_SIZE;
  if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 8 != 0)
    return PKV_ERR_SHAPE;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_NULL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
  const int64_t block_vecs = (int64_t)num_kv_heads * kBlockSize * head_dim / 8;
  const int64_t total = (int64_t)num_pairs * block_vecs;
  const int threads = 256;
  const cudaError_t e = launch_pdl(
      block_copy_kernel, dim3(grid_for(total, threads)), dim3(threads), 0, (cudaStream_t)stream,
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), block_pairs, total,
      block_vecs, num_blocks, err_flag);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"

// Shared by the per-cache and per-KV-head entry points (k_scales null: per cache).
static int write_fp8_impl(const uint16_t *k_new, const uint16_t *v_new,
                          const int64_t *slot_mapping, int num_tokens, uint8_t *k_cache,
                          uint8_t *v_cache, int num_blocks, int num_kv_heads, int head_dim,
                          int block_size, float k_scale, float v_scale, const float *k_scales,
                          const float *v_scales, int32_t *err_flag, void *stream) {
  if (block_size != kBlockSize) return PKV_ERR_BLOCK_SIZE;
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 16 != 0 || !(k_scale > 0.f) || !(v_scale > 0.f))
    return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ALIGN;
  const int row_vecs = head_dim / 8;
  const int64_t total = (int64_t)num_tokens * num_kv_heads * row_vecs;
  const int threads = 256;
  const cudaError_t e = launch_pdl(
      kv_write_fp8_kernel, dim3(grid_for(total, threads)), dim3(threads), 0, (cudaStream_t)stream,
      reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
      slot_mapping, total, row_vecs, num_kv_heads, (int64_t)num_blocks * kBlockSize,
      reinterpret_cast<uint2 *>(k_cache), v_cache, k_scale, v_scale, k_scales, v_scales,
      err_flag);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" {

int paged_kv_write_fp8(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slot_mapping,
                       int num_tokens, uint8_t *k_cache, uint8_t *v_cache, int num_blocks,
                       int num_kv_heads, int head_dim, int block_size, float k_scale,
                       float v_scale, int32_t *err_flag, void *stream) {
  return write_fp8_impl(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks,
                        num_kv_heads, head_dim, block_size, k_scale, v_scale, nullptr, nullptr,
                        err_flag, stream);
}

int paged_kv_write_fp8_per_head(const uint16_t *k_new, const uint16_t *v_new,
                                const int64_t *slot_mapping, int num_tokens, uint8_t *k_cache,
                                uint8_t *v_cache, int num_blocks, int num_kv_heads,
                                int head_dim, int block_size, const float *k_scales,
                                const float *v_scales, int32_t *err_flag, void *stream) {
  if (num_tokens > 0 && (!k_scales || !v_scales)) return PKV_ERR_NULL;
  return write_fp8_impl(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks,
                        num_kv_heads, head_dim, block_size, 1.f, 1.f, k_scales, v_scales,
                        err_flag, stream);
}

int paged_block_copy_fp8(uint8_t *k_cache, uint8_t *v_cache, const int32_t *block_pairs,
                         int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                         int block_size, int32_t *err_flag, void *stream) {
  if (block_size != kBlockSize) return PKV_ERR_BLOCK_SIZE;
  if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 16 != 0)
    return PKV_ERR_SHAPE;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_NULL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
  const int64_t block_vecs = (int64_t)num_kv_heads * kBlockSize * head_dim / 16;
  const int64_t total = (int64_t)num_pairs * block_vecs;
  const int threads = 256;
  const cudaError_t e = launch_pdl(
      block_copy_kernel, dim3(grid_for(total, threads)), dim3(threads), 0, (cudaStream_t)stream,
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), block_pairs, total,
      block_vecs, num_blocks, err_flag);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"
