// Shared device helpers of libpagedkv.so (CUDA, sm_103a).
#pragma once

#include <atomic>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kBlockSize = 16;  // tokens per physical KV block

// Record a device-side error bit (never traps).
__device__ __forceinline__ void flag_error(int32_t *err, int bit) {
  if (err) atomicOr(err, bit);
}

// 16-byte read-only load of streamed data: bypass L1 allocation; the KV cache is read
// once per step so L1 reuse is nil.
// L2 policy for data read once (streamed KV tiles): its lines are the first replaced, so
// the lines other data keeps (partial results, queries) survive the stream.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy for data written now and read back soon by another kernel (split-K partial
// results): its lines are replaced last, so the streamed KV tiles do not push them to DRAM.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// fp32 store with an L2 cache policy.
__device__ __forceinline__ void st_f32_hint(float *p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol)
               : "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// The same with an L2 cache policy (see l2_evict_first_policy).
__device__ __forceinline__ uint4 ld_stream_v4_hint(const void *p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

// bf16 pair (one 32-bit word, low half = lower address) -> two fp32.  Exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&h);
}

// Programmatic dependent launch.  Every kernel of this library is launched with
// launch_pdl, so it may become resident while the previous kernel on the stream is
// still running; it calls pdl_wait() before it touches any memory, which returns once
// that kernel has completed and its writes are visible (at once when there is no such
// kernel).  pdl_trigger() lets the next kernel start its own launch early.  Only launch
// latency and prologues overlap; no data dependency is relaxed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifdef __CUDACC__
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}
#endif

// Host-side helpers ------------------------------------------------------------------
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count();  // cached per device

// Per-device launch set-up (a kernel attribute, an occupancy figure), computed on the
// first call that runs with a device current and kept for that device: `compute`
// returns a positive value to keep, or a non-positive one (an error) that is returned
// and not kept.  Safe under concurrent first calls from several host threads (each may
// compute; every access is atomic); devices beyond the table are not cached.
constexpr int kMaxDevices = 64;
template <typename F>
int per_device_setup(std::atomic<int> (&slots)[kMaxDevices], F compute) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (dev >= 0 && dev < kMaxDevices) {
    const int v = slots[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
  }
  const int v = compute();
  if (v > 0 && dev >= 0 && dev < kMaxDevices) slots[dev].store(v, std::memory_order_release);
  return v;
}

}  // namespace pkv
