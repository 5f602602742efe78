// Self-test of the kernels' failure path: a bounded wait that runs out.
//
// Every wait inside the library's kernels (on a TMA copy's completion, a ring slot, a
// tensor-core product) is bounded; when one gives up, the kernel raises its CTA's abort
// flag, ORs PKV_DEV_TIMEOUT into the caller's error word and returns, so the context stays
// usable.  Nothing in a correct call ever gets there, so this entry point makes it
// happen on purpose, without any fault: one thread waits, with the same helpers and a
// caller-chosen short limit, on an mbarrier phase that nothing completes.
#include <cuda_runtime.h>

#include "pagedkv.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

__global__ void wait_timeout_kernel(int32_t *err, long long limit, int spin, long long *result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);  // one arrival completes phase 0; nothing arrives
  abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const long long t0 = clock64();
  const bool ok = spin ? mbar_spin_wait(b, 0u, &abort_flag, err, limit)
                       : mbar_wait(b, 0u, &abort_flag, err, limit);
  result[0] = ok ? 1 : 0;
  result[1] = clock64() - t0;
  result[2] = abort_flag;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_selftest_bounded_wait(int32_t *err_flag, long long *result,
                                         long long limit_cycles, int use_spin, void *stream) {
  if (!err_flag || !result) return PKV_ERR_NULL;
  if (limit_cycles <= 0 || limit_cycles > pkv::kWaitCycles) return PKV_ERR_SHAPE;
  pkv::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err_flag, limit_cycles,
                                                               use_spin ? 1 : 0, result);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
