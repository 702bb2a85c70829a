// Self-checks of the library's error paths.
//
// Failure-detection check (moe_check_wait_timeout): the bounded mbarrier wait
// of the grouped-matmul pipelines, exercised on a barrier that nothing
// completes.  Thread 0 of warp 0 waits with the given limit and raises the
// shared abort flag when it expires; lane 0 of warp 1 waits on a second
// barrier with a far longer limit and must stop because of the flag, as the
// other roles of a pipeline do.  The kernel then records MOE_ERR_TIMEOUT.
//
// Bounds-check check (moe_check_bounds): one thread asks the kernels' bounds
// check about index n of an n-element range, and accesses nothing.  The
// bounds-checking build records MOE_ERR_BOUNDS; the release build has no
// check, and the status stays MOE_OK.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bars[2];
  __shared__ uint32_t abort_flag;
  const int tid = threadIdx.x;
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  volatile uint32_t* abort = &abort_flag;
  bool expired = false;
  if (tid == 0) {
    expired = !mbar_wait_bounded(smem_u32(&bars[0]), 0, abort, timeout_ns);   // nothing arrives
  } else if (tid == 32) {
    // gives up only through the flag: its own limit is far beyond the first wait's
    mbar_wait_bounded(smem_u32(&bars[1]), 0, abort, timeout_ns + 2000000000ull);
  }
  __syncthreads();
  if (tid == 0 && expired && abort_flag) set_status(status, MOE_ERR_TIMEOUT);
}

__global__ void bounds_check_kernel(uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = 1 + threadIdx.x;   // index n of an n-element range: one past the end
  (void)in_bounds(n, n, status);
}

}  // namespace

moe_status_t launch_bounds_check(uint32_t* status, cudaStream_t s) {
  return launch_pdl(bounds_check_kernel, dim3(1), dim3(1), 0, s, 1, status) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t launch_wait_timeout_check(uint32_t* status, uint64_t timeout_ns, cudaStream_t s) {
  return launch_pdl(wait_timeout_kernel, dim3(1), dim3(64), 0, s, 1, status, timeout_ns) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

}  // namespace moe
