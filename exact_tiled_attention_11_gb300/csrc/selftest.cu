// Self-test of the bounded pipeline waits (sm_103a).
//
// Every mbarrier wait in the library's kernels goes through mbar_wait
// (common.cuh): it gives up after a fixed time, records ATTN_DEVERR_WAIT_TIMEOUT
// in the device error word, raises the CTA's abort flag so that the other warps
// stop waiting too, and the kernel returns.  This kernel exercises exactly that
// path: its two warps wait on mbarriers that nothing ever arrives on.  The first
// wait to run out raises the shared abort flag, and the other then gives up
// through it (or at its own limit, if both run out together).  Nothing traps;
// the kernel returns after about one wait limit and the context stays usable.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(int *gave_up) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int w = threadIdx.x >> 5;
  // phase 0 of a fresh barrier completes only when one thread arrives, and none does
  const bool completed = mbar_wait(smem_u32(&bar[w]), 0, &abort_flag);
  if ((threadIdx.x & 31) == 0) gave_up[w] = completed ? 0 : 1;
}

}  // namespace

ATTN_DEFINE_ERROR_ACCESSOR(device_error_selftest)

cudaError_t launch_wait_timeout_selftest(int *gave_up, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(gave_up);
  return cudaGetLastError();
}

}  // namespace attn
