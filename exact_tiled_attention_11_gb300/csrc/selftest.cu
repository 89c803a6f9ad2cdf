// Diagnostics (sm_103a): a self-test of the bounded pipeline waits, and a clock probe.
//
// Every mbarrier wait in the library's kernels goes through mbar_wait
// (common.cuh): it gives up after a fixed time, records ATTN_DEVERR_WAIT_TIMEOUT
// in the device error word, raises the CTA's abort flag so that the other warps
// stop waiting too, and the kernel returns.  This kernel exercises exactly that
// path: its two warps wait on mbarriers that nothing ever arrives on.  The first
// wait to run out raises the shared abort flag, and the other then gives up
// through it (or at its own limit, if both run out together).  Nothing traps;
// the kernel returns after about one wait limit and the context stays usable.
//
// The clock probe records %globaltimer (ns) and %clock64 (SM cycles) on one SM.
// Two probes around a stretch of work on one stream give the average SM clock
// over it.  %clock64 is a per-SM counter, so the second probe records on the SM
// the first one used: every block reads %smid, and only the first block on that
// SM (claimed through an atomic on the output) writes.
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

// out: {globaltimer, clock64, smid, claim}; match: NULL (any SM) or an earlier probe's out
__global__ void __launch_bounds__(32) clock_probe_kernel(unsigned long long *out, const unsigned long long *match) {
  if (threadIdx.x != 0) return;
  unsigned int smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  if (match != nullptr && smid != static_cast<unsigned int>(match[2])) return;
  if (atomicCAS(&out[3], 0ull, 1ull) != 0ull) return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  out[0] = t;
  out[1] = static_cast<unsigned long long>(clock64());
  out[2] = smid;
}

}  // namespace

ATTN_DEFINE_ERROR_ACCESSOR(device_error_selftest)

cudaError_t launch_wait_timeout_selftest(int *gave_up, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(gave_up);
  return cudaGetLastError();
}

cudaError_t launch_clock_probe(unsigned long long *out, const unsigned long long *match, int blocks,
                               cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(out, 0, 4 * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  clock_probe_kernel<<<blocks, 32, 0, stream>>>(out, match);
  return cudaGetLastError();
}

}  // namespace attn
