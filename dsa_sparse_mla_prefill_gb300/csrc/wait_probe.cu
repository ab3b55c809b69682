// A bounded wait that runs out, on purpose: the check that a kernel whose
// barrier never completes gives up after the wait limit, records the timeout
// in the device error counters, releases the tensor memory it holds and
// returns, leaving the context usable (dsa_debug_wait_timeout).  One CTA:
// warp 0 holds 32 TMEM columns for the duration, warp 1 waits on an mbarrier
// that nothing arrives on, with the same bounded wait every pipeline uses.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace probe {

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) mbar_wait_warp(&bar, 0, &abort_flag, err);   // nothing completes phase 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem_base, 32);
}

}  // namespace probe

int launch_wait_timeout(unsigned int* err, cudaStream_t stream) {
  probe::wait_timeout_kernel<<<1, 64, 0, stream>>>(err);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace dsa
