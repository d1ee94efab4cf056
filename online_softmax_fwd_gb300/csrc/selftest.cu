// Self-test of the kernels' bounded waits: a kernel whose two warps wait on
// mbarriers that nothing completes, through the same wait function the
// attention kernels use. Warp 0 gives up after the given limit, records
// ATTN_ERR_TIMEOUT in the status word and raises the CTA's abort flag; warp 1,
// with 64 times the limit, must return early on that flag. The kernel ends
// after about one limit, and the context stays usable.
#include <cuda_runtime.h>

#include "fwd_bf16.cuh"
#include "fwd_dispatch.h"

namespace attn {

__global__ void wait_timeout_selftest_kernel(unsigned int* status, long long limit_cycles) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t abort_word;
  volatile uint32_t* abort_flag = &abort_word;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bars[0]), 1);
    mbar_init(smem_addr(&bars[1]), 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on either barrier
  if (warp == 0)
    wait_bar_limit(smem_addr(&bars[0]), 0, abort_flag, status, 60, limit_cycles);
  else
    wait_bar_limit(smem_addr(&bars[1]), 0, abort_flag, status, 61, 64 * limit_cycles);
  __syncthreads();
}

cudaError_t launch_wait_timeout_selftest(unsigned int* status, long long limit_cycles, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 64, 0, stream>>>(status, limit_cycles);
  return cudaGetLastError();
}

}  // namespace attn
