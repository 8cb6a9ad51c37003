// Self-test of the bounded-wait machinery used by the pipelined kernels: one
// thread waits on an mbarrier that nothing arrives at. The wait gives up
// after `limit` polls, records W4_ERR_TIMEOUT in the status word and returns,
// so the context stays usable.
#include "common.cuh"
#include "launch.h"

namespace w4 {
namespace {

__global__ void bounded_wait_kernel(long long limit, unsigned int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait_bounded(&bar, 0, limit, status);
  __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(long long limit, unsigned int* status, cudaStream_t s) {
  bounded_wait_kernel<<<1, 32, 0, s>>>(limit, status);
  return cudaGetLastError();
}

}  // namespace w4
