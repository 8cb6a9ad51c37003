// placeholder until the tensor-core kernels land
#include "common.cuh"
#include "launch.h"
namespace w4 {
cudaError_t launch_w4a8_dense(const W4A8Args&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_w4afp8_experts(const W4A8Args&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace w4
