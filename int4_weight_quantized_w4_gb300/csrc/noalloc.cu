// w4a8_gemm_noalloc: the W4A8 GEMM for callers that cannot allocate device
// memory.
//
// w4a8_gemm needs a device workspace (the int8 activations widened once to
// exact fp16, M * K * 2 bytes) that the caller allocates. Some callers cannot
// call cudaMalloc or any allocator: code that runs inside a framework that
// owns all device memory, a plugin given only the tensors it reads and writes,
// or code on a path where allocating would synchronize the device or is
// simply forbidden. This entry point serves them with a fixed workspace that
// is part of the library itself: a file-scope device array that every GPU
// which loads the library holds until the process exits.
//
// The array is a host-side symbol, not a device address: handing its name to
// a kernel from host code would fault (or, where the GPU can reach host
// memory, quietly use the wrong memory). Its device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, the first
// time the entry point runs on that device.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB: M * K <= 16,777,216

static __device__ __align__(256) unsigned char g_w4a8_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the array (looked up once).
cudaError_t scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_w4a8_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" w4_status w4a8_gemm_noalloc(const void* qx, const float* x_scale, const void* qweight,
                                       const void* w_scale, int32_t w_scale_dtype, int32_t group,
                                       const void* bias, void* y, int64_t M, int64_t N, int64_t K,
                                       void* stream) {
  if (M > 0 && K > 0) {
    const size_t need = w4_workspace_bytes(W4_OP_W4A8, M, N, K, group);
    if (need > kScratchBytes) {
      char msg[200];
      snprintf(msg, sizeof(msg),
               "w4a8_gemm_noalloc: M*K = %lld needs %zu bytes of workspace, above its fixed %zu "
               "(M*K must be at most %zu); use w4a8_gemm with a workspace",
               (long long)M * (long long)K, need, kScratchBytes, kScratchBytes / 2);
      return w4::report_error(W4_ERR_UNSUPPORTED, msg);
    }
  }
  void* ws = nullptr;
  if (M > 0) {
    const cudaError_t e = scratch_ptr(&ws);
    if (e != cudaSuccess) {
      char msg[200];
      snprintf(msg, sizeof(msg), "w4a8_gemm_noalloc: looking up the built-in workspace failed: %s",
               cudaGetErrorString(e));
      return w4::report_error(W4_ERR_CUDA, msg);
    }
  }
  // The widening pass overwrites every byte of the workspace it later reads,
  // so nothing in the array needs to start at zero.
  return w4a8_gemm(qx, x_scale, qweight, w_scale, w_scale_dtype, group, bias, y, M, N, K, ws, kScratchBytes,
                   stream);
}
