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
// memory, quietly use the wrong memory). Its device address is looked up with
// cudaGetSymbolAddress, with the device current, the first time the entry
// point runs in a CUDA context, and looked up again whenever the current
// context differs from the one the address was taken in (a device reset
// creates a new context, in which the module and its array may sit at a new
// address).
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB: M * K <= 16,777,216
constexpr size_t kMaxElems = kScratchBytes / 2;      // 2 bytes of workspace per activation

static __device__ __align__(256) unsigned char g_w4a8_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  CUcontext ctx;   // the context the address belongs to
  void* ptr;
};
Cached g_scratch[kMaxDevices] = {};

using CtxGetCurrent = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, found through the runtime (looked up once).
CtxGetCurrent ctx_get_current() {
  static const CtxGetCurrent fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<CtxGetCurrent>(f);
  }();
  return fn;
}

// Device address of the array in the current device's current context.
cudaError_t scratch_ptr(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrent get = ctx_get_current();
  if (get == nullptr) return cudaErrorNotSupported;
  // null until the runtime has made a context current on this thread
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lk(g_mu);
  if (ctx == nullptr || g_scratch[dev].ptr == nullptr || g_scratch[dev].ctx != ctx) {
    // the lookup also sets up the runtime's context on the device if needed
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_w4a8_scratch);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
    g_scratch[dev].ctx = ctx;
    g_scratch[dev].ptr = p;
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" w4_status w4a8_gemm_noalloc(const void* qx, const float* x_scale, const void* qweight,
                                       const void* w_scale, int32_t w_scale_dtype, int32_t group,
                                       const void* bias, void* y, int64_t M, int64_t N, int64_t K,
                                       void* stream) {
  // the size limit, checked without forming M * K (which could wrap)
  if (M > 0 && K > 0 && (static_cast<uint64_t>(K) > kMaxElems ||
                         static_cast<uint64_t>(M) > kMaxElems / static_cast<uint64_t>(K))) {
    char msg[220];
    snprintf(msg, sizeof(msg),
             "w4a8_gemm_noalloc: M=%lld, K=%lld needs more than its fixed %zu-byte workspace "
             "(M*K must be at most %zu); use w4a8_gemm with a workspace",
             (long long)M, (long long)K, kScratchBytes, kMaxElems);
    return w4::report_error(W4_ERR_UNSUPPORTED, msg);
  }
  void* ws = nullptr;
  if (M > 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && stream != nullptr) {
      // the array is looked up on the current device: the stream must belong to it
      int sdev = 0;
      e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev);
      if (e == cudaSuccess && sdev != dev) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "w4a8_gemm_noalloc: the stream belongs to device %d but device %d is current; make the "
                 "stream's device current before the call",
                 sdev, dev);
        return w4::report_error(W4_ERR_CUDA, msg);
      }
    }
    if (e == cudaSuccess) e = scratch_ptr(dev, &ws);
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
