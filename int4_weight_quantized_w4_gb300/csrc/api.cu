// Public C entry points: host-side argument validation, then one launch.
// Nothing is launched when validation fails; the status says why and
// w4_last_error() holds a message for the calling thread.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

thread_local char g_last_error[512] = "";

w4_status fail(w4_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

w4_status ok() {
  g_last_error[0] = '\0';
  return W4_OK;
}

w4_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(W4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device status word; bounded waits in the kernels record timeouts here.
__device__ unsigned int g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};

// Address of this device's status word (looked up once per device).
cudaError_t status_ptr(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

// Shared checks for the packed-weight GEMMs. On success *geff is the
// effective group (K for -1).
w4_status check_dims_group(int64_t M, int64_t N, int64_t K, int32_t group, int32_t* geff) {
  if (M < 0 || N <= 0 || K <= 0) return fail(W4_ERR_SHAPE, "sizes must be M >= 0, N > 0, K > 0 (M=%lld N=%lld K=%lld)",
                                             (long long)M, (long long)N, (long long)K);
  if (N % 8 != 0 || K % 8 != 0)
    return fail(W4_ERR_ALIGN, "N and K must be multiples of 8, got N=%lld K=%lld", (long long)N, (long long)K);
  if (group == -1) {
    if (K > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "K=%lld too large for one group", (long long)K);
    *geff = static_cast<int32_t>(K);
  } else {
    if (group <= 0 || K % group != 0)
      return fail(W4_ERR_GROUP, "group %d must be -1 or a positive divisor of K=%lld", group, (long long)K);
    *geff = group;
  }
  return W4_OK;
}

}  // namespace

namespace w4 {
// Lets other translation units report a status with a message for w4_last_error().
w4_status report_error(w4_status st, const char* msg) { return fail(st, "%s", msg); }
}  // namespace w4

extern "C" {

const char* w4_last_error(void) { return g_last_error; }

const char* w4_status_string(int32_t st) {
  switch (st) {
    case W4_OK: return "W4_OK";
    case W4_ERR_NULL: return "W4_ERR_NULL";
    case W4_ERR_ALIGN: return "W4_ERR_ALIGN";
    case W4_ERR_GROUP: return "W4_ERR_GROUP";
    case W4_ERR_DTYPE: return "W4_ERR_DTYPE";
    case W4_ERR_UNSUPPORTED: return "W4_ERR_UNSUPPORTED";
    case W4_ERR_SHAPE: return "W4_ERR_SHAPE";
    case W4_ERR_CUDA: return "W4_ERR_CUDA";
    case W4_ERR_TIMEOUT: return "W4_ERR_TIMEOUT";
    case W4_ERR_WORKSPACE: return "W4_ERR_WORKSPACE";
    default: return "W4_ERR_UNKNOWN";
  }
}

w4_status w4_quant_act_per_token(const void* x, int32_t x_dtype, int64_t M, int64_t K, int32_t q_dtype,
                                 void* q, float* scale, void* stream) {
  if (M < 0 || K <= 0) return fail(W4_ERR_SHAPE, "sizes must be M >= 0, K > 0 (M=%lld K=%lld)", (long long)M, (long long)K);
  if (x_dtype != W4_BF16 && x_dtype != W4_FP16) return fail(W4_ERR_DTYPE, "x_dtype must be W4_BF16 or W4_FP16");
  if (q_dtype != W4_INT8 && q_dtype != W4_FP8_E4M3) return fail(W4_ERR_DTYPE, "q_dtype must be W4_INT8 or W4_FP8_E4M3");
  if (K % 8 != 0) return fail(W4_ERR_ALIGN, "K must be a multiple of 8, got %lld", (long long)K);
  if (M == 0) return ok();
  if (!x || !q || !scale) return fail(W4_ERR_NULL, "x, q and scale must be non-NULL");
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return fail(W4_ERR_ALIGN, "x and q must be 16-byte aligned, scale 4-byte aligned");
  if (M > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "M too large");
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  return from_cuda(w4::launch_quant_per_token(x, x_dtype == W4_FP16, M, K, q_dtype == W4_FP8_E4M3, q, scale, status,
                                              static_cast<cudaStream_t>(stream)),
                   "w4_quant_act_per_token launch");
}

size_t w4_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int32_t group) {
  if (M <= 0 || K <= 0) return 0;
  if (op == W4_OP_W4A8) {
    // room for split-K partial sums too when this shape would be split
    const int64_t g = group == -1 ? K : group;
    if (N > 0 && N % 8 == 0 && g > 0 && K % g == 0) return w4::w4a8_workspace_bytes_split(M, N, K, static_cast<int32_t>(g));
    return w4::w4a8_workspace_bytes(M, K);
  }
  if (op == W4_OP_W4AFP8_MOE) return w4::w4a8_workspace_bytes(M, K);
  if (op == W4_OP_MOE_ROUTE) return (N > 0 && N <= 1024) ? w4::moe_route_workspace_bytes(M, static_cast<int32_t>(N)) : 0;
  return 0;
}

static w4_status check_workspace(void* ws, size_t bytes, int64_t rows, int64_t K) {
  const size_t need = w4::w4a8_workspace_bytes(rows, K);
  if (ws == nullptr || bytes < need || !aligned(ws, 16))
    return fail(W4_ERR_WORKSPACE, "workspace must be 16-byte aligned and at least %zu bytes (got %zu)", need, bytes);
  return W4_OK;
}

static w4_status w4a8_common(const void* qx, const float* x_scale, const void* qweight, const void* w_scale,
                             int32_t w_scale_dtype, int32_t group, const void* bias, void* out,
                             int64_t M, int64_t N, int64_t K, bool partials, void* workspace,
                             size_t workspace_bytes, void* stream) {
  int32_t g = 0;
  w4_status st = check_dims_group(M, N, K, group, &g);
  if (st != W4_OK) return st;
  if (!partials && w_scale_dtype != W4_FP16)
    return fail(W4_ERR_DTYPE, "w4a8_gemm reads weight scales as fp16; pass fp16 scales (W4_FP16)");
  if (K % 16 != 0 || g % 16 != 0)
    return fail(W4_ERR_UNSUPPORTED, "w4a8 tiles need K and the group to be multiples of 16 (K=%lld group=%d)",
                (long long)K, g);
  if (partials && g > 16384) return fail(W4_ERR_UNSUPPORTED, "partials need group <= 16384 to stay exact");
  if (M == 0) return ok();
  if (!qx || !qweight || !out || (!partials && (!x_scale || !w_scale)))
    return fail(W4_ERR_NULL, "required pointer is NULL");
  if (!aligned(qx, 16) || !aligned(qweight, 16) || !aligned(out, 16) ||
      (!partials && (!aligned(w_scale, 8) || !aligned(x_scale, 4))) || (bias && !aligned(bias, 8)))
    return fail(W4_ERR_ALIGN, "matrices must be 16-byte aligned, vectors 8-byte aligned");
  if (M > INT32_MAX || N > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "M or N too large");
  st = check_workspace(workspace, workspace_bytes, M, K);
  if (st != W4_OK) return st;
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  w4::W4A8Args a{qx, x_scale, qweight, w_scale, partials ? nullptr : bias, out, nullptr, 1, M, N, K, g, partials,
                 status, workspace, false, false, workspace_bytes};
  return from_cuda(w4::launch_w4a8_dense(a, static_cast<cudaStream_t>(stream)), "w4a8 launch");
}

w4_status w4a8_gemm(const void* qx, const float* x_scale, const void* qweight, const void* w_scale,
                    int32_t w_scale_dtype, int32_t group, const void* bias, void* y,
                    int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
  return w4a8_common(qx, x_scale, qweight, w_scale, w_scale_dtype, group, bias, y, M, N, K, false, workspace,
                     workspace_bytes, stream);
}

w4_status w4a8_gemm_bf16in(const void* x, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                           int32_t group, const void* bias, void* y, float* x_scale, int64_t M, int64_t N, int64_t K,
                           void* workspace, size_t workspace_bytes, void* stream) {
  int32_t g = 0;
  w4_status st = check_dims_group(M, N, K, group, &g);
  if (st != W4_OK) return st;
  if (w_scale_dtype != W4_FP16)
    return fail(W4_ERR_DTYPE, "w4a8_gemm_bf16in reads weight scales as fp16; pass fp16 scales (W4_FP16)");
  if (K % 16 != 0 || g % 16 != 0)
    return fail(W4_ERR_UNSUPPORTED, "w4a8 tiles need K and the group to be multiples of 16 (K=%lld group=%d)",
                (long long)K, g);
  if (M == 0) return ok();
  if (!x || !qweight || !w_scale || !y || !x_scale) return fail(W4_ERR_NULL, "required pointer is NULL");
  if (!aligned(x, 16) || !aligned(qweight, 16) || !aligned(y, 16) || !aligned(w_scale, 8) ||
      !aligned(x_scale, 4) || (bias && !aligned(bias, 8)))
    return fail(W4_ERR_ALIGN, "matrices must be 16-byte aligned, vectors 8-byte aligned");
  if (M > INT32_MAX || N > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "M or N too large");
  st = check_workspace(workspace, workspace_bytes, M, K);
  if (st != W4_OK) return st;
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = w4::launch_quant_widen(x, M, K, false, workspace, x_scale, status, s);
  if (e != cudaSuccess) return from_cuda(e, "quantize-and-widen launch");
  w4::W4A8Args a{nullptr, x_scale, qweight, w_scale, bias, y, nullptr, 1, M, N, K, g, false, status, workspace, true,
                 false, workspace_bytes};
  return from_cuda(w4::launch_w4a8_dense(a, s), "w4a8 launch");
}

w4_status w4a8_group_partials(const void* qx, const void* qweight, int32_t group, int32_t* partials,
                              int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return w4a8_common(qx, nullptr, qweight, nullptr, W4_FP16, group, nullptr, partials, M, N, K, true, workspace,
                     workspace_bytes, stream);
}

// The checks of w4a16_gemm; `check_ptrs` false stops after the ones that do
// not look at the pointers (a zero-size call).
static w4_status check_w4a16(const void* x, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                             const void* zeros, const void* bias, const void* y, int64_t M, int64_t N, int64_t K,
                             int32_t group, int32_t* g, bool check_ptrs) {
  w4_status st = check_dims_group(M, N, K, group, g);
  if (st != W4_OK) return st;
  if (w_scale_dtype != W4_FP16 && w_scale_dtype != W4_BF16)
    return fail(W4_ERR_DTYPE, "w4a16_gemm scales must be W4_FP16 or W4_BF16");
  if (K % 64 != 0 || *g % 64 != 0)
    return fail(W4_ERR_UNSUPPORTED, "w4a16 tiles need K and the group to be multiples of 64 (K=%lld group=%d)",
                (long long)K, *g);
  if (w4::w4a16_smem_bytes(N, K, *g) > 227 * 1024)
    return fail(W4_ERR_UNSUPPORTED, "w4a16 keeps a token row of x in shared memory: K=%lld is too long", (long long)K);
  if (!check_ptrs) return W4_OK;
  if (!x || !qweight || !w_scale || !y) return fail(W4_ERR_NULL, "x, qweight, w_scale and y must be non-NULL");
  if (!aligned(x, 16) || !aligned(qweight, 16) || !aligned(y, 8) || !aligned(w_scale, 16) ||
      (zeros && !aligned(zeros, 16)) || (bias && !aligned(bias, 8)))
    return fail(W4_ERR_ALIGN, "x, qweight, scales and zeros must be 16-byte aligned; y and bias 8-byte aligned");
  if (M > INT32_MAX || N > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "M or N too large");
  return W4_OK;
}

// The device address of page-locked (registered or cudaHostAlloc'd) host
// memory, or null for anything else: pageable memory, device memory, or a
// pointer the runtime does not know.
static const void* page_locked(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();   // clear the error the query left
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

static w4_status launch_w4a16_checked(const void* x, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                                      const void* zeros, int32_t g, const void* bias, void* y, int64_t M, int64_t N,
                                      int64_t K, cudaStream_t s, const void* x_host = nullptr,
                                      void* y_host = nullptr) {
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  w4::W4A16Args a{x, qweight, w_scale, w_scale_dtype == W4_BF16, zeros, bias, y, M, N, K, g, status};
  a.x_host = x_host;
  a.y_host = y_host;
  return from_cuda(w4::launch_w4a16(a, s), "w4a16 launch");
}

w4_status w4a16_gemm(const void* x, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                     const void* zeros, int32_t group, const void* bias, void* y,
                     int64_t M, int64_t N, int64_t K, void* stream) {
  int32_t g = 0;
  w4_status st = check_w4a16(x, qweight, w_scale, w_scale_dtype, zeros, bias, y, M, N, K, group, &g, M > 0);
  if (st != W4_OK) return st;
  if (M == 0) return ok();
  return launch_w4a16_checked(x, qweight, w_scale, w_scale_dtype, zeros, g, bias, y, M, N, K,
                              static_cast<cudaStream_t>(stream));
}

w4_status w4a16_gemm_host(const void* x_host, void* x_dev, const void* qweight, const void* w_scale,
                          int32_t w_scale_dtype, const void* zeros, int32_t group, const void* bias, void* y_dev,
                          void* y_host, int64_t M, int64_t N, int64_t K, void* stream) {
  int32_t g = 0;
  w4_status st = check_w4a16(x_dev, qweight, w_scale, w_scale_dtype, zeros, bias, y_dev, M, N, K, group, &g, M > 0);
  if (st != W4_OK) return st;
  if (M == 0) return ok();
  if (!x_host || !y_host) return fail(W4_ERR_NULL, "x_host and y_host must be non-NULL");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = static_cast<size_t>(M) * K * 2, yb = static_cast<size_t>(M) * N * 2;
  // page-locked host buffers (the device address of each, asked per call):
  // the L2-prefetch grid copies x in and the GEMV writes y out as well, so
  // the call launches no more grids than w4a16_gemm
  const void* xh = page_locked(x_host);
  void* yh = const_cast<void*>(page_locked(y_host));
  if (xh && yh && aligned(xh, 16) && aligned(yh, 2) && xb % 16 == 0)
    return launch_w4a16_checked(x_dev, qweight, w_scale, w_scale_dtype, zeros, g, bias, y_dev, M, N, K, s, xh, yh);
  cudaError_t e = cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return from_cuda(e, "copy of x to the device");
  st = launch_w4a16_checked(x_dev, qweight, w_scale, w_scale_dtype, zeros, g, bias, y_dev, M, N, K, s);
  if (st != W4_OK) return st;
  return from_cuda(cudaMemcpyAsync(y_host, y_dev, yb, cudaMemcpyDeviceToHost, s), "copy of y to the host");
}

static w4_status check_experts(int64_t R, int64_t N, int64_t K, int32_t group, int32_t E, int32_t w_scale_dtype,
                               int32_t* g) {
  w4_status st = check_dims_group(R, N, K, group, g);
  if (st != W4_OK) return st;
  if (E <= 0) return fail(W4_ERR_SHAPE, "E must be positive, got %d", E);
  if (w_scale_dtype != W4_FP16) return fail(W4_ERR_DTYPE, "expert weight scales must be fp16 (W4_FP16)");
  if (K % 32 != 0 || *g % 16 != 0)
    return fail(W4_ERR_UNSUPPORTED, "expert tiles need K % 32 == 0 and the group a multiple of 16 (K=%lld group=%d)",
                (long long)K, *g);
  if ((R + 127) / 128 + E > 65535) return fail(W4_ERR_UNSUPPORTED, "too many row tiles plus experts");
  return W4_OK;
}

w4_status w4afp8_moe_grouped_gemm(const void* qx, const float* x_scale, const int32_t* expert_offsets, int32_t E,
                                  const void* qweight, const void* w_scale, int32_t w_scale_dtype, int32_t group,
                                  void* y, int64_t R, int64_t N, int64_t K, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  int32_t g = 0;
  w4_status st = check_experts(R, N, K, group, E, w_scale_dtype, &g);
  if (st != W4_OK) return st;
  if (R == 0) return ok();
  if (!qx || !x_scale || !expert_offsets || !qweight || !w_scale || !y)
    return fail(W4_ERR_NULL, "required pointer is NULL");
  if (!aligned(qx, 16) || !aligned(qweight, 16) || !aligned(y, 16) || !aligned(w_scale, 8) ||
      !aligned(x_scale, 4) || !aligned(expert_offsets, 4))
    return fail(W4_ERR_ALIGN, "matrices must be 16-byte aligned, vectors aligned to their element size");
  if (R > INT32_MAX || N > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "R or N too large");
  st = check_workspace(workspace, workspace_bytes, R, K);
  if (st != W4_OK) return st;
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  w4::W4A8Args a{qx, x_scale, qweight, w_scale, nullptr, y, expert_offsets, E, R, N, K, g, false, status, workspace,
                 false, w4::w4afp8_fp8_path(g)};
  return from_cuda(w4::launch_w4afp8_experts(a, static_cast<cudaStream_t>(stream)), "w4afp8 experts launch");
}

w4_status w4_quantize_groupwise(const void* w, int32_t w_dtype, int64_t N, int64_t K, int32_t group,
                                void* packed, float* scale, float* zero, void* stream) {
  if (N < 0 || K <= 0) return fail(W4_ERR_SHAPE, "sizes must be N >= 0, K > 0 (N=%lld K=%lld)", (long long)N,
                                   (long long)K);
  if (w_dtype != W4_BF16 && w_dtype != W4_FP16) return fail(W4_ERR_DTYPE, "w must be W4_BF16 or W4_FP16");
  const int64_t g = group == -1 ? K : group;
  if (g <= 0 || K % g != 0 || g > INT32_MAX)
    return fail(W4_ERR_GROUP, "group %d must be -1 or a positive divisor of K=%lld", group, (long long)K);
  if (K % 2 != 0 || g % 2 != 0)
    return fail(W4_ERR_UNSUPPORTED, "K and the group must be even (two codes per byte), got K=%lld group=%lld",
                (long long)K, (long long)g);
  if (N == 0) return ok();
  if (!w || !packed || !scale || !zero) return fail(W4_ERR_NULL, "w, packed, scale and zero must be non-NULL");
  if (!aligned(w, 4) || !aligned(scale, 4) || !aligned(zero, 4))
    return fail(W4_ERR_ALIGN, "w, scale and zero must be 4-byte aligned");
  return from_cuda(w4::launch_quantize_groupwise(w, w_dtype == W4_FP16, N, K, static_cast<int32_t>(g),
                                                 static_cast<uint8_t*>(packed), scale, zero,
                                                 static_cast<cudaStream_t>(stream)),
                   "quantize_groupwise launch");
}

w4_status w4_repack_s4_to_uint4b8(const void* src, void* dst, int64_t n_bytes, void* stream) {
  if (n_bytes < 0) return fail(W4_ERR_SHAPE, "n_bytes must be >= 0");
  if (n_bytes == 0) return ok();
  if (!src || !dst) return fail(W4_ERR_NULL, "src and dst must be non-NULL");
  if (!aligned(src, 16) || !aligned(dst, 16)) return fail(W4_ERR_ALIGN, "src and dst must be 16-byte aligned");
  return from_cuda(w4::launch_xor88(src, dst, n_bytes, static_cast<cudaStream_t>(stream)), "repack launch");
}

w4_status w4_moe_route(const void* logits, int32_t logits_f32, int64_t T, int32_t E, int32_t top_k,
                       int32_t renormalize, int32_t* topk_ids, float* topk_weights, int32_t* offsets,
                       int32_t* row_token, int32_t* row_of, void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0) return fail(W4_ERR_SHAPE, "T must be >= 0");
  if (E < 1 || E > 1024) return fail(W4_ERR_UNSUPPORTED, "E must be in [1, 1024], got %d", E);
  if (top_k < 1 || top_k > E || top_k > 64)
    return fail(W4_ERR_SHAPE, "top_k must be in [1, min(E, 64)], got %d (E=%d)", top_k, E);
  if (T * top_k > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "T * top_k rows must fit in int32");
  if (T == 0) return ok();
  if (!logits || !topk_ids || !topk_weights || !offsets || !row_token || !row_of)
    return fail(W4_ERR_NULL, "logits and every output must be non-NULL");
  if (!aligned(logits, logits_f32 ? 4 : 2) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4) ||
      !aligned(offsets, 4) || !aligned(row_token, 4) || !aligned(row_of, 4))
    return fail(W4_ERR_ALIGN, "route buffers must be aligned to their element size");
  const size_t need = w4::moe_route_workspace_bytes(T, E);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 4))
    return fail(W4_ERR_WORKSPACE, "route workspace must be 4-byte aligned and at least %zu bytes (got %zu)", need,
                workspace_bytes);
  return from_cuda(w4::launch_moe_route(logits, logits_f32 == 0, T, E, top_k, renormalize != 0, topk_ids,
                                        topk_weights, offsets, row_token, row_of, workspace,
                                        static_cast<cudaStream_t>(stream)),
                   "moe route launch");
}

w4_status w4_moe_gather_quant_fp8(const void* x, int64_t T, int64_t K, const int32_t* row_token, int64_t R,
                                  void* q, float* scale, void* stream) {
  if (T < 0 || R < 0 || K <= 0) return fail(W4_ERR_SHAPE, "sizes must be T >= 0, R >= 0, K > 0");
  if (K % 8 != 0) return fail(W4_ERR_ALIGN, "K must be a multiple of 8, got %lld", (long long)K);
  if (R == 0) return ok();
  if (!x || !row_token || !q || !scale) return fail(W4_ERR_NULL, "x, row_token, q and scale must be non-NULL");
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4) || !aligned(row_token, 4))
    return fail(W4_ERR_ALIGN, "x and q must be 16-byte aligned; scale and row_token 4-byte aligned");
  if (R > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "R too large");
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  return from_cuda(w4::launch_quant_gather(x, T, K, row_token, R, true, false, q, scale, status,
                                           static_cast<cudaStream_t>(stream)),
                   "gather-quant launch");
}

w4_status w4afp8_moe_gemm_bf16in(const void* x, int64_t T, const int32_t* row_token, const int32_t* expert_offsets,
                                 int32_t E, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                                 int32_t group, void* y, float* x_scale, int64_t R, int64_t N, int64_t K,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  int32_t g = 0;
  w4_status st = check_experts(R, N, K, group, E, w_scale_dtype, &g);
  if (st != W4_OK) return st;
  if (T < 0) return fail(W4_ERR_SHAPE, "T must be >= 0");
  if (row_token == nullptr && R != T) return fail(W4_ERR_SHAPE, "without row_token R must equal T");
  if (R == 0) return ok();
  if (!x || !x_scale || !expert_offsets || !qweight || !w_scale || !y)
    return fail(W4_ERR_NULL, "required pointer is NULL");
  if (!aligned(x, 16) || !aligned(qweight, 16) || !aligned(y, 16) || !aligned(w_scale, 8) ||
      !aligned(x_scale, 4) || !aligned(expert_offsets, 4) || (row_token && !aligned(row_token, 4)))
    return fail(W4_ERR_ALIGN, "matrices must be 16-byte aligned, vectors aligned to their element size");
  if (R > INT32_MAX || N > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "R or N too large");
  st = check_workspace(workspace, workspace_bytes, R, K);
  if (st != W4_OK) return st;
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the fp8 path reads the gathered e4m3 codes from the workspace as they are;
  // the fp16 path (groups that are not multiples of 32) their widened values
  const bool fp8 = w4::w4afp8_fp8_path(g);
  e = w4::launch_quant_gather(x, T, K, row_token, R, true, !fp8, workspace, x_scale, status, s);
  if (e != cudaSuccess) return from_cuda(e, "gather-quant launch");
  w4::W4A8Args a{fp8 ? workspace : nullptr, x_scale, qweight, w_scale, nullptr, y, expert_offsets, E, R, N, K, g,
                 false, status, workspace, !fp8, fp8};
  return from_cuda(w4::launch_w4afp8_experts(a, s), "w4afp8 experts launch");
}

w4_status w4_moe_silu_mul_quant_fp8(const void* h, int64_t R, int64_t I, void* q, float* scale, void* act,
                                    void* stream) {
  if (R < 0 || I <= 0) return fail(W4_ERR_SHAPE, "sizes must be R >= 0, I > 0");
  if (I % 8 != 0) return fail(W4_ERR_ALIGN, "I must be a multiple of 8, got %lld", (long long)I);
  if (R == 0) return ok();
  if (!h || !q || !scale) return fail(W4_ERR_NULL, "h, q and scale must be non-NULL");
  if (!aligned(h, 16) || !aligned(q, 16) || !aligned(scale, 4) || (act && !aligned(act, 16)))
    return fail(W4_ERR_ALIGN, "h, q and act must be 16-byte aligned, scale 4-byte aligned");
  if (R > INT32_MAX || I / 8 > INT32_MAX) return fail(W4_ERR_UNSUPPORTED, "R or I too large");
  return from_cuda(w4::launch_silu_mul_quant(h, R, I, q, scale, act, static_cast<cudaStream_t>(stream)),
                   "silu-mul-quant launch");
}

w4_status w4_moe_combine(const void* y, int64_t R, int64_t H, const float* topk_weights, const int32_t* row_of,
                         int64_t T, int32_t top_k, void* out, void* stream) {
  if (R < 0 || T < 0 || H <= 0 || top_k < 1) return fail(W4_ERR_SHAPE, "sizes must be R, T >= 0, H > 0, top_k >= 1");
  if (H % 8 != 0) return fail(W4_ERR_ALIGN, "H must be a multiple of 8, got %lld", (long long)H);
  if (T == 0) return ok();
  if (!y || !topk_weights || !row_of || !out) return fail(W4_ERR_NULL, "y, topk_weights, row_of, out must be non-NULL");
  if (!aligned(y, 16) || !aligned(out, 16) || !aligned(topk_weights, 4) || !aligned(row_of, 4))
    return fail(W4_ERR_ALIGN, "y and out must be 16-byte aligned; weights and row_of 4-byte aligned");
  if (H / 8 > INT32_MAX || T * (H / 8) > (int64_t(1) << 40)) return fail(W4_ERR_UNSUPPORTED, "T or H too large");
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  return from_cuda(w4::launch_moe_combine(y, R, H, topk_weights, row_of, T, top_k, out, status,
                                          static_cast<cudaStream_t>(stream)),
                   "combine launch");
}

static w4_status check_table(int64_t V, int64_t D, int32_t group, int32_t* geff) {
  if (V <= 0 || D <= 0) return fail(W4_ERR_SHAPE, "table sizes must be V > 0, D > 0 (V=%lld D=%lld)", (long long)V,
                                    (long long)D);
  const int64_t g = group == -1 ? D : group;
  if (g <= 0 || D % g != 0 || g > INT32_MAX)
    return fail(W4_ERR_GROUP, "group %d must be -1 or a positive divisor of D=%lld", group, (long long)D);
  if (D % 8 != 0 || g % 8 != 0)
    return fail(W4_ERR_ALIGN, "D and the group must be multiples of 8 (D=%lld group=%lld)", (long long)D,
                (long long)g);
  *geff = static_cast<int32_t>(g);
  return W4_OK;
}

w4_status w4_embedding_gather(const int32_t* ids, int64_t T, const void* table, const float* scale,
                              const float* zero, int64_t V, int64_t D, int32_t group, void* out, void* stream) {
  int32_t g = 0;
  w4_status st = check_table(V, D, group, &g);
  if (st != W4_OK) return st;
  if (T < 0) return fail(W4_ERR_SHAPE, "T must be >= 0");
  if (T == 0) return ok();
  if (!ids || !table || !scale || !zero || !out) return fail(W4_ERR_NULL, "ids, table, scale, zero, out must be non-NULL");
  if (!aligned(ids, 4) || !aligned(table, 4) || !aligned(scale, 4) || !aligned(zero, 4) || !aligned(out, 16))
    return fail(W4_ERR_ALIGN, "out must be 16-byte aligned; ids, table, scale, zero 4-byte aligned");
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  return from_cuda(w4::launch_embedding_gather(ids, T, table, scale, zero, V, D, g, out, status,
                                               static_cast<cudaStream_t>(stream)),
                   "embedding gather launch");
}

w4_status w4_lm_head_gemv(const void* h, int64_t M, const void* table, const float* scale, const float* zero,
                          int64_t V, int64_t D, int32_t group, void* y, void* stream) {
  int32_t g = 0;
  w4_status st = check_table(V, D, group, &g);
  if (st != W4_OK) return st;
  if (M < 0) return fail(W4_ERR_SHAPE, "M must be >= 0");
  if (D % 32 != 0) return fail(W4_ERR_UNSUPPORTED, "the head reads rows 32 codes at a time: D=%lld", (long long)D);
  // 8 rows of h in shared memory: as fp16 in MMA order (D and the group multiples of 128), else as fp32 padded to
  // 36 floats per 32 plus D/8 word sums each
  const bool tc = D % 128 == 0 && g % 128 == 0;
  if (tc ? D > 8192 : D * 40 > 227 * 1024)
    return fail(W4_ERR_UNSUPPORTED, "the head keeps 8 rows of h in shared memory: D=%lld is too long", (long long)D);
  if (M == 0) return ok();
  if (!h || !table || !scale || !zero || !y) return fail(W4_ERR_NULL, "h, table, scale, zero, y must be non-NULL");
  if (!aligned(h, 2) || !aligned(table, 16) || !aligned(scale, 4) || !aligned(zero, 4) || !aligned(y, 2))
    return fail(W4_ERR_ALIGN, "table must be 16-byte aligned; scale, zero 4-byte; h, y 2-byte");
  return from_cuda(w4::launch_lm_head(h, M, table, scale, zero, V, D, g, y, static_cast<cudaStream_t>(stream)),
                   "lm_head launch");
}

w4_status w4_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e, "cudaStreamSynchronize");
  unsigned int* p = nullptr;
  e = status_ptr(&p);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  unsigned int v = 0;
  e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e, "read device status");
  if (v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return from_cuda(e, "clear device status");
    return fail(static_cast<w4_status>(v), "a kernel recorded %s", w4_status_string(static_cast<int32_t>(v)));
  }
  return ok();
}

w4_status w4_selftest_bounded_wait(int64_t spin_limit, void* stream) {
  if (spin_limit <= 0) return fail(W4_ERR_SHAPE, "spin_limit must be positive");
  unsigned int* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return from_cuda(e, "device status word");
  return from_cuda(w4::launch_bounded_wait_selftest(spin_limit, status, static_cast<cudaStream_t>(stream)),
                   "selftest launch");
}

}  // extern "C"
