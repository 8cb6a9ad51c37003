// Internal host-side launch functions, one per kernel family. The public
// entry points in api.cu validate arguments and then call these; each returns
// the cudaError_t of its launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "w4.h"

namespace w4 {

// SMs of the current device, asked on every call: the runtime answers from its
// own cache, the status is checked before the value is used, and the answer
// is right for whichever device the caller has made current.
inline int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0)
    n = 152;
  return n;
}

// Polls a bounded wait makes before it gives up (about a second of spinning).
constexpr long long kWaitLimit = 1LL << 24;

// status: the device status word (a timed-out wait records W4_ERR_TIMEOUT there).
cudaError_t launch_quant_per_token(const void* x, bool x_f16, int64_t M, int64_t K, bool fp8, void* q,
                                   float* scale, unsigned int* status, cudaStream_t s);

struct W4A16Args {
  const void* x;
  const void* qweight;
  const void* w_scale;
  bool scale_bf16;
  const void* zeros;
  const void* bias;
  void* y;
  int64_t M, N, K;
  int32_t group;  // effective group (K when the caller passed -1)
  unsigned int* status;
  // host entry point, page-locked host buffers (device addresses): x is copied
  // from x_host into x by the L2-prefetch grid, y written to y_host as well
  const void* x_host = nullptr;
  void* y_host = nullptr;
};
cudaError_t launch_w4a16(const W4A16Args& a, cudaStream_t s);
// Per-token quantization whose output is the codes' exact fp16 values in the
// W4A8 operand order (fp16 [M, K] into `wide`), plus the fp32 scales.
cudaError_t launch_quant_widen(const void* x, int64_t M, int64_t K, bool fp8, void* wide, float* scale,
                               unsigned int* status, cudaStream_t s);
// Shared memory the decode kernel needs for one token row beside a minimal ring.
size_t w4a16_smem_bytes(int64_t N, int64_t K, int32_t group);

struct W4A8Args {
  const void* act;        // int8 [M,K] (dense) or e4m3 [R,K] (experts)
  const float* x_scale;   // [M] (ignored for partials)
  const void* qweight;    // GPTQ [K/8,N] (dense) or CT [E,N,K/8] (experts)
  const void* w_scale;    // fp16 [G,N] (dense) or [E,N,G] (experts)
  const void* bias;       // bf16 [N] or nullptr
  void* out;              // bf16 [M,N], or int32 [M,G,N] for partials
  const int32_t* expert_offsets;  // device [E+1] (experts only)
  int32_t E;
  int64_t M, N, K;
  int32_t group;          // effective group
  bool partials;          // write int32 group partials instead of y
  unsigned int* status;
  void* workspace;        // fp16 [rows, K]: the activations widened once per call
  bool prewidened;        // the workspace already holds them (act unused)
  bool fp8_act;           // experts: act holds e4m3 codes [R, K] that the fp8 tensor path reads directly
  size_t workspace_bytes; // dense y: a workspace this large may also hold split-K partial sums
};
size_t w4a8_workspace_bytes(int64_t rows, int64_t K);
// The dense W4A8 workspace with room for the split-K partial sums that
// M x N x K at this group would use (fp32 [splits][M][N] after the widened
// activations); equal to w4a8_workspace_bytes when the GEMM is not split.
size_t w4a8_workspace_bytes_split(int64_t M, int64_t N, int64_t K, int32_t group);
// Sets the calling thread's w4_last_error() message and returns `st`.
w4_status report_error(w4_status st, const char* msg);
cudaError_t launch_w4a8_dense(const W4A8Args& a, cudaStream_t s);
cudaError_t launch_w4afp8_experts(const W4A8Args& a, cudaStream_t s);
// Expert GEMMs whose (effective) group is a multiple of 32 run on the fp8
// tensor path (kind::f8f6f4, 32 k per MMA); others widen to fp16 first.
bool w4afp8_fp8_path(int32_t group);

cudaError_t launch_quantize_groupwise(const void* w, bool f16, int64_t N, int64_t K, int32_t group, uint8_t* packed,
                                      float* scale, float* zero, cudaStream_t s);
cudaError_t launch_xor88(const void* src, void* dst, int64_t n_bytes, cudaStream_t s);
cudaError_t launch_embedding_gather(const int32_t* ids, int64_t T, const void* table, const float* scale,
                                    const float* zero, int64_t V, int64_t D, int32_t group, void* out,
                                    unsigned int* status, cudaStream_t s);
cudaError_t launch_lm_head(const void* h, int64_t M, const void* table, const float* scale, const float* zero,
                           int64_t V, int64_t D, int32_t group, void* y, cudaStream_t s);
cudaError_t launch_quant_gather(const void* x, int64_t T, int64_t K, const int32_t* rows, int64_t R, bool fp8,
                                bool widen, void* q, float* scale, unsigned int* status, cudaStream_t s);
size_t moe_route_workspace_bytes(int64_t T, int32_t E);
cudaError_t launch_moe_route(const void* logits, bool bf16, int64_t T, int32_t E, int32_t k, bool renorm,
                             int32_t* ids, float* wts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                             void* workspace, cudaStream_t s);
cudaError_t launch_silu_mul_quant(const void* h, int64_t R, int64_t I, void* q, float* scale, void* act,
                                  cudaStream_t s);
cudaError_t launch_moe_combine(const void* y, int64_t R, int64_t H, const float* w, const int32_t* row_of, int64_t T,
                               int32_t k, void* out, unsigned int* status, cudaStream_t s);
cudaError_t launch_bounded_wait_selftest(long long limit, unsigned int* status, cudaStream_t s);

}  // namespace w4
