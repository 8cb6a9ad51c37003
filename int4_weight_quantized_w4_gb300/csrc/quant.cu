// Dynamic per-token symmetric activation quantization (int8 or e4m3).
//
// vLLM API docs, inc.schemes.inc_w4a8_linear, INCXPUW4A8LinearMethod.apply_weights:
// activations are quantized per token, symmetric, to 8 bits right before the
// W4A8 GEMM. vLLM API docs, quantization.w4afp8, W4AFP8Config.__init__: the
// expert activations are 8-bit float, symmetric, per token, dynamic.
//
// The activations may be bf16 or fp16 (the INC class docstring allows both).
// Per row: amax = max |x|; s = amax / Q (IEEE fp32 divide; s = 1 if amax = 0);
// int8: q = clamp(rne(x / s), -127, 127); e4m3: q = satfinite-rne(x / s).
//
// One CTA per row. Each thread keeps its 8-element chunks of the row in
// registers (16-byte loads), the row maximum is a warp-shuffle butterfly plus
// one shared-memory step, and the quantized chunks leave as 8-byte stores, so
// HBM sees the row read once and the codes written once (3 bytes per element).
// The fused form for the W4A8 GEMM stores each chunk's codes instead as their
// exact fp16 values in the GEMM's operand order (4 bytes per element, no int8
// round trip). The gathered form quantizes row gather[r] of x into row r (the
// expert-sorted rows of a routed MoE layer): the codes are those of
// quantizing x and then gathering, without the intermediate copy.
#include "common.cuh"
#include "launch.h"

namespace w4 {
namespace {

constexpr int kMaxThreads = 256;

W4_DEV float row_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = (blockDim.x + 31) >> 5;
  float m = 0.f;
  for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
  return m;
}

// The two 16-bit activations of a word as fp32 (exact): bf16, or fp16 (kF16).
template <bool kF16>
W4_DEV float act_lo(uint32_t w) {
  return kF16 ? half_bits_to_f32(w & 0xFFFFu) : bf16_lo(w);
}
template <bool kF16>
W4_DEV float act_hi(uint32_t w) {
  return kF16 ? half_bits_to_f32(w >> 16) : bf16_hi(w);
}

template <bool kF16>
W4_DEV float chunk_absmax(const uint4& v) {
  float m = fmaxf(fabsf(act_lo<kF16>(v.x)), fabsf(act_hi<kF16>(v.x)));
  m = fmaxf(m, fmaxf(fabsf(act_lo<kF16>(v.y)), fabsf(act_hi<kF16>(v.y))));
  m = fmaxf(m, fmaxf(fabsf(act_lo<kF16>(v.z)), fabsf(act_hi<kF16>(v.z))));
  m = fmaxf(m, fmaxf(fabsf(act_lo<kF16>(v.w)), fabsf(act_hi<kF16>(v.w))));
  return m;
}

// The codes are those of the IEEE quotient fl(x / s), taken from y = x * r
// with r = fl(1 / s), the correctly rounded reciprocal. y and x / s differ by
// at most |x / s| (2^-23 + 2^-48) and fl(x / s) is within |x / s| 2^-24 of
// x / s, so for |x / s| <= 127.0001 (int8: |x| <= amax, s = fl(amax / 127))
// |y - fl(x / s)| <= 2.3e-5 < 2^-15. Where y is more than 2^-15 from every
// half-integer, y and fl(x / s) round to the same integer; nearer than that
// the quotient is formed with the IEEE divide itself (a few elements per row
// at most).
W4_DEV uint32_t q_int8(float x, float s, float r) {
  const float y = x * r;
  float q = rintf(y);
  if (fabsf(0.5f - fabsf(y - q)) < 3.0517578125e-5f) q = rintf(__fdiv_rn(x, s));
  q = fmaxf(-127.f, fminf(127.f, q));
  return static_cast<uint32_t>(static_cast<int>(q)) & 0xFFu;
}

// Two int8 codes from one word of two activations, low element in the low byte.
template <bool kF16>
W4_DEV uint32_t q_int8_pair(uint32_t w, float s, float r) {
  return q_int8(act_lo<kF16>(w), s, r) | (q_int8(act_hi<kF16>(w), s, r) << 8);
}

// Two e4m3 codes from one word of two activations, low element in the low
// byte: the codes of fl(x / s) (e4m3x2_of_quotient).
template <bool kF16>
W4_DEV uint32_t q_e4m3_pair(uint32_t w, float s, float r) {
  return e4m3x2_of_quotient(act_lo<kF16>(w), act_hi<kF16>(w), s, r);
}

template <bool FP8, bool kF16>
W4_DEV uint2 quant_chunk(const uint4& v, float s, float r) {
  uint2 o;
  if (FP8) {
    o.x = q_e4m3_pair<kF16>(v.x, s, r) | (q_e4m3_pair<kF16>(v.y, s, r) << 16);
    o.y = q_e4m3_pair<kF16>(v.z, s, r) | (q_e4m3_pair<kF16>(v.w, s, r) << 16);
  } else {
    o.x = q_int8_pair<kF16>(v.x, s, r) | (q_int8_pair<kF16>(v.y, s, r) << 16);
    o.y = q_int8_pair<kF16>(v.z, s, r) | (q_int8_pair<kF16>(v.w, s, r) << 16);
  }
  return o;
}

// The codes of one 8-chunk as stored: 8 bytes, or (kWiden) the exact fp16
// values of the codes in the W4A8 operand order (16 bytes).
template <bool FP8, bool kWiden, bool kF16>
W4_DEV void store_chunk(void* q, size_t i, const uint4& v, float s, float r) {
  const uint2 c = quant_chunk<FP8, kF16>(v, s, r);
  if (kWiden)
    static_cast<uint4*>(q)[i] = FP8 ? widen_e4m3(c.x, c.y) : widen_i8(c.x, c.y);
  else
    static_cast<uint2*>(q)[i] = c;
}

// NCH > 0: the row fits in registers, NCH chunks per thread.
// NCH == 0: long rows, read twice (the second read mostly hits L2).
// gather (may be null): source row of each output row, checked against T; an
// id outside [0, T) gives a zero row with scale 1 and W4_ERR_SHAPE in status.
template <int NCH, bool FP8, bool kWiden, bool kF16>
__global__ void __launch_bounds__(kMaxThreads) quant_rows(const uint4* __restrict__ x, int K8,
                                                          void* __restrict__ q, float* __restrict__ scale,
                                                          const int32_t* __restrict__ gather, int64_t T,
                                                          unsigned int* status) {
  __shared__ float red[kMaxThreads / 32];
  const size_t row = blockIdx.x;
  const size_t q0 = row * static_cast<size_t>(K8);
  size_t src = row;
  if (gather != nullptr) {
    const int64_t g = gather[row];
    if (g < 0 || g >= T) {     // the same for the whole block: no barrier is skipped by part of it
      for (int i = threadIdx.x; i < K8; i += blockDim.x) {
        if (kWiden)
          static_cast<uint4*>(q)[q0 + i] = make_uint4(0, 0, 0, 0);
        else
          static_cast<uint2*>(q)[q0 + i] = make_uint2(0, 0);
      }
      if (threadIdx.x == 0) {
        scale[row] = 1.f;
        report(status, W4_ERR_SHAPE);
      }
      return;
    }
    src = static_cast<size_t>(g);
  }
  const uint4* xr = x + src * static_cast<size_t>(K8);
  constexpr float kQ = FP8 ? 448.f : 127.f;
  if constexpr (NCH > 0) {
    uint4 v[NCH];
    float m = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int i = threadIdx.x + c * blockDim.x;
      v[c] = (i < K8) ? ld_stream_v4(xr + i) : make_uint4(0, 0, 0, 0);
      m = fmaxf(m, chunk_absmax<kF16>(v[c]));
    }
    const float amax = row_max(m, red);
    const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, kQ);
    const float r = __frcp_rn(s);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int i = threadIdx.x + c * blockDim.x;
      if (i < K8) store_chunk<FP8, kWiden, kF16>(q, q0 + i, v[c], s, r);
    }
    if (threadIdx.x == 0) scale[row] = s;
  } else {
    float m = 0.f;
    for (int i = threadIdx.x; i < K8; i += blockDim.x) m = fmaxf(m, chunk_absmax<kF16>(ld_nc_v4(xr + i)));
    const float amax = row_max(m, red);
    const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, kQ);
    const float r = __frcp_rn(s);
    for (int i = threadIdx.x; i < K8; i += blockDim.x)
      store_chunk<FP8, kWiden, kF16>(q, q0 + i, ld_stream_v4(xr + i), s, r);
    if (threadIdx.x == 0) scale[row] = s;
  }
}

template <bool FP8, bool kWiden, bool kF16 = false>
cudaError_t launch(const void* x, int64_t M, int64_t K, void* q, float* scale, cudaStream_t s,
                   const int32_t* gather = nullptr, int64_t T = 0, unsigned int* status = nullptr) {
  const int K8 = static_cast<int>(K / 8);
  int threads = ((K8 + 31) / 32) * 32;
  if (threads > kMaxThreads) threads = kMaxThreads;
  const int nch = (K8 + threads - 1) / threads;
  const dim3 grid(static_cast<unsigned>(M));
  auto xp = static_cast<const uint4*>(x);
  switch (nch) {
    case 1: quant_rows<1, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 2: quant_rows<2, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 3: quant_rows<3, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 4: quant_rows<4, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    default: quant_rows<0, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_per_token(const void* x, bool x_f16, int64_t M, int64_t K, bool fp8, void* q, float* scale,
                                   cudaStream_t s) {
  if (K / 8 > INT32_MAX) return cudaErrorInvalidValue;
  if (x_f16)
    return fp8 ? launch<true, false, true>(x, M, K, q, scale, s) : launch<false, false, true>(x, M, K, q, scale, s);
  return fp8 ? launch<true, false>(x, M, K, q, scale, s) : launch<false, false>(x, M, K, q, scale, s);
}

cudaError_t launch_quant_widen(const void* x, int64_t M, int64_t K, bool fp8, void* wide, float* scale,
                               cudaStream_t s) {
  if (K / 8 > INT32_MAX) return cudaErrorInvalidValue;
  return fp8 ? launch<true, true>(x, M, K, wide, scale, s) : launch<false, true>(x, M, K, wide, scale, s);
}

cudaError_t launch_quant_gather(const void* x, int64_t T, int64_t K, const int32_t* rows, int64_t R, bool fp8,
                                bool widen, void* q, float* scale, unsigned int* status, cudaStream_t s) {
  if (K / 8 > INT32_MAX) return cudaErrorInvalidValue;
  if (fp8)
    return widen ? launch<true, true>(x, R, K, q, scale, s, rows, T, status)
                 : launch<true, false>(x, R, K, q, scale, s, rows, T, status);
  return widen ? launch<false, true>(x, R, K, q, scale, s, rows, T, status)
               : launch<false, false>(x, R, K, q, scale, s, rows, T, status);
}

}  // namespace w4
