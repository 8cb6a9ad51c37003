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
// Many rows of up to 3072 elements take one warp each, other rows one CTA each.
// Every thread keeps its 8-element chunks of the row in registers (16-byte
// loads); the row maximum is a halfwise bf16x2 (fp16x2) magnitude maximum per
// thread and a warp-shuffle butterfly (plus one shared-memory step across the
// warps of a CTA); the quantized chunks leave as 8-byte stores, so HBM sees the
// row read once and the codes written once (3 bytes per element). Every
// element costs a handful of instructions: packed fp32 pairs, a magic-number
// rounding for int8, an e4m3x2 conversion per pair for e4m3. A warp per row
// keeps many rows in flight per SM and pays no block barrier; with a CTA per
// row and a few elements per thread, the barrier, the cross-warp maximum and
// the row's index arithmetic cost more than the elements themselves.
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
  // every group of 8 lanes holds the (up to 8) warp maxima, zero past the last
  // warp; a butterfly within the group leaves the row maximum in every lane
  float m = (lane & 7) < static_cast<int>((blockDim.x + 31) >> 5) ? red[lane & 7] : 0.f;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// Halfwise magnitude maximum of a chunk (two bf16 or fp16 magnitudes per word).
template <bool kF16>
W4_DEV uint32_t chunk_absmax2(uint32_t m, const uint4& v) {
  return absmax2<kF16>(absmax2<kF16>(m, v.x), absmax2<kF16>(absmax2<kF16>(v.y, v.z), v.w));
}

// The row maximum |x| of a halfwise maximum word, as fp32 (exact).
template <bool kF16>
W4_DEV float absmax_of(uint32_t m) {
  return fmaxf(fabsf(act_lo<kF16>(m)), fabsf(act_hi<kF16>(m)));
}

template <bool FP8, bool kF16>
W4_DEV uint2 quant_chunk(const uint4& v, const QuotientBracket& b) {
  return FP8 ? quant_e4m3_chunk<kF16>(v, b) : quant_int8_chunk<kF16>(v, b);
}

// The codes of one 8-chunk as stored: 8 bytes, or (kWiden) the exact fp16
// values of the codes in the W4A8 operand order (16 bytes).
template <bool FP8, bool kWiden, bool kF16>
W4_DEV void store_chunk(void* q, size_t i, const uint4& v, const QuotientBracket& b) {
  const uint2 c = quant_chunk<FP8, kF16>(v, b);
  if (kWiden)
    static_cast<uint4*>(q)[i] = FP8 ? widen_e4m3(c.x, c.y) : widen_i8(c.x, c.y);
  else
    static_cast<uint2*>(q)[i] = c;
}

// One CTA per row (rows longer than 3072 elements, or few rows).
// NCH > 0: the row fits in registers, NCH chunks per thread (chunks past the
// row are masked, so NCH may round the count up).
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
    uint32_t m2 = 0;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int i = threadIdx.x + c * blockDim.x;
      v[c] = (i < K8) ? ld_stream_v4(xr + i) : make_uint4(0, 0, 0, 0);
      m2 = chunk_absmax2<kF16>(m2, v[c]);
    }
    const float amax = row_max(absmax_of<kF16>(m2), red);
    const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, kQ);
    const QuotientBracket b = quotient_bracket(s);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int i = threadIdx.x + c * blockDim.x;
      if (i < K8) store_chunk<FP8, kWiden, kF16>(q, q0 + i, v[c], b);
    }
    if (threadIdx.x == 0) scale[row] = s;
  } else {
    uint32_t m2 = 0;
    for (int i = threadIdx.x; i < K8; i += blockDim.x) m2 = chunk_absmax2<kF16>(m2, ld_nc_v4(xr + i));
    const float amax = row_max(absmax_of<kF16>(m2), red);
    const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, kQ);
    const QuotientBracket b = quotient_bracket(s);
    for (int i = threadIdx.x; i < K8; i += blockDim.x)
      store_chunk<FP8, kWiden, kF16>(q, q0 + i, ld_stream_v4(xr + i), b);
    if (threadIdx.x == 0) scale[row] = s;
  }
}

// One warp per row for rows of up to 32 * NCH chunks (K <= 3072): lane l
// holds chunks l, l + 32, ...; the row maximum is a shuffle butterfly, with no
// block barrier, and four rows share a CTA. Each warp has the whole row in
// flight at once.
constexpr int kRowsPerCta = 4;

template <int NCH, bool FP8, bool kWiden, bool kF16>
__global__ void __launch_bounds__(32 * kRowsPerCta) quant_warp_rows(const uint4* __restrict__ x, int64_t M, int K8,
                                                                     void* __restrict__ q, float* __restrict__ scale,
                                                                     const int32_t* __restrict__ gather, int64_t T,
                                                                     unsigned int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
  if (row >= M) return;                       // the whole warp
  const size_t q0 = static_cast<size_t>(row) * static_cast<size_t>(K8);
  int64_t src = row;
  if (gather != nullptr) {
    src = gather[row];
    if (src < 0 || src >= T) {
      for (int i = lane; i < K8; i += 32) {
        if (kWiden)
          static_cast<uint4*>(q)[q0 + i] = make_uint4(0, 0, 0, 0);
        else
          static_cast<uint2*>(q)[q0 + i] = make_uint2(0, 0);
      }
      if (lane == 0) {
        scale[row] = 1.f;
        report(status, W4_ERR_SHAPE);
      }
      return;
    }
  }
  const uint4* xr = x + static_cast<size_t>(src) * static_cast<size_t>(K8);
  uint4 v[NCH];
  uint32_t m2 = 0;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = lane + 32 * j;
    v[j] = c < K8 ? ld_stream_v4(xr + c) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < NCH; ++j) m2 = chunk_absmax2<kF16>(m2, v[j]);
  float amax = absmax_of<kF16>(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  constexpr float kQ = FP8 ? 448.f : 127.f;
  const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, kQ);
  const QuotientBracket b = quotient_bracket(s);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = lane + 32 * j;
    if (c < K8) store_chunk<FP8, kWiden, kF16>(q, q0 + c, v[j], b);
  }
  if (lane == 0) scale[row] = s;
}

// Chunks per lane of the warp form for M rows of K8 chunks, or 0 for the
// CTA form. Measured on GB300 over M x K from 256 x 1024 to 65536 x 4096: the
// warp form wins once the rows are short and many (1.4x to 2.4x at 32768 x
// 2048 and 65536 x 1024, even at 4096 x 2048); a CTA per row wins at K = 4096,
// where a warp's row of 16 chunks a lane leaves too few warps per SM to cover
// its own arithmetic, and for few rows, where 8 warps on one row finish it
// sooner than 1.
inline int warp_chunks(int64_t M, int K8) {
  if (K8 > 384 || M * K8 < (int64_t{1} << 19)) return 0;
  const int need = (K8 + 31) / 32;
  for (int n : {1, 2, 3, 4, 6, 8, 12})
    if (need <= n) return n;
  return 0;
}

template <bool FP8, bool kWiden, bool kF16 = false>
cudaError_t launch(const void* x, int64_t M, int64_t K, void* q, float* scale, cudaStream_t s,
                   const int32_t* gather = nullptr, int64_t T = 0, unsigned int* status = nullptr) {
  const int K8 = static_cast<int>(K / 8);
  if (M == 0 || K8 == 0) return cudaSuccess;
  auto xp = static_cast<const uint4*>(x);
  const int wn = warp_chunks(M, K8);
  if (wn > 0) {
    const dim3 grid(static_cast<unsigned>((M + kRowsPerCta - 1) / kRowsPerCta));
    constexpr int kT = 32 * kRowsPerCta;
    switch (wn) {
#define W4_WARP_CASE(n) \
  case n: quant_warp_rows<n, FP8, kWiden, kF16><<<grid, kT, 0, s>>>(xp, M, K8, q, scale, gather, T, status); break;
      W4_WARP_CASE(1) W4_WARP_CASE(2) W4_WARP_CASE(3) W4_WARP_CASE(4)
      W4_WARP_CASE(6) W4_WARP_CASE(8) W4_WARP_CASE(12)
#undef W4_WARP_CASE
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  // one CTA per row, the row's chunks in registers up to K = 8192, read twice
  // beyond. With at least 8 rows per SM a row gets at most 128 threads (up to
  // 8 chunks each): twice the rows in flight per SM and a cheaper cross-warp
  // maximum, measured 11.2 -> 9.9 us at 4096 x 4096 and 39.4 -> 32.2 us at
  // 16384 x 4096 on GB300. Fewer rows keep up to 256 threads, so that each row
  // finishes sooner (128 threads measured 3.97 -> 4.92 us at 1024 x 4096).
  const int cap = M >= 8 * static_cast<int64_t>(current_sm_count()) ? 128 : kMaxThreads;
  int threads = ((K8 + 31) / 32) * 32;
  if (threads > cap) threads = cap;
  int nch = (K8 + threads - 1) / threads;
  if (nch == 5 || nch == 7) ++nch;   // chunks past the row are masked
  const dim3 grid(static_cast<unsigned>(M));
  switch (nch) {
    case 1: quant_rows<1, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 2: quant_rows<2, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 3: quant_rows<3, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 4: quant_rows<4, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 6: quant_rows<6, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    case 8: quant_rows<8, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
    default: quant_rows<0, FP8, kWiden, kF16><<<grid, threads, 0, s>>>(xp, K8, q, scale, gather, T, status); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_per_token(const void* x, bool x_f16, int64_t M, int64_t K, bool fp8, void* q, float* scale,
                                   unsigned int* status, cudaStream_t s) {
  if (K / 8 > INT32_MAX) return cudaErrorInvalidValue;
  if (x_f16)
    return fp8 ? launch<true, false, true>(x, M, K, q, scale, s, nullptr, 0, status)
               : launch<false, false, true>(x, M, K, q, scale, s, nullptr, 0, status);
  return fp8 ? launch<true, false>(x, M, K, q, scale, s, nullptr, 0, status)
             : launch<false, false>(x, M, K, q, scale, s, nullptr, 0, status);
}

cudaError_t launch_quant_widen(const void* x, int64_t M, int64_t K, bool fp8, void* wide, float* scale,
                               unsigned int* status, cudaStream_t s) {
  if (K / 8 > INT32_MAX) return cudaErrorInvalidValue;
  return fp8 ? launch<true, true>(x, M, K, wide, scale, s, nullptr, 0, status)
             : launch<false, true>(x, M, K, wide, scale, s, nullptr, 0, status);
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
