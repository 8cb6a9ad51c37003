// Weight-side tools: the asymmetric min/max group quantizer and the signed
// int4 -> uint4b8 repack.
//
// vllm-omni quantization/cpu_int4.py, quantize_groupwise: per group of
// `group` consecutive input columns of w [N, K], scale = max(max - min, 1e-9)
// / 15 and zero = min + 8 scale in fp32, codes q = clamp(round((w - min) /
// scale), 0, 15) (round half to even), packed two per byte low nibble first
// (pack_nibbles). The fp32 steps are taken with IEEE rounding (__fsub_rn,
// __fdiv_rn, rintf; the code of an element comes from a reciprocal product
// wherever that provably rounds like the IEEE quotient, see quant_code), so
// codes, scales and zeros are bit-exact.
//
// vLLM API docs, quantization.w4afp8, _repack_signed_int4_to_uint4b8:
// signed int4 nibbles become uint4b8 (q + 8 mod 16) by XOR 0x88 on every byte.
//
// Both are bandwidth-bound load-time passes. Groups are contiguous in memory
// (row n's group j starts at element n K + j group), so for groups of 8 to
// 256 elements the quantizer walks the weight as one flat array of 8-element
// chunks (16-byte loads, kept in registers; two chunks per thread for groups
// of 16 or more, so a group's scale and reciprocal serve 16 elements). The
// group's neighbouring lanes reduce its min and max with shuffles and every
// thread stores its codes as 32-bit words. Other groups take one warp per
// (row, group), reading the group twice (the second time from L1). The
// repack moves 16-byte vectors.
#include "common.cuh"
#include "launch.h"

namespace w4 {
namespace {

template <bool kF16>
W4_DEV float2 load_pair(const uint16_t* w, size_t i) {
  const uint32_t v = *reinterpret_cast<const uint32_t*>(w + i);
  if (kF16) return make_float2(half_bits_to_f32(v & 0xFFFFu), half_bits_to_f32(v >> 16));
  return make_float2(bf16_lo(v), bf16_hi(v));
}

template <bool kF16>
__global__ void __launch_bounds__(256) quantize_groupwise_kernel(const uint16_t* w, int64_t N, int64_t K, int group,
                                                                 uint8_t* packed, float* scale, float* zero) {
  const int64_t G = K / group;
  const int64_t id = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (id >= N * G) return;
  const int lane = threadIdx.x & 31;
  const int64_t n = id / G, g = id % G;
  const size_t base = static_cast<size_t>(n) * K + static_cast<size_t>(g) * group;   // even: group, K even
  const int pairs = group / 2;
  float mn = INFINITY, mx = -INFINITY;
  for (int p = lane; p < pairs; p += 32) {
    const float2 v = load_pair<kF16>(w, base + 2 * p);
    mn = fminf(mn, fminf(v.x, v.y));
    mx = fmaxf(mx, fmaxf(v.x, v.y));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float s = __fdiv_rn(fmaxf(__fsub_rn(mx, mn), 1e-9f), 15.0f);
  const float z = __fadd_rn(mn, __fmul_rn(8.0f, s));
  for (int p = lane; p < pairs; p += 32) {
    const float2 v = load_pair<kF16>(w, base + 2 * p);
    const float q0 = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v.x, mn), s)), 0.f), 15.f);
    const float q1 = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v.y, mn), s)), 0.f), 15.f);
    packed[base / 2 + p] = static_cast<uint8_t>(static_cast<int>(q0) | (static_cast<int>(q1) << 4));
  }
  if (lane == 0) {
    scale[id] = s;
    zero[id] = z;
  }
}

// rint(fl(d / s)) for 0 <= d <= fl(max - min) and s = fl(max(fl(max - min),
// 1e-9) / 15), without an IEEE divide on the common path. With r = fl(1/s)
// and y = fl(d r), y = Q (1 + e1)(1 + e2) for Q = d / s and |e1|, |e2| <=
// 2^-24, while fl(Q) = Q (1 + e3); Q < 15.001, so |y - fl(Q)| < 3.0001 * 2^-24
// * 15.001 < 2^-18. When y is more than 2^-17 away from every half-integer
// (|y - rint(y)| < 1/2 - 2^-17), fl(Q) lies strictly on the same side of each
// as y and rounds to the same integer; otherwise the IEEE quotient decides.
// The code is in [0, 15] either way (0 <= Q < 15.5), so no clamp is needed.
W4_DEV uint32_t quant_code(float d, float s, float r) {
  const float y = __fmul_rn(d, r);
  const float qf = rintf(y);
  if (fabsf(y - qf) < 0.49999237060546875f) return static_cast<uint32_t>(qf);
  return static_cast<uint32_t>(__float2int_rn(__fdiv_rn(d, s)));
}

// kC chunks of 8 elements per group (1..32, a power of two), kCPT of them
// per thread (consecutive); thread i takes chunks kCPT i .. kCPT i + kCPT - 1,
// all in group kCPT i / kC.
template <bool kF16, int kC, int kCPT>
__global__ void __launch_bounds__(256) quantize_chunks_kernel(const uint4* __restrict__ w, int64_t threads,
                                                              uint32_t* __restrict__ packed, float* __restrict__ scale,
                                                              float* __restrict__ zero) {
  constexpr int kLanes = kC / kCPT;   // lanes per group
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool live = i < threads;   // dead lanes still join the shuffles
  float v[kCPT][8];
#pragma unroll
  for (int c = 0; c < kCPT; ++c) {
    if (live) {
      const uint4 q = ld_stream_v4(w + i * kCPT + c);
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[c][2 * j] = kF16 ? half_bits_to_f32(u[j] & 0xFFFFu) : bf16_lo(u[j]);
        v[c][2 * j + 1] = kF16 ? half_bits_to_f32(u[j] >> 16) : bf16_hi(u[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[c][j] = 0.f;
    }
  }
  float mn = v[0][0], mx = v[0][0];
#pragma unroll
  for (int c = 0; c < kCPT; ++c)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      mn = fminf(mn, v[c][j]);
      mx = fmaxf(mx, v[c][j]);
    }
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (!live) return;
  const float s = __fdiv_rn(fmaxf(__fsub_rn(mx, mn), 1e-9f), 15.0f);
  const float r = __frcp_rn(s);
#pragma unroll
  for (int c = 0; c < kCPT; ++c) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) word |= quant_code(__fsub_rn(v[c][j], mn), s, r) << (4 * j);
    packed[i * kCPT + c] = word;
  }
  if ((i & (kLanes - 1)) == 0) {
    scale[i / kLanes] = s;
    zero[i / kLanes] = __fadd_rn(mn, __fmul_rn(8.0f, s));
  }
}

__global__ void __launch_bounds__(256) xor88_kernel(const uint4* src, uint4* dst, size_t n16, const uint8_t* src_tail,
                                                    uint8_t* dst_tail, int tail) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    uint4 v = ld_nc_v4(src + i);
    v.x ^= 0x88888888u;
    v.y ^= 0x88888888u;
    v.z ^= 0x88888888u;
    v.w ^= 0x88888888u;
    dst[i] = v;
  }
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x] ^ 0x88u;
}

int sm_count_tools() { return current_sm_count(); }

}  // namespace

template <bool kF16, int kC, int kCPT>
void launch_cpt(const uint4* wp, int64_t chunks, uint32_t* pp, float* scale, float* zero, cudaStream_t s) {
  const int64_t threads = chunks / kCPT;
  const unsigned int blocks = static_cast<unsigned int>((threads + 255) / 256);
  quantize_chunks_kernel<kF16, kC, kCPT><<<blocks, 256, 0, s>>>(wp, threads, pp, scale, zero);
}

template <bool kF16>
cudaError_t launch_chunks(const void* w, int64_t chunks, int32_t group, uint8_t* packed, float* scale, float* zero,
                          cudaStream_t s) {
  auto wp = static_cast<const uint4*>(w);
  auto pp = reinterpret_cast<uint32_t*>(packed);
  switch (group / 8) {   // groups of 16 or more: two chunks per thread
    case 1: launch_cpt<kF16, 1, 1>(wp, chunks, pp, scale, zero, s); break;
    case 2: launch_cpt<kF16, 2, 2>(wp, chunks, pp, scale, zero, s); break;
    case 4: launch_cpt<kF16, 4, 2>(wp, chunks, pp, scale, zero, s); break;
    case 8: launch_cpt<kF16, 8, 2>(wp, chunks, pp, scale, zero, s); break;
    case 16: launch_cpt<kF16, 16, 2>(wp, chunks, pp, scale, zero, s); break;
    default: launch_cpt<kF16, 32, 2>(wp, chunks, pp, scale, zero, s); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_groupwise(const void* w, bool f16, int64_t N, int64_t K, int32_t group, uint8_t* packed,
                                      float* scale, float* zero, cudaStream_t s) {
  const bool chunked = K % 8 == 0 && (group == 8 || group == 16 || group == 32 || group == 64 || group == 128 ||
                                      group == 256) &&
                       reinterpret_cast<uintptr_t>(w) % 16 == 0 && reinterpret_cast<uintptr_t>(packed) % 4 == 0;
  if (chunked) {
    const int64_t chunks = N * K / 8;
    return f16 ? launch_chunks<true>(w, chunks, group, packed, scale, zero, s)
               : launch_chunks<false>(w, chunks, group, packed, scale, zero, s);
  }
  const int64_t warps = N * (K / group);
  const unsigned int blocks = static_cast<unsigned int>((warps + 7) / 8);
  if (f16)
    quantize_groupwise_kernel<true><<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(w), N, K, group, packed, scale,
                                                           zero);
  else
    quantize_groupwise_kernel<false><<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(w), N, K, group, packed,
                                                            scale, zero);
  return cudaGetLastError();
}

cudaError_t launch_xor88(const void* src, void* dst, int64_t n_bytes, cudaStream_t s) {
  const size_t n16 = static_cast<size_t>(n_bytes) / 16;
  const int tail = static_cast<int>(n_bytes - static_cast<int64_t>(n16) * 16);
  size_t want = (n16 + 255) / 256;
  const size_t cap = static_cast<size_t>(sm_count_tools()) * 8;
  const unsigned int blocks = static_cast<unsigned int>(want < 1 ? 1 : (want > cap ? cap : want));
  xor88_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16,
                                      static_cast<const uint8_t*>(src) + n16 * 16,
                                      static_cast<uint8_t*>(dst) + n16 * 16, tail);
  return cudaGetLastError();
}

}  // namespace w4
