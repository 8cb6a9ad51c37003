// Weight-side tools: the asymmetric min/max group quantizer and the signed
// int4 -> uint4b8 repack.
//
// vllm-omni quantization/cpu_int4.py, quantize_groupwise: per group of
// `group` consecutive input columns of w [N, K], scale = max(max - min, 1e-9)
// / 15 and zero = min + 8 scale in fp32, codes q = clamp(round((w - min) /
// scale), 0, 15) (round half to even), packed two per byte low nibble first
// (pack_nibbles). The fp32 steps are taken with IEEE rounding (__fsub_rn,
// __fdiv_rn, rintf; the code of an element comes from reciprocal products
// wherever they provably round like the IEEE quotient, see code_chunk), so
// codes, scales and zeros are bit-exact.
//
// vLLM API docs, quantization.w4afp8, _repack_signed_int4_to_uint4b8:
// signed int4 nibbles become uint4b8 (q + 8 mod 16) by XOR 0x88 on every byte.
//
// Both are bandwidth-bound load-time passes. Groups are contiguous in memory
// (row n's group j starts at element n K + j group), so for groups of 8 to
// 256 elements the quantizer walks the weight as one flat array of 8-element
// chunks (16-byte loads, kept in registers; two chunks per thread for groups
// of 16, four for 32 or more). The
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

// Halfwise minimum / maximum of two words of two 16-bit floats (bf16, or
// fp16 with kF16).
template <bool kF16>
W4_DEV uint32_t min2h(uint32_t a, uint32_t b) {
  uint32_t d;
  if (kF16)
    asm("min.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <bool kF16>
W4_DEV uint32_t max2h(uint32_t a, uint32_t b) {
  uint32_t d;
  if (kF16)
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The codes rint(fl(d / s)) of the 8 elements of a 16-byte chunk, d =
// fl(w - min), packed as 8 nibbles (element j in bits 4j..4j+3). For
// 0 <= d <= fl(max - min) and s = fl(max(fl(max - min), 1e-9) / 15), Q = d / s
// lies in [0, 15.5), so every code is in [0, 15] without a clamp. With r =
// fl(1 / s), rlo = fl(r (1 - 2^-20)) and rhi = fl(r (1 + 2^-20)), fl(d rlo)
// and fl(d rhi) bracket fl(Q) (each product is Q (1 -+ 2^-20)(1 + e) with
// |e| < 3.1 * 2^-24; a subnormal d gives a Q far below 1/2 at both ends).
// Rounding is monotone, so equal integers at both ends are rint(fl(Q)); a
// pair of elements where some element's ends differ takes the IEEE divide for
// both (per pair: a warp runs a fallback whenever any lane needs one, and on
// GB300 this measured faster here than one test per chunk, 29.1 against
// 29.8 us at 14336 x 4096 g128).
// Adding 1.5 * 2^23 rounds a value in [0, 2^22) to an integer (half to even)
// and leaves it in the low bits of the sum; PRMTs gather the low bytes and a
// shift-or folds two codes into each byte.
template <bool kF16>
W4_DEV uint32_t code_chunk(const uint4& v, float nmn, float s, float rlo, float rhi) {
  constexpr float kMagic = 12582912.f;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t t[8], diff[4];
  float d[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float d0, d1, l0, l1, h0, h1;
    add2(d0, d1, act_lo<kF16>(w[i]), act_hi<kF16>(w[i]), nmn);   // fl(w - min)
    mul2(l0, l1, d0, d1, rlo);
    mul2(h0, h1, d0, d1, rhi);
    add2(l0, l1, l0, l1, kMagic);
    add2(h0, h1, h0, h1, kMagic);
    d[2 * i] = d0;
    d[2 * i + 1] = d1;
    t[2 * i] = __float_as_uint(l0);
    t[2 * i + 1] = __float_as_uint(l1);
    diff[i] = (t[2 * i] ^ __float_as_uint(h0)) | (t[2 * i + 1] ^ __float_as_uint(h1));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (diff[i] != 0) {
      t[2 * i] = __float_as_uint(rintf(__fdiv_rn(d[2 * i], s)) + kMagic);
      t[2 * i + 1] = __float_as_uint(rintf(__fdiv_rn(d[2 * i + 1], s)) + kMagic);
    }
  }
  uint32_t a = prmt(prmt(t[0], t[1], 0x0040u), prmt(t[2], t[3], 0x0040u), 0x5410u);   // bytes q0 q1 q2 q3
  uint32_t b = prmt(prmt(t[4], t[5], 0x0040u), prmt(t[6], t[7], 0x0040u), 0x5410u);
  a = (a | (a >> 4)) & 0x00FF00FFu;   // bytes (q0 | q1 << 4), 0, (q2 | q3 << 4), 0
  b = (b | (b >> 4)) & 0x00FF00FFu;
  return prmt(a, b, 0x6420u);
}

// kC chunks of 8 elements per group (1..32, a power of two), kCPT of them
// per thread (consecutive); thread i takes chunks kCPT i .. kCPT i + kCPT - 1,
// all in group kCPT i / kC. The chunks stay packed in registers: the group's
// minimum and maximum are halfwise bf16x2 (fp16x2) min / max, exact.
template <bool kF16, int kC, int kCPT>
__global__ void __launch_bounds__(256) quantize_chunks_kernel(const uint4* __restrict__ w, int64_t threads,
                                                              uint32_t* __restrict__ packed, float* __restrict__ scale,
                                                              float* __restrict__ zero) {
  constexpr int kLanes = kC / kCPT;   // lanes per group
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool live = i < threads;   // dead lanes still join the shuffles
  uint4 v[kCPT];
#pragma unroll
  for (int c = 0; c < kCPT; ++c) v[c] = live ? ld_nc_v4(w + i * kCPT + c) : make_uint4(0, 0, 0, 0);
  uint32_t mn2 = v[0].x, mx2 = v[0].x;
#pragma unroll
  for (int c = 0; c < kCPT; ++c) {
    mn2 = min2h<kF16>(mn2, min2h<kF16>(min2h<kF16>(v[c].x, v[c].y), min2h<kF16>(v[c].z, v[c].w)));
    mx2 = max2h<kF16>(mx2, max2h<kF16>(max2h<kF16>(v[c].x, v[c].y), max2h<kF16>(v[c].z, v[c].w)));
  }
  float mn = fminf(act_lo<kF16>(mn2), act_hi<kF16>(mn2));
  float mx = fmaxf(act_lo<kF16>(mx2), act_hi<kF16>(mx2));
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (!live) return;
  const float s = __fdiv_rn(fmaxf(__fsub_rn(mx, mn), 1e-9f), 15.0f);
  const float r = __frcp_rn(s);
  const float rlo = r * 0.99999904632568359375f, rhi = r * 1.00000095367431640625f;
#pragma unroll
  for (int c = 0; c < kCPT; ++c) packed[i * kCPT + c] = code_chunk<kF16>(v[c], -mn, s, rlo, rhi);
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
  // up to four consecutive chunks (64 bytes) per thread: more bytes in flight,
  // and the L1-allocating loads serve the sectors a thread's neighbouring
  // chunks share (measured on GB300 at 14336 x 4096 g128: 4.21 -> 4.60 TB/s)
  switch (group / 8) {
    case 1: launch_cpt<kF16, 1, 1>(wp, chunks, pp, scale, zero, s); break;
    case 2: launch_cpt<kF16, 2, 2>(wp, chunks, pp, scale, zero, s); break;
    case 4: launch_cpt<kF16, 4, 4>(wp, chunks, pp, scale, zero, s); break;
    case 8: launch_cpt<kF16, 8, 4>(wp, chunks, pp, scale, zero, s); break;
    case 16: launch_cpt<kF16, 16, 4>(wp, chunks, pp, scale, zero, s); break;
    default: launch_cpt<kF16, 32, 4>(wp, chunks, pp, scale, zero, s); break;
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
