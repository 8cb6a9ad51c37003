// Quantized embedding table, used as the vocabulary lookup and as the tied
// output head.
//
// vllm-omni quantization/cpu_int4.py, CPUInt4EmbeddingMethod: the table is
// packed [V, D/2] bytes (two 4-bit codes per byte, low nibble first:
// pack_nibbles), with fp32 scale and zero [V, D/group] from
// quantize_groupwise, kept row major; tie_weights shares the same tensors
// with the output head. embedding(): the selected rows dequantize as
// (q - 8) * scale + zero in fp32, then round to bf16.
//
// Gather: one thread per 8 codes; the fp32 steps are taken one by one with
// IEEE rounding (__fmul_rn, __fadd_rn), so the rows are bit-exact.
//
// Head: logits[m, v] = sum_d h[m, d] * w[v, d] for decode (M <= 8 tokens).
// One warp per vocabulary row at a time (the row is D/2 contiguous bytes, read
// with 16-byte loads), h held in shared memory as fp32. A nibble becomes its
// float exactly by placing it in the mantissa of 2^23 (0x4B000000 | q is
// 2^23 + q) and subtracting 2^23; per 8-code word the partial is folded as
// s * (sum h q - 8 sum h) + z * sum h, so no weight is ever dequantized.
// Bound: HBM (the table is read once per call).
#include "common.cuh"
#include "launch.h"

namespace w4 {
namespace {

constexpr int kHeadWarps = 8;
constexpr int kHeadTok = 8;

__global__ void __launch_bounds__(256) embedding_gather_kernel(const int32_t* ids, int64_t T, const uint32_t* table,
                                                               const float* scale, const float* zero, int64_t V,
                                                               int64_t D, int group, uint16_t* out,
                                                               unsigned int* status) {
  const int64_t words = D / 8;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= T * words) return;
  const int64_t t = i / words, wi = i % words;
  const int64_t v = ids[t];
  uint4* dst = reinterpret_cast<uint4*>(out + t * D + wi * 8);
  if (v < 0 || v >= V) {   // out-of-range id: zeros, and the status word says so
    *dst = make_uint4(0, 0, 0, 0);
    report(status, W4_ERR_SHAPE);
    return;
  }
  const uint32_t w = table[v * words + wi];
  const int64_t G = D / group;
  const int64_t g = (wi * 8) / group;   // group % 8 == 0: one group per word
  const float s = scale[v * G + g], z = zero[v * G + g];
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float q0 = static_cast<float>((w >> (8 * j)) & 0xFu), q1 = static_cast<float>((w >> (8 * j + 4)) & 0xFu);
    const float d0 = __fadd_rn(__fmul_rn(q0 - 8.f, s), z), d1 = __fadd_rn(__fmul_rn(q1 - 8.f, s), z);
    o[j] = f32_to_bf16_bits(d0) | (f32_to_bf16_bits(d1) << 16);
  }
  *dst = make_uint4(o[0], o[1], o[2], o[3]);
}

// kCPL: 16-byte chunks (32 codes) of a row per lane, at most (D <= 1024 kCPL;
// lanes past the row's end idle). kM: tokens the kernel is built for, of
// which the first Mact are real (the rest read as zeros and are not written). The
// next row's chunks and scales are loaded before the current row is
// computed, so every lane keeps 2 kCPL 16-byte loads in flight; per-word sums
// of h come from shared memory (computed once per call).
template <int kM, int kCPL>
__global__ void __launch_bounds__(kHeadWarps * 32) lm_head_kernel(const uint16_t* h, const uint4* table,
                                                                   const float* scale, const float* zero, int64_t V,
                                                                   int D, int group, uint16_t* y, int Mact) {
  // h as fp32 with 4 floats of padding after every 32 (a lane reads one
  // 32-float block: the padding puts a quarter-warp's 16-byte reads in 8
  // different bank groups), then the per-word sums of h, word-major
  // ([kM][4][chunks]: neighbouring lanes read neighbouring floats)
  extern __shared__ float hs[];
  const int chunks = D / 32;
  const int Dp = chunks * 36;
  float* hw = hs + kM * Dp;
  for (int i = threadIdx.x; i < kM * D; i += blockDim.x) {
    const int m = i / D, d = i % D;
    hs[m * Dp + d + (d >> 5) * 4] = i < Mact * D ? __uint_as_float(static_cast<uint32_t>(h[i]) << 16) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kM * (D / 8); i += blockDim.x) {
    const int m = i / (D / 8), wi = i % (D / 8);     // word wi = chunk wi / 4, slot wi % 4
    const float* p = hs + m * Dp + (wi >> 2) * 36 + (wi & 3) * 8;
    hw[(m * 4 + (wi & 3)) * chunks + (wi >> 2)] = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int G = D / group;
  const bool chunk_group = group % 32 == 0;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kHeadWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kHeadWarps;
  uint4 cur[kCPL];
  float cs[kCPL], cz[kCPL];   // scale and zero of the group of each chunk's first code
  auto fetch = [&](int64_t v, uint4 (&q)[kCPL], float (&sv)[kCPL], float (&zv)[kCPL]) {
    const uint4* row = table + v * chunks;
#pragma unroll
    for (int i = 0; i < kCPL; ++i) {
      const int c = lane + 32 * i;
      if (c < chunks) {
        q[i] = ld_nc_v4(row + c);
        const int g = (c * 32) / group;
        sv[i] = __ldg(scale + v * G + g);
        zv[i] = __ldg(zero + v * G + g);
      }
    }
  };
  int64_t v = warp0;
  if (v < V) fetch(v, cur, cs, cz);
  for (; v < V; v += nwarps) {
    uint4 nxt[kCPL];
    float ns[kCPL], nz[kCPL];
    const int64_t vn = v + nwarps;
    if (vn < V) fetch(vn, nxt, ns, nz);
    float acc[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) acc[m] = 0.f;
#pragma unroll
    for (int i = 0; i < kCPL; ++i) {
      const uint32_t wv[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
      const int c = lane + 32 * i;
      if (c >= chunks) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // groups of 8 or 16 codes: words past the first group of the chunk
        // read their own scale and zero (same row, cached)
        const int gj = (c * 32 + j * 8) / group;
        const float s = chunk_group ? cs[i] : __ldg(scale + v * G + gj);
        const float z = chunk_group ? cz[i] : __ldg(zero + v * G + gj);
        const float b = fmaf(-8.f, s, z);
        float qf[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          qf[e] = __uint_as_float(0x4B000000u | ((wv[j] >> (4 * e)) & 0xFu)) - 8388608.f;
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const float* hm = hs + m * Dp + c * 36 + j * 8;
          const float4 h0 = *reinterpret_cast<const float4*>(hm), h1 = *reinterpret_cast<const float4*>(hm + 4);
          const float hq = fmaf(h0.x, qf[0], fmaf(h0.y, qf[1], fmaf(h0.z, qf[2], fmaf(h0.w, qf[3],
                           fmaf(h1.x, qf[4], fmaf(h1.y, qf[5], fmaf(h1.z, qf[6], h1.w * qf[7])))))));
          acc[m] = fmaf(s, hq, fmaf(b, hw[(m * 4 + j) * chunks + c], acc[m]));
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      float a = acc[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (lane == 0 && m < Mact) y[static_cast<int64_t>(m) * V + v] = static_cast<uint16_t>(f32_to_bf16_bits(a));
    }
#pragma unroll
    for (int i = 0; i < kCPL; ++i) {
      cur[i] = nxt[i];
      cs[i] = ns[i];
      cz[i] = nz[i];
    }
  }
}

int sm_count_embed() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

template <int kM, int kCPL>
cudaError_t launch_head(const void* h, int Mact, const void* table, const float* scale, const float* zero, int64_t V,
                        int D, int group, void* y, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(kM) * (D / 32 * 36 + D / 8) * sizeof(float);
  auto k = lm_head_kernel<kM, kCPL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kHeadWarps * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (V + kHeadWarps - 1) / kHeadWarps;
  const int64_t cap = static_cast<int64_t>(sm_count_embed()) * per_sm;   // one wave
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  k<<<grid, kHeadWarps * 32, smem, s>>>(static_cast<const uint16_t*>(h), static_cast<const uint4*>(table), scale,
                                         zero, V, D, group, static_cast<uint16_t*>(y), Mact);
  return cudaGetLastError();
}

template <int kM>
cudaError_t head_cpl(const void* h, int Mact, const void* table, const float* scale, const float* zero, int64_t V,
                     int D, int group, void* y, cudaStream_t s) {
  const int cpl = (D + 1023) / 1024;
  if (cpl <= 1) return launch_head<kM, 1>(h, Mact, table, scale, zero, V, D, group, y, s);
  if (cpl <= 2) return launch_head<kM, 2>(h, Mact, table, scale, zero, V, D, group, y, s);
  if (cpl <= 4) return launch_head<kM, 4>(h, Mact, table, scale, zero, V, D, group, y, s);
  return launch_head<kM, 8>(h, Mact, table, scale, zero, V, D, group, y, s);
}

}  // namespace

cudaError_t launch_embedding_gather(const int32_t* ids, int64_t T, const void* table, const float* scale,
                                    const float* zero, int64_t V, int64_t D, int32_t group, void* out,
                                    unsigned int* status, cudaStream_t s) {
  const int64_t n = T * (D / 8);
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  embedding_gather_kernel<<<blocks, 256, 0, s>>>(ids, T, static_cast<const uint32_t*>(table), scale, zero, V, D,
                                                  group, static_cast<uint16_t*>(out), status);
  return cudaGetLastError();
}

cudaError_t launch_lm_head(const void* h, int64_t M, const void* table, const float* scale, const float* zero,
                           int64_t V, int64_t D, int32_t group, void* y, cudaStream_t s) {
  const int Di = static_cast<int>(D);
  for (int64_t m0 = 0; m0 < M; m0 += kHeadTok) {
    const int mb = static_cast<int>(M - m0 < kHeadTok ? M - m0 : kHeadTok);
    const void* hb = static_cast<const uint16_t*>(h) + m0 * D;
    void* yb = static_cast<uint16_t*>(y) + m0 * V;
    cudaError_t e;
    if (mb == 1) {
      e = head_cpl<1>(hb, mb, table, scale, zero, V, Di, group, yb, s);
    } else if (mb <= 2) {
      e = head_cpl<2>(hb, mb, table, scale, zero, V, Di, group, yb, s);
    } else if (mb <= 4) {
      e = head_cpl<4>(hb, mb, table, scale, zero, V, Di, group, yb, s);
    } else {
      e = head_cpl<8>(hb, mb, table, scale, zero, V, Di, group, yb, s);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w4
