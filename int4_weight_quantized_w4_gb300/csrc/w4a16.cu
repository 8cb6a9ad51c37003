// W4A16 skinny GEMM for decode: y[M,N] = x[M,K] . W^T with W as GPTQ int4.
//
// vLLM API docs, inc.schemes.inc_w4a8_linear (class docstring): the W4A16
// path reads the same GPTQ "NT" qweight [K/8, N] as the W4A8 path.
// vllm-omni quantization/cpu_int4.py (module docstring): decode is a bandwidth
// problem -- the whole weight is read for one token, so bits per weight set
// the token rate -- and the weight is w = (q - 8) * scale + zero.
//
// Design (GB300):
//  * Swap-AB on the warp-level tensor core: 16 output features are the MMA's
//    M rows, up to 8 tokens are its N columns (m16n8k16, bf16 in, fp32 acc).
//    Each product (q-8)*x is exact in fp32; sums are fp32.
//  * A nibble becomes the exact bf16 value q - 8 without a convert: OR it into
//    the mantissa of 128.0 (0x4300 | q == 128 + q) and subtract 136. Nibbles
//    i and i+4 of a word land in one bf16x2 register with one shift + LOP3.
//    The MMA's k order inside each 16-wide step is permuted to match (pairs
//    (k, k+4)); the token operand is permuted the same way with PRMT.
//  * Lane (r, c) of a warp loads 16-byte runs of 4 output columns for word row
//    kb = 4*step + c, so a warp reads full 128-byte lines; a warp step covers
//    64 outputs x 32 inputs. Scales (and zeros) fold into fp32 totals once per
//    group, as s * sum + z * sum(x).
//  * Split-K across the CTAs of a thread-block cluster; partial tiles are
//    summed through distributed shared memory, so no workspace is needed and
//    the output is written once, in bf16, with the bias added.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace w4 {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileN = 64;   // outputs per CTA tile
constexpr int kTok = 8;      // tokens per MMA column block
constexpr int kUnroll = 4;   // 32-wide k steps whose loads are issued together

struct Params {
  const uint16_t* x;     // bf16 [M, K]
  const uint32_t* qw;    // [K/8, N]
  const uint16_t* sc;    // fp16 or bf16 [G, N]
  const uint16_t* zr;    // bf16 [G, N] or null
  const uint16_t* bias;  // bf16 [N] or null
  uint16_t* y;           // bf16 [M, N]
  int M, N, K, group;
  int csize;             // CTAs per cluster (split-K factor)
};

W4_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                     uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16x2 (nibble i - 8, nibble i+4 - 8) of word w, exactly.
template <int I>
W4_DEV uint32_t nib_pair_bf16(uint32_t w) {
  const uint32_t t = and_or(I ? (w >> (4 * I)) : w, 0x000F000Fu, 0x43004300u);
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(0x43084308u));
  return d;
}

template <bool kScaleBf16>
W4_DEV float scale_at(uint32_t bits16) {
  return kScaleBf16 ? __uint_as_float(bits16 << 16) : half_bits_to_f32(bits16);
}

// Four consecutive 16-bit values starting at p (8-byte aligned), or zeros.
W4_DEV uint2 ld4x16(const uint16_t* p, bool in) { return in ? ld_nc_v2(p) : make_uint2(0, 0); }

template <bool kScaleBf16, bool kZero, bool kBias>
__global__ void __launch_bounds__(kThreads, 4) w4a16_kernel(const Params p) {
  __shared__ float red[kWarps][kTok * kTileN];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int nb = blockIdx.x * kTileN;
  const int m0 = blockIdx.z * kTok;
  const int N = p.N;

  // k steps of this warp: the cluster splits K, the CTA's warps split its part
  const int S = p.K / 32;
  const int rank = blockIdx.y;
  const int cs0 = (int)((long long)S * rank / p.csize), cs1 = (int)((long long)S * (rank + 1) / p.csize);
  const int t0 = cs0 + (cs1 - cs0) * warp / kWarps, t1 = cs0 + (cs1 - cs0) * (warp + 1) / kWarps;

  const int n_lo = nb + 4 * r, n_hi = nb + 32 + 4 * r;
  const bool in_lo = n_lo < N, in_hi = n_hi < N;
  const int tok = m0 + r;
  const bool tok_in = tok < p.M;
  const uint16_t* xrow = p.x + (size_t)(tok_in ? tok : 0) * p.K;

  float tot[4][4], acc[4][4], xs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) tot[j][e] = acc[j][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) xs[e] = 0.f;

  int cur_g = (t0 * 32) / p.group;

  auto fold = [&](int g) {
    const uint16_t* sp = p.sc + (size_t)g * N;
    const uint2 slo = ld4x16(sp + n_lo, in_lo), shi = ld4x16(sp + n_hi, in_hi);
    const uint32_t sl[4] = {slo.x & 0xFFFFu, slo.x >> 16, slo.y & 0xFFFFu, slo.y >> 16};
    const uint32_t sh[4] = {shi.x & 0xFFFFu, shi.x >> 16, shi.y & 0xFFFFu, shi.y >> 16};
    uint32_t zl[4] = {0, 0, 0, 0}, zh[4] = {0, 0, 0, 0};
    if (kZero) {
      const uint16_t* zp = p.zr + (size_t)g * N;
      const uint2 zlo = ld4x16(zp + n_lo, in_lo), zhi = ld4x16(zp + n_hi, in_hi);
      zl[0] = zlo.x & 0xFFFFu; zl[1] = zlo.x >> 16; zl[2] = zlo.y & 0xFFFFu; zl[3] = zlo.y >> 16;
      zh[0] = zhi.x & 0xFFFFu; zh[1] = zhi.x >> 16; zh[2] = zhi.y & 0xFFFFu; zh[3] = zhi.y >> 16;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float s_lo = scale_at<kScaleBf16>(sl[j]), s_hi = scale_at<kScaleBf16>(sh[j]);
      tot[j][0] = fmaf(s_lo, acc[j][0], tot[j][0]);
      tot[j][1] = fmaf(s_lo, acc[j][1], tot[j][1]);
      tot[j][2] = fmaf(s_hi, acc[j][2], tot[j][2]);
      tot[j][3] = fmaf(s_hi, acc[j][3], tot[j][3]);
      if (kZero) {
        const float z_lo = __uint_as_float(zl[j] << 16), z_hi = __uint_as_float(zh[j] << 16);
        tot[j][0] = fmaf(z_lo, xs[0], tot[j][0]);
        tot[j][1] = fmaf(z_lo, xs[1], tot[j][1]);
        tot[j][2] = fmaf(z_hi, xs[0], tot[j][2]);
        tot[j][3] = fmaf(z_hi, xs[1], tot[j][3]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) xs[e] = 0.f;
  };

  for (int t = t0; t < t1; t += kUnroll) {
    uint4 wl[kUnroll], wh[kUnroll], xv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int tt = t + u;
      const bool live = tt < t1;
      const size_t kb = (size_t)tt * 4 + c;
      const uint32_t* row = p.qw + kb * N;
      wl[u] = (live && in_lo) ? ld_stream_v4(row + n_lo) : make_uint4(0, 0, 0, 0);
      wh[u] = (live && in_hi) ? ld_stream_v4(row + n_hi) : make_uint4(0, 0, 0, 0);
      xv[u] = (live && tok_in) ? ld_nc_v4(xrow + kb * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int tt = t + u;
      if (tt >= t1) break;
      const int g = (tt * 32) / p.group;
      if (g != cur_g) {
        fold(cur_g);
        cur_g = g;
      }
      const uint32_t b00 = prmt(xv[u].x, xv[u].z, 0x5410u), b01 = prmt(xv[u].x, xv[u].z, 0x7632u);
      const uint32_t b10 = prmt(xv[u].y, xv[u].w, 0x5410u), b11 = prmt(xv[u].y, xv[u].w, 0x7632u);
      const uint32_t wlo[4] = {wl[u].x, wl[u].y, wl[u].z, wl[u].w};
      const uint32_t whi[4] = {wh[u].x, wh[u].y, wh[u].z, wh[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mma_bf16(acc[j], nib_pair_bf16<0>(wlo[j]), nib_pair_bf16<0>(whi[j]), nib_pair_bf16<1>(wlo[j]),
                 nib_pair_bf16<1>(whi[j]), b00, b01);
        mma_bf16(acc[j], nib_pair_bf16<2>(wlo[j]), nib_pair_bf16<2>(whi[j]), nib_pair_bf16<3>(wlo[j]),
                 nib_pair_bf16<3>(whi[j]), b10, b11);
      }
      if (kZero) {
        constexpr uint32_t one = 0x3F803F80u;  // bf16x2 (1, 1): the MMA sums x over k
        mma_bf16(xs, one, one, one, one, b00, b01);
        mma_bf16(xs, one, one, one, one, b10, b11);
      }
    }
  }
  if (t1 > t0) fold(cur_g);

  // CTA reduction: warp partials -> red[0]
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int nn = 4 * r + j;
    red[warp][(2 * c) * kTileN + nn] = tot[j][0];
    red[warp][(2 * c + 1) * kTileN + nn] = tot[j][1];
    red[warp][(2 * c) * kTileN + nn + 32] = tot[j][2];
    red[warp][(2 * c + 1) * kTileN + nn + 32] = tot[j][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTok * kTileN; i += kThreads) {
    float v = red[0][i];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) v += red[w][i];
    red[0][i] = v;
  }

  // cluster reduction through distributed shared memory; each CTA finishes a slice
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int per = (kTok * kTileN) / p.csize;
  const int i0 = rank * per;
  for (int i = i0 + threadIdx.x; i < i0 + per; i += kThreads) {
    float v = 0.f;
    for (int q = 0; q < p.csize; ++q) v += cluster.map_shared_rank(&red[0][0], q)[i];
    const int m = m0 + i / kTileN, n = nb + i % kTileN;
    if (m < p.M && n < N) {
      if (kBias) v += __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16);
      p.y[(size_t)m * N + n] = static_cast<uint16_t>(f32_to_bf16_bits(v));
    }
  }
  cluster.sync();
}

template <bool kScaleBf16, bool kZero, bool kBias>
cudaError_t launch_t(const Params& p, dim3 grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = p.csize;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w4a16_kernel<kScaleBf16, kZero, kBias>, p);
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

}  // namespace

cudaError_t launch_w4a16(const W4A16Args& a, cudaStream_t s) {
  Params p;
  p.x = static_cast<const uint16_t*>(a.x);
  p.qw = static_cast<const uint32_t*>(a.qweight);
  p.sc = static_cast<const uint16_t*>(a.w_scale);
  p.zr = static_cast<const uint16_t*>(a.zeros);
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.y = static_cast<uint16_t*>(a.y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.group = a.group;

  // Split K over a cluster so that every SM streams weights: aim for a few
  // CTAs per SM with at least 4 k steps (4 KB of weights) per warp.
  const int n_tiles = (p.N + kTileN - 1) / kTileN;
  const int m_chunks = (p.M + kTok - 1) / kTok;
  const int steps = p.K / 32;
  int csize = 1;
  while (csize < 8 && (long long)n_tiles * m_chunks * csize < 4LL * sm_count() &&
         steps / (csize * 2 * kWarps) >= 4)
    csize *= 2;
  p.csize = csize;
  if (m_chunks > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(n_tiles, csize, m_chunks);
  const bool bf = a.scale_bf16, z = a.zeros != nullptr, b = a.bias != nullptr;
  if (bf) {
    if (z) return b ? launch_t<true, true, true>(p, grid, s) : launch_t<true, true, false>(p, grid, s);
    return b ? launch_t<true, false, true>(p, grid, s) : launch_t<true, false, false>(p, grid, s);
  }
  if (z) return b ? launch_t<false, true, true>(p, grid, s) : launch_t<false, true, false>(p, grid, s);
  return b ? launch_t<false, false, true>(p, grid, s) : launch_t<false, false, false>(p, grid, s);
}

}  // namespace w4
