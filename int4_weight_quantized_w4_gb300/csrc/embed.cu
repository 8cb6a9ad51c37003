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
// Head: logits[m, v] = sum_d h[m, d] * w[v, d] for decode, tokens in blocks
// of 8 (one pass over the table per block). Bound: HBM (the table is read
// once per pass). Per scale group the partial is folded as
// s * (sum h q - 8 sum h) + z * sum h, so no weight is ever dequantized.
//
// Tensor-core form (D and the group multiples of 128, D <= 8192): a warp
// owns 16-row tiles of the table and runs swap-AB m16n8k16 MMAs (table rows
// are the MMA rows, the 8 tokens its columns, fp16 in, fp32 accumulate) over
// 128-code segments. Lane (g, t) loads bytes [16t, 16t + 16) of the segment
// from rows g and g + 8 straight from global memory, 4 segments ahead, and
// turns every word into 4 A registers with one AND each: nibbles in bits 0-3
// of an fp16 half are the exact subnormal q 2^-24, nibbles in bits 4-7 are
// 16 q 2^-24 (the h values they meet carry an extra 1/16). The k order inside
// a segment is permuted the same way for h, which every CTA stages once in
// shared memory as fp16 2^e h, with 2^e a power of two per (segment, token)
// that puts the segment's largest |h| in [2^14, 2^15) (exact; the fold
// multiplies by 2^-e). For a single token (decode) its own kernel puts
// eight segments in the MMA columns instead of eight tokens, so the fold
// runs once per eight segments, and splits the table evenly: each CTA takes
// a contiguous run of tiles and its warps equal runs of (tile, segment)
// positions. Other shapes: one warp per row on the FMA pipes, a nibble
// becoming its float as float(0x4B000000 | q) - 2^23.
#include <cuda_fp16.h>

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

constexpr int kTcWarps = 20;   // one CTA per SM (640 threads, up to 96 registers): h is staged once per SM
constexpr int kTcAhead = 4;        // segments of loads in flight per warp
constexpr int kSegBytes = 288;     // one (segment, token) block of staged h: 4 x 64 B + 32 B of padding

W4_DEV void mma_f16_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Staged h for one (segment, token, lane quad position t): the 32 codes
// [32t, 32t + 32) of the segment in MMA order. For word c' (codes 32t + 8c'
// + j) and half h' the B registers are (x[2h'], x[2h' + 4]) and
// (x[2h' + 1], x[2h' + 5]) / 16 with x the word's 8 values.
W4_DEV int stage_offset(int seg, int token, int t) { return (seg * 8 + token) * kSegBytes + t * 64 + (t >> 1) * 16; }

__global__ void __launch_bounds__(kTcWarps * 32) lm_head_tc_kernel(const uint16_t* __restrict__ h, int Mact,
                                                                     const uint8_t* __restrict__ table,
                                                                     const float* __restrict__ scale,
                                                                     const float* __restrict__ zero, int64_t V,
                                                                     int D, int group, uint16_t* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int S = D / 128;
  float4* fold = reinterpret_cast<float4*>(smem + S * 8 * kSegBytes);   // [S][4]: (X_2t, X_2t+1, f_2t, f_2t+1)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  // --- stage h: one warp per (segment, token); lane i holds codes 4i..4i+3
  for (int task = warp; task < S * 8; task += kTcWarps) {
    const int seg = task >> 3, tok = task & 7;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (tok < Mact) {
      const uint16_t* hp = h + static_cast<int64_t>(tok) * D + seg * 128 + lane * 4;   // h is only 2-byte aligned
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(static_cast<uint32_t>(hp[i]) << 16);
    }
    float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    float sm = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      sm += __shfl_xor_sync(0xffffffffu, sm, o);
    }
    // 2^e with the largest |h| 2^e in [2^14, 2^15): from the exponent field
    // of mx (mx in [2^(E-127), 2^(E-126))), clamped so that 2^e, 2^(e-4) and
    // 2^-e are normal floats (every bf16 magnitude stays in range)
    const int E = static_cast<int>(__float_as_uint(mx) >> 23);
    const int e = mx > 0.f ? min(max(141 - E, -113), 121) : 0;
    const float sc = __int_as_float((127 + e) << 23), sc16 = __int_as_float((123 + e) << 23);
    // code c = 4 lane + i sits in quad position tt = c / 32, word c' = (c % 32) / 8, slot j = c % 8;
    // slot j -> B register 4 c' + 2 h' + odd (h' = (j / 2) % 2, odd = j % 2), half j / 4
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane * 4 + i;
      const int tt = c >> 5, cw = (c & 31) >> 3, j = c & 7;
      const int hp = (j >> 1) & 1, odd = j & 1, hi = j >> 2;
      const __half hv = __float2half_rn(v[i] * (odd ? sc16 : sc));
      reinterpret_cast<uint16_t*>(smem + stage_offset(seg, tok, tt))[(cw * 4 + hp * 2 + odd) * 2 + hi] =
          __half_as_ushort(hv);
    }
    if (lane == 0) {
      // fold data for the token pair (tok & ~1, tok | 1) lives at fold[seg * 4 + tok / 2]
      float* f = reinterpret_cast<float*>(&fold[seg * 4 + (tok >> 1)]);
      f[tok & 1] = sm * 5.9604644775390625e-8f;            // 2^-24 sum h, exact scaling
      f[2 + (tok & 1)] = __int_as_float((127 - e) << 23);  // 2^-e
    }
  }
  __syncthreads();

  const int64_t ntiles = (V + 15) / 16;
  const int64_t wg = static_cast<int64_t>(blockIdx.x) * kTcWarps + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kTcWarps;
  if (wg >= ntiles) return;
  // 32-bit position counters: a warp's share of any table that fits in memory is far below 2^31 segments
  const int npos = static_cast<int>((ntiles - 1 - wg) / nw + 1) * S;
  const int64_t rowb = D / 2;
  const int G = D / group, spg = group / 128;   // segments per scale group

  // load cursor: rows g and g + 8 of tile ltile (clamped into the table), at segment lseg
  int64_t ltile = wg;
  int lseg = 0;
  const uint8_t* la;
  const uint8_t* lb;
  auto rows_of = [&](int64_t tile, int64_t& r0, int64_t& r1) {
    r0 = tile * 16 + g;
    r1 = r0 + 8;
    r0 = r0 < V ? r0 : V - 1;
    r1 = r1 < V ? r1 : V - 1;
  };
  auto set_load_tile = [&]() {
    int64_t r0, r1;
    rows_of(ltile, r0, r1);
    la = table + r0 * rowb + t * 16;
    lb = table + r1 * rowb + t * 16;
  };
  set_load_tile();
  auto load = [&](uint4& a, uint4& b) {
    a = ld_stream_v4(la + lseg * 64);
    b = ld_stream_v4(lb + lseg * 64);
    if (++lseg == S) {
      lseg = 0;
      ltile += nw;
      if (ltile < ntiles) set_load_tile();
    }
  };
  uint4 A[kTcAhead][2];
#pragma unroll
  for (int p = 0; p < kTcAhead; ++p)
    if (p < npos) load(A[p][0], A[p][1]);

  // compute cursor: tile ctile at segment cseg, its rows' scale and zero rows
  int64_t ctile = wg;
  int cseg = 0, cgrp = 0, cin = 0;   // segment, its scale group, segments left in the group
  const float* sa;
  const float* sb;
  const float* za;
  const float* zb;
  auto set_compute_tile = [&]() {
    int64_t r0, r1;
    rows_of(ctile, r0, r1);
    sa = scale + r0 * G;
    sb = scale + r1 * G;
    za = zero + r0 * G;
    zb = zero + r1 * G;
  };
  set_compute_tile();
  const uint8_t* bbase = smem + stage_offset(0, g, t);
  float tot[4] = {0.f, 0.f, 0.f, 0.f};
  float s0 = 0.f, s1 = 0.f, b0 = 0.f, b1 = 0.f;
  for (int pos0 = 0; pos0 < npos; pos0 += kTcAhead) {
#pragma unroll
    for (int p = 0; p < kTcAhead; ++p) {
      if (pos0 + p < npos) {
        if (cin == 0) {                           // a new scale group for this tile's rows
          s0 = __ldg(sa + cgrp);
          s1 = __ldg(sb + cgrp);
          b0 = fmaf(-8.f, s0, __ldg(za + cgrp));
          b1 = fmaf(-8.f, s1, __ldg(zb + cgrp));
          ++cgrp;
          cin = spg;
        }
        --cin;
        const uint4* bp = reinterpret_cast<const uint4*>(bbase + cseg * (8 * kSegBytes));
        const uint4 B0 = bp[0], B1 = bp[1], B2 = bp[2], B3 = bp[3];
        const uint32_t b[16] = {B0.x, B0.y, B0.z, B0.w, B1.x, B1.y, B1.z, B1.w,
                                B2.x, B2.y, B2.z, B2.w, B3.x, B3.y, B3.z, B3.w};
        const uint32_t wv[4] = {A[p][0].x, A[p][0].y, A[p][0].z, A[p][0].w};
        const uint32_t vv[4] = {A[p][1].x, A[p][1].y, A[p][1].z, A[p][1].w};
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cw = 0; cw < 4; ++cw) {
          mma_f16_acc(acc, wv[cw] & 0x000F000Fu, vv[cw] & 0x000F000Fu, wv[cw] & 0x00F000F0u, vv[cw] & 0x00F000F0u,
                      b[cw * 4 + 0], b[cw * 4 + 1]);
          const uint32_t w2 = wv[cw] >> 8, v2 = vv[cw] >> 8;
          mma_f16_acc(acc, w2 & 0x000F000Fu, v2 & 0x000F000Fu, w2 & 0x00F000F0u, v2 & 0x00F000F0u, b[cw * 4 + 2],
                      b[cw * 4 + 3]);
        }
        if (pos0 + p + kTcAhead < npos) load(A[p][0], A[p][1]);
        const float4 f = fold[cseg * 4 + t];
        tot[0] = fmaf(s0 * f.z, acc[0], fmaf(b0, f.x, tot[0]));
        tot[1] = fmaf(s0 * f.w, acc[1], fmaf(b0, f.y, tot[1]));
        tot[2] = fmaf(s1 * f.z, acc[2], fmaf(b1, f.x, tot[2]));
        tot[3] = fmaf(s1 * f.w, acc[3], fmaf(b1, f.y, tot[3]));
        if (++cseg == S) {                        // tile done: rows g, g + 8; tokens 2t, 2t + 1
          const int64_t r0 = ctile * 16 + g, r1 = r0 + 8;
          const int m0 = 2 * t, m1 = 2 * t + 1;
          if (r0 < V && m0 < Mact) y[m0 * V + r0] = static_cast<uint16_t>(f32_to_bf16_bits(tot[0] * 16777216.f));
          if (r0 < V && m1 < Mact) y[m1 * V + r0] = static_cast<uint16_t>(f32_to_bf16_bits(tot[1] * 16777216.f));
          if (r1 < V && m0 < Mact) y[m0 * V + r1] = static_cast<uint16_t>(f32_to_bf16_bits(tot[2] * 16777216.f));
          if (r1 < V && m1 < Mact) y[m1 * V + r1] = static_cast<uint16_t>(f32_to_bf16_bits(tot[3] * 16777216.f));
          tot[0] = tot[1] = tot[2] = tot[3] = 0.f;
          cseg = 0;
          cgrp = 0;
          cin = 0;
          ctile += nw;
          if (ctile < ntiles) set_compute_tile();
        }
      }
    }
  }
}

// One token (decode): 24 warps a CTA, 3 segments of row loads in flight per
// warp (up to 85 registers a thread).
constexpr int kTc1Warps = 24;
constexpr int kTc1Ahead = 3;

// The tensor-core head for a single token. B column n carries segment 8w + n
// of each window of eight segments: the lanes whose column matches the
// segment's place in the window read the token's staged h, the others a
// zero block. So column n accumulates segment 8w + n alone, the
// accumulators run over the whole window, and the fold (lane (g, t) folds
// segments 8w + 2t and 8w + 2t + 1 of rows g and g + 8) runs once per window.
//
// Work split: CTA b takes the tiles [b T / grid, (b + 1) T / grid) and its
// warps split their (tile, segment) positions, tile-major, into equal runs,
// so every SM and every warp has the same work to within one tile and one
// segment. A warp writes the rows of every tile it covers whole; a tile
// shared by several warps leaves one partial row sum per warp in shared
// memory, which the warp holding the tile's first segment adds up in warp
// order at the end.
__global__ void __launch_bounds__(kTc1Warps * 32) lm_head_tc1_kernel(const uint16_t* __restrict__ h,
                                                                       const uint8_t* __restrict__ table,
                                                                       const float* __restrict__ scale,
                                                                       const float* __restrict__ zero, int64_t V,
                                                                       int D, int group, uint16_t* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int S = D / 128, S8 = (S + 7) & ~7;
  // staged h: [S][2] blocks of kSegBytes, (segment, 0) the token's, (segment, 1) zeros, each in
  // stage_offset's order
  // fold data [S8 / 2]: (X_2j, X_2j+1, f_2j, f_2j+1) for segment pairs, X = 2^-24 sum h, f = 2^-e
  float4* fold = reinterpret_cast<float4*>(smem + S * 2 * kSegBytes);
  float* part = reinterpret_cast<float*>(fold + S8 / 2);                // [kTc1Warps][2][16] partial rows
  uint8_t* gos = reinterpret_cast<uint8_t*>(part + kTc1Warps * 2 * 16);  // scale group of each segment
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t ntiles = (V + 15) / 16;
  const int64_t rowb = D / 2;
  const int G = D / group, spg = group / 128;   // segments per scale group
  auto blk = [](int seg, int zblk, int tt) { return (seg * 2 + zblk) * kSegBytes + tt * 64 + (tt >> 1) * 16; };

  // this warp's run [p0, p1) of the CTA's positions (every CTA has a tile)
  int npos;   // positions in the run: 32 bits, far more than a warp's share of any table that fits in memory
  int64_t tile0;
  int seg0;
  {
    const int64_t T0 = static_cast<int64_t>(blockIdx.x) * ntiles / gridDim.x;
    const int64_t P = (static_cast<int64_t>(blockIdx.x + 1) * ntiles / gridDim.x - T0) * S;
    const int64_t p0 = warp * P / kTc1Warps;
    npos = static_cast<int>((warp + 1) * P / kTc1Warps - p0);
    tile0 = T0 + p0 / S;
    seg0 = static_cast<int>(p0 % S);
  }

  // --- stage h: one warp per (segment, block); lane i holds codes 4i..4i+3
  if (threadIdx.x < S) gos[threadIdx.x] = static_cast<uint8_t>(threadIdx.x / spg);
  for (int task = warp; task < S8 * 2; task += kTc1Warps) {
    const int seg = task >> 1, zblk = task & 1;
    if (seg >= S) {   // columns past the last segment of a partial window fold zeros
      if (lane == 0 && zblk == 0) {
        float* f = reinterpret_cast<float*>(&fold[seg >> 1]);
        f[seg & 1] = 0.f;
        f[2 + (seg & 1)] = 0.f;
      }
      continue;
    }
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (zblk == 0) {
      const uint16_t* hp = h + seg * 128 + lane * 4;   // h is only 2-byte aligned
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(static_cast<uint32_t>(hp[i]) << 16);
    }
    float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    float sm = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      sm += __shfl_xor_sync(0xffffffffu, sm, o);
    }
    // the segment's power of two, as in lm_head_tc_kernel
    const int E = static_cast<int>(__float_as_uint(mx) >> 23);
    const int e = mx > 0.f ? min(max(141 - E, -113), 121) : 0;
    const float sc = __int_as_float((127 + e) << 23), sc16 = __int_as_float((123 + e) << 23);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane * 4 + i;
      const int tt = c >> 5, cw = (c & 31) >> 3, j = c & 7;
      const int hp = (j >> 1) & 1, odd = j & 1, hi = j >> 2;
      const __half hv = __float2half_rn(v[i] * (odd ? sc16 : sc));
      reinterpret_cast<uint16_t*>(smem + blk(seg, zblk, tt))[(cw * 4 + hp * 2 + odd) * 2 + hi] = __half_as_ushort(hv);
    }
    if (lane == 0 && zblk == 0) {   // segment pair seg / 2, member seg % 2
      float* f = reinterpret_cast<float*>(&fold[seg >> 1]);
      f[seg & 1] = sm * 5.9604644775390625e-8f;          // 2^-24 sum h, exact scaling
      f[2 + (seg & 1)] = __int_as_float((127 - e) << 23);  // 2^-e
    }
  }
  __syncthreads();

  if (npos > 0) {
    // load cursor: rows g and g + 8 of tile ltile (clamped into the table), at segment lseg
    int64_t ltile = tile0;
    int lseg = seg0;
    const uint8_t* la;
    const uint8_t* lb;
    auto rows_of = [&](int64_t tile, int64_t& r0, int64_t& r1) {
      r0 = tile * 16 + g;
      r1 = r0 + 8;
      r0 = r0 < V ? r0 : V - 1;
      r1 = r1 < V ? r1 : V - 1;
    };
    auto set_load_tile = [&]() {
      int64_t r0, r1;
      rows_of(ltile, r0, r1);
      la = table + r0 * rowb + t * 16;
      lb = table + r1 * rowb + t * 16;
    };
    set_load_tile();
    auto load = [&](uint4& a, uint4& b) {
      a = ld_stream_v4(la + lseg * 64);
      b = ld_stream_v4(lb + lseg * 64);
      if (++lseg == S) {
        lseg = 0;
        ++ltile;
        if (ltile < ntiles) set_load_tile();
      }
    };
    uint4 A[kTc1Ahead][2];
#pragma unroll
    for (int p = 0; p < kTc1Ahead; ++p)
      if (p < npos) load(A[p][0], A[p][1]);

    // compute cursor: tile ctile at segment cseg; this warp's piece of the
    // tile began at pstart; piece 0 is the warp's first tile, piece 1 its last
    int64_t ctile = tile0;
    int cseg = seg0, pstart = seg0, piece = 0;
    const float* sa;
    const float* sb;
    const float* za;
    const float* zb;
    auto set_compute_tile = [&]() {
      int64_t r0, r1;
      rows_of(ctile, r0, r1);
      sa = scale + r0 * G;
      sb = scale + r1 * G;
      za = zero + r0 * G;
      zb = zero + r1 * G;
    };
    set_compute_tile();
    float tot0 = 0.f, tot1 = 0.f;   // rows g, g + 8
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    // scale s and b = z - 8 s of rows g, g + 8 for segments 8w + 2t (s0, s1) and 8w + 2t + 1 (s2, s3)
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
    for (int pos0 = 0; pos0 < npos; pos0 += kTc1Ahead) {
#pragma unroll
      for (int p = 0; p < kTc1Ahead; ++p) {
        if (pos0 + p < npos) {
          if ((cseg & 7) == 0 || cseg == pstart) {   // window start: this lane's two segments' groups
            const int ga = gos[min((cseg & ~7) + 2 * t, S - 1)], gb = gos[min((cseg & ~7) + 2 * t + 1, S - 1)];
            s0 = __ldg(sa + ga);
            s1 = __ldg(sb + ga);
            s2 = __ldg(sa + gb);
            s3 = __ldg(sb + gb);
            b0 = fmaf(-8.f, s0, __ldg(za + ga));
            b1 = fmaf(-8.f, s1, __ldg(zb + ga));
            b2 = fmaf(-8.f, s2, __ldg(za + gb));
            b3 = fmaf(-8.f, s3, __ldg(zb + gb));
          }
          const uint4* bp = reinterpret_cast<const uint4*>(smem + blk(cseg, g == (cseg & 7) ? 0 : 1, t));
          const uint4 B0 = bp[0], B1 = bp[1], B2 = bp[2], B3 = bp[3];
          const uint32_t b[16] = {B0.x, B0.y, B0.z, B0.w, B1.x, B1.y, B1.z, B1.w,
                                  B2.x, B2.y, B2.z, B2.w, B3.x, B3.y, B3.z, B3.w};
          const uint32_t wv[4] = {A[p][0].x, A[p][0].y, A[p][0].z, A[p][0].w};
          const uint32_t vv[4] = {A[p][1].x, A[p][1].y, A[p][1].z, A[p][1].w};
#pragma unroll
          for (int cw = 0; cw < 4; ++cw) {
            mma_f16_acc(acc, wv[cw] & 0x000F000Fu, vv[cw] & 0x000F000Fu, wv[cw] & 0x00F000F0u,
                        vv[cw] & 0x00F000F0u, b[cw * 4 + 0], b[cw * 4 + 1]);
            const uint32_t w2 = wv[cw] >> 8, v2 = vv[cw] >> 8;
            mma_f16_acc(acc, w2 & 0x000F000Fu, v2 & 0x000F000Fu, w2 & 0x00F000F0u, v2 & 0x00F000F0u,
                        b[cw * 4 + 2], b[cw * 4 + 3]);
          }
          if (pos0 + p + kTc1Ahead < npos) load(A[p][0], A[p][1]);
          const bool tile_end = cseg == S - 1, last = pos0 + p + 1 == npos;
          if ((cseg & 7) == 7 || tile_end || last) {   // fold the window's segments in [pstart, cseg]
            const float4 f = fold[(cseg >> 3) * 4 + t];
            const int se = (cseg & ~7) + 2 * t;
            if (se >= pstart && se <= cseg) {
              tot0 = fmaf(s0 * f.z, acc[0], fmaf(b0, f.x, tot0));
              tot1 = fmaf(s1 * f.z, acc[2], fmaf(b1, f.x, tot1));
            }
            if (se + 1 >= pstart && se + 1 <= cseg) {
              tot0 = fmaf(s2 * f.w, acc[1], fmaf(b2, f.y, tot0));
              tot1 = fmaf(s3 * f.w, acc[3], fmaf(b3, f.y, tot1));
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
          }
          if (tile_end || last) {   // this warp's piece of the tile is done; the quad's lanes hold different segments
            tot0 += __shfl_xor_sync(0xffffffffu, tot0, 1);
            tot1 += __shfl_xor_sync(0xffffffffu, tot1, 1);
            tot0 += __shfl_xor_sync(0xffffffffu, tot0, 2);
            tot1 += __shfl_xor_sync(0xffffffffu, tot1, 2);
            if (t == 0) {
              const int64_t r0 = ctile * 16 + g, r1 = r0 + 8;
              if (pstart == 0 && tile_end) {   // the whole tile
                if (r0 < V) y[r0] = static_cast<uint16_t>(f32_to_bf16_bits(tot0 * 16777216.f));
                if (r1 < V) y[r1] = static_cast<uint16_t>(f32_to_bf16_bits(tot1 * 16777216.f));
              } else {   // part of a tile that other warps of this CTA share: kept for the end
                part[(warp * 2 + piece) * 16 + g] = tot0;
                part[(warp * 2 + piece) * 16 + g + 8] = tot1;
              }
            }
            tot0 = tot1 = 0.f;
          }
          if (tile_end) {
            cseg = 0;
            pstart = 0;
            piece = 1;
            ++ctile;
            if (ctile < ntiles) set_compute_tile();
          } else {
            ++cseg;
          }
        }
      }
    }
  }

  __syncthreads();
  {
    // the run's bounds again, from fresh reads of the CTA index (cheaper than
    // keeping them in registers through the main loop)
    unsigned bx, nb;
    asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(bx));
    asm volatile("mov.u32 %0, %%nctaid.x;" : "=r"(nb));
    const int64_t T0 = static_cast<int64_t>(bx) * ntiles / nb;
    const int64_t P = (static_cast<int64_t>(bx + 1) * ntiles / nb - T0) * S;
    const int64_t p0 = warp * P / kTc1Warps, p1 = (warp + 1) * P / kTc1Warps;
    const int64_t tl = (p1 - 1) / S;   // the warp's last tile, CTA-local
    // a shared tile whose first segment this warp holds: add the pieces in warp order
    if (p1 > p0 && p1 % S != 0 && p0 <= tl * S && lane < 16) {
      float a = part[(warp * 2 + (p0 / S == tl ? 0 : 1)) * 16 + lane];
      for (int w = warp + 1; w < kTc1Warps; ++w) {   // the later warps' first pieces
        const int64_t q0 = w * P / kTc1Warps, q1 = (w + 1) * P / kTc1Warps;
        if (q0 >= (tl + 1) * S) break;
        if (q1 > q0) a += part[(w * 2) * 16 + lane];
      }
      const int64_t r = (T0 + tl) * 16 + lane;
      if (r < V) y[r] = static_cast<uint16_t>(f32_to_bf16_bits(a * 16777216.f));
    }
  }
}

int sm_count_embed() { return current_sm_count(); }

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

cudaError_t launch_head_tc(const void* h, int Mact, const void* table, const float* scale, const float* zero,
                           int64_t V, int D, int group, void* y, cudaStream_t s) {
  const int S = D / 128;
  const size_t smem = static_cast<size_t>(S) * 8 * kSegBytes + static_cast<size_t>(S) * 4 * sizeof(float4);
  cudaError_t e = cudaFuncSetAttribute(lm_head_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lm_head_tc_kernel, kTcWarps * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t ntiles = (V + 15) / 16;
  const int64_t want = (ntiles + kTcWarps - 1) / kTcWarps;
  const int64_t cap = static_cast<int64_t>(sm_count_embed()) * per_sm;   // one wave
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  lm_head_tc_kernel<<<grid, kTcWarps * 32, smem, s>>>(static_cast<const uint16_t*>(h), Mact,
                                                      static_cast<const uint8_t*>(table), scale, zero, V, D, group,
                                                      static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

cudaError_t launch_head_tc1(const void* h, const void* table, const float* scale, const float* zero, int64_t V, int D,
                            int group, void* y, cudaStream_t s) {
  const int S = D / 128, S8 = (S + 7) & ~7;
  const size_t smem = static_cast<size_t>(S) * 2 * kSegBytes + static_cast<size_t>(S8 / 2) * sizeof(float4) +
                      static_cast<size_t>(kTc1Warps) * 2 * 16 * sizeof(float) + 64;
  cudaError_t e = cudaFuncSetAttribute(lm_head_tc1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lm_head_tc1_kernel, kTc1Warps * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t ntiles = (V + 15) / 16;
  const int64_t cap = static_cast<int64_t>(sm_count_embed()) * per_sm;   // one wave, every CTA with a tile
  const unsigned grid = static_cast<unsigned>(ntiles < cap ? ntiles : cap);
  lm_head_tc1_kernel<<<grid, kTc1Warps * 32, smem, s>>>(static_cast<const uint16_t*>(h),
                                                        static_cast<const uint8_t*>(table), scale, zero, V, D, group,
                                                        static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

cudaError_t launch_lm_head(const void* h, int64_t M, const void* table, const float* scale, const float* zero,
                           int64_t V, int64_t D, int32_t group, void* y, cudaStream_t s) {
  const int Di = static_cast<int>(D);
  const bool tc = D % 128 == 0 && group % 128 == 0 && D <= 8192;
  for (int64_t m0 = 0; m0 < M; m0 += kHeadTok) {
    const int mb = static_cast<int>(M - m0 < kHeadTok ? M - m0 : kHeadTok);
    const void* hb = static_cast<const uint16_t*>(h) + m0 * D;
    void* yb = static_cast<uint16_t*>(y) + m0 * V;
    cudaError_t e;
    if (tc && mb == 1) {
      e = launch_head_tc1(hb, table, scale, zero, V, Di, group, yb, s);
    } else if (tc) {
      e = launch_head_tc(hb, mb, table, scale, zero, V, Di, group, yb, s);
    } else if (mb == 1) {
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
