// The routed MoE layer around the grouped W4AFP8 GEMM: top-k routing with the
// expert-sorted row order, SiLU(gate) * up with per-row e4m3 requantization
// between the two GEMMs, and the weighted combine of the k expert rows of
// every token.
//
// vLLM API docs, quantization.w4afp8 (module docstring, W4AFP8Config
// get_quant_method): int4 group-128 weights serve the routed experts, with
// 8-bit float activations quantized per token. The pages print no routing or
// activation formula; the plain top-k MoE layer is taken:
//   * per token, the k experts with the largest router logits (equal logits:
//     lower expert index first); weight = softmax probability, divided by
//     the sum over the k chosen when renormalizing;
//   * rows (token, choice) listed by expert, then token;
//   * act = silu(gate) * up in fp32 (gate = first half of the gate_up
//     columns), rounded to bf16, quantized per row like the first input;
//   * out[t] = sum_j w[t, j] * y[row(t, j)].
//
// Routing is four short launches: a warp per token selects the k experts; a
// block per 256-token tile counts each expert's rows in the tile; one block
// turns the counts into expert offsets and per-tile bases; a block per tile
// ranks its rows inside each expert by token (bit masks of the tile's tokens
// per expert and popcounts) and writes the row order and its inverse. The
// activation and combine kernels are bandwidth-bound row passes.
#include "common.cuh"
#include "launch.h"

namespace w4 {
namespace {

constexpr int kTile = 256;   // tokens per tile (8 warps)
constexpr int kTileWarps = kTile / 32;

// Top-k selection and softmax weights, one warp per token. Lane l holds the
// logits of experts l, l + 32, ...
template <int kEPL>
__global__ void __launch_bounds__(256) route_kernel(const void* __restrict__ logits, bool bf16, int64_t T, int E,
                                                    int k, bool renorm, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nw) {
    float v[kEPL];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kEPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        v[i] = bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(logits)[t * E + e]) << 16)
                    : static_cast<const float*>(logits)[t * E + e];
        if (isnan(v[i])) v[i] = -INFINITY;   // out of contract; keeps every selection in [0, E)
        mx = fmaxf(mx, v[i]);
      } else {
        v[i] = -INFINITY;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < kEPL; ++i)
      if (lane + 32 * i < E) sum += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

    uint32_t taken = 0;          // bit i: expert lane + 32 i already chosen
    float pj[2] = {0.f, 0.f};    // choice j's unnormalized probability, on lane j % 32
    int ej[2] = {0, 0};
    float chosen = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < kEPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if (lane == (be & 31)) taken |= 1u << (be >> 5);
      const float p = expf(bv - mx);
      chosen += p;
      if (lane == (j & 31)) {
        if (j < 32) {
          pj[0] = p;
          ej[0] = be;
        } else {
          pj[1] = p;
          ej[1] = be;
        }
      }
    }
    const float den = renorm ? chosen : sum;
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const int j = lane + 32 * s2;
      if (j < k) {
        ids[t * k + j] = ej[s2];
        wts[t * k + j] = __fdiv_rn(pj[s2], den);
      }
    }
  }
}

// Per 256-token tile and expert: kPlace false writes the tile's row count to
// tile_rows[tile][e]; kPlace true takes tile_rows as the tile's first row in
// each expert and writes row_token and row_of. ids are the route kernel's
// (all in [0, E)).
template <bool kPlace>
__global__ void __launch_bounds__(kTile) tile_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int E,
                                                     int32_t* __restrict__ tile_rows, int32_t* __restrict__ row_token,
                                                     int32_t* __restrict__ row_of) {
  extern __shared__ uint32_t sm[];
  uint32_t* bits = sm;                                   // [8 warps][E]: lanes of the warp that chose e
  int32_t* first = reinterpret_cast<int32_t*>(sm + kTileWarps * E);   // [8][E] (kPlace)
  const int tile = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kTileWarps * E; i += kTile) bits[i] = 0;
  __syncthreads();
  const int64_t t = static_cast<int64_t>(tile) * kTile + threadIdx.x;
  if (t < T)
    for (int j = 0; j < k; ++j) atomicOr(&bits[warp * E + ids[t * k + j]], 1u << lane);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kTile) {
    int run = kPlace ? tile_rows[static_cast<int64_t>(tile) * E + e] : 0;
    for (int w = 0; w < kTileWarps; ++w) {
      if (kPlace) first[w * E + e] = run;
      run += __popc(bits[w * E + e]);
    }
    if (!kPlace) tile_rows[static_cast<int64_t>(tile) * E + e] = run;
  }
  if (!kPlace) return;
  __syncthreads();
  if (t < T) {
    const uint32_t below = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j];
      const int r = first[warp * E + e] + __popc(bits[warp * E + e] & below);
      row_token[r] = static_cast<int32_t>(t);
      row_of[t * k + j] = r;
    }
  }
}

// Expert offsets and per-tile bases from the per-tile counts (one block).
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) scan_kernel(int32_t* __restrict__ tile_rows, int ntiles, int E,
                                                            int32_t* __restrict__ offsets) {
  __shared__ int32_t part[kScanThreads / 32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e0 = 0; e0 < E; e0 += kScanThreads) {
    const int e = e0 + threadIdx.x;
    int total = 0;
    if (e < E) {
      for (int tl = 0; tl < ntiles; ++tl) {       // tile bases inside the expert
        const int c = tile_rows[static_cast<int64_t>(tl) * E + e];
        tile_rows[static_cast<int64_t>(tl) * E + e] = total;
        total += c;
      }
    }
    int inc = total;                              // block-wide inclusive scan of the totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    if (lane == 31) part[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int w = part[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      part[lane] = w;
    }
    __syncthreads();
    const int base = carry + (warp > 0 ? part[warp - 1] : 0) + inc - total;
    if (e < E) {
      offsets[e] = base;
      for (int tl = 0; tl < ntiles; ++tl) tile_rows[static_cast<int64_t>(tl) * E + e] += base;
    }
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) carry += part[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[E] = carry;
}

// silu(g) = g / (1 + e^-g) in fp32 with the fast exponential and divide (a
// few ulp; the bf16 result it feeds is what the reading fixes), written with
// the one exponential t = e^-|g| in (0, 1]: g / (1 + t) for g >= 0 and
// g t / (1 + t) for g < 0 (numerator and denominator multiplied by e^g). The
// denominator stays in [1, 2], inside the fast divide's range for every g.
W4_DEV float silu_f32(float g) {
  const float t = __expf(-fabsf(g));
  return __fdividef(g >= 0.f ? g : g * t, 1.f + t);
}

// act = bf16(silu(g) * u) for one chunk of 8 gate and 8 up values.
W4_DEV uint4 silu_mul_chunk(const uint4& g, const uint4& u) {
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a0 = silu_f32(bf16_lo(gw[i])) * bf16_lo(uw[i]);
    const float a1 = silu_f32(bf16_hi(gw[i])) * bf16_hi(uw[i]);
    o[i] = pack_bf16x2(a0, a1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Halfwise magnitude maximum of a chunk of bf16 pairs.
W4_DEV uint32_t chunk_absmax2_bf16(uint32_t m, const uint4& v) {
  return absmax2<false>(absmax2<false>(m, v.x), absmax2<false>(absmax2<false>(v.y, v.z), v.w));
}

// One CTA per row; NCH chunks of 8 per thread kept in registers (NCH == 0:
// long rows, computed twice).
constexpr int kActThreads = 256;
template <int NCH>
__global__ void __launch_bounds__(kActThreads) silu_mul_quant_kernel(const uint4* __restrict__ h, int I8,
                                                                     uint2* __restrict__ q, float* __restrict__ scale,
                                                                     uint4* __restrict__ act) {
  __shared__ float red[kActThreads / 32];
  const size_t row = blockIdx.x;
  const uint4* hr = h + row * 2 * static_cast<size_t>(I8);
  const size_t o0 = row * static_cast<size_t>(I8);
  auto amax_of = [&](float m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int lane = threadIdx.x & 31;
    if (lane == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    // every group of 8 lanes holds the (up to 8) warp maxima, zero past the
    // last warp; a butterfly within the group leaves the maximum in every lane
    float r = (lane & 7) < static_cast<int>(blockDim.x >> 5) ? red[lane & 7] : 0.f;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, o));
    return r;
  };
  auto store = [&](size_t i, const uint4& a, const QuotientBracket& b) {
    q[o0 + i] = quant_e4m3_chunk<false>(a, b);
    if (act != nullptr) act[o0 + i] = a;
  };
  auto amax_word = [](uint32_t m2) { return fmaxf(fabsf(bf16_lo(m2)), fabsf(bf16_hi(m2))); };
  if constexpr (NCH > 0) {
    uint4 a[NCH];
    uint32_t m2 = 0;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int i = threadIdx.x + c * blockDim.x;
      a[c] = i < I8 ? silu_mul_chunk(ld_stream_v4(hr + i), ld_stream_v4(hr + I8 + i)) : make_uint4(0, 0, 0, 0);
      m2 = chunk_absmax2_bf16(m2, a[c]);
    }
    const float amax = amax_of(amax_word(m2));
    const float s = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
    const QuotientBracket b = quotient_bracket(s);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int i = threadIdx.x + c * blockDim.x;
      if (i < I8) store(i, a[c], b);
    }
    if (threadIdx.x == 0) scale[row] = s;
  } else {
    uint32_t m2 = 0;
    for (int i = threadIdx.x; i < I8; i += blockDim.x)
      m2 = chunk_absmax2_bf16(m2, silu_mul_chunk(ld_nc_v4(hr + i), ld_nc_v4(hr + I8 + i)));
    const float amax = amax_of(amax_word(m2));
    const float s = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
    const QuotientBracket b = quotient_bracket(s);
    for (int i = threadIdx.x; i < I8; i += blockDim.x)
      store(i, silu_mul_chunk(ld_stream_v4(hr + i), ld_stream_v4(hr + I8 + i)), b);
    if (threadIdx.x == 0) scale[row] = s;
  }
}

// One warp per row for many rows of I up to 2048 (NCH <= 8 chunks per lane),
// four rows a CTA: the gate and up chunks of the whole row are loaded before
// any is used, the row maximum is a shuffle butterfly with no block barrier.
constexpr int kActRowsPerCta = 4;
template <int NCH>
__global__ void __launch_bounds__(32 * kActRowsPerCta) silu_mul_quant_warp(const uint4* __restrict__ h, int64_t R,
                                                                          int I8, uint2* __restrict__ q,
                                                                          float* __restrict__ scale,
                                                                          uint4* __restrict__ act) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kActRowsPerCta + (threadIdx.x >> 5);
  if (row >= R) return;                       // the whole warp
  const uint4* hr = h + static_cast<size_t>(row) * 2 * static_cast<size_t>(I8);
  const size_t o0 = static_cast<size_t>(row) * static_cast<size_t>(I8);
  uint4 g[NCH], u[NCH];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = lane + 32 * j;
    g[j] = c < I8 ? ld_stream_v4(hr + c) : make_uint4(0, 0, 0, 0);
    u[j] = c < I8 ? ld_stream_v4(hr + I8 + c) : make_uint4(0, 0, 0, 0);
  }
  uint32_t m2 = 0;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    g[j] = silu_mul_chunk(g[j], u[j]);        // zero chunks give zero activations
    m2 = chunk_absmax2_bf16(m2, g[j]);
  }
  float amax = fmaxf(fabsf(bf16_lo(m2)), fabsf(bf16_hi(m2)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
  const QuotientBracket b = quotient_bracket(s);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = lane + 32 * j;
    if (c < I8) {
      q[o0 + c] = quant_e4m3_chunk<false>(g[j], b);
      if (act != nullptr) act[o0 + c] = g[j];
    }
  }
  if (lane == 0) scale[row] = s;
}

// out[t, 8c..8c+7] = bf16(sum_j w[t, j] * y[row_of[t, j], 8c..8c+7]), fp32,
// choices in order. A row index outside [0, R) counts as a zero row and sets
// W4_ERR_SHAPE.
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y, int64_t R, int H8,
                                                      const float* __restrict__ w, const int32_t* __restrict__ row_of,
                                                      int64_t T, int k, uint4* __restrict__ out,
                                                      unsigned int* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= T * H8) return;
  const int64_t t = i / H8;
  const int c = static_cast<int>(i % H8);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < k; ++j) {
    const int64_t r = row_of[t * k + j];
    const float wj = w[t * k + j];
    if (r < 0 || r >= R) {
      report(status, W4_ERR_SHAPE);
      continue;
    }
    const uint4 v = ld_stream_v4(y + r * H8 + c);
    acc[0] = fmaf(wj, bf16_lo(v.x), acc[0]);
    acc[1] = fmaf(wj, bf16_hi(v.x), acc[1]);
    acc[2] = fmaf(wj, bf16_lo(v.y), acc[2]);
    acc[3] = fmaf(wj, bf16_hi(v.y), acc[3]);
    acc[4] = fmaf(wj, bf16_lo(v.z), acc[4]);
    acc[5] = fmaf(wj, bf16_hi(v.z), acc[5]);
    acc[6] = fmaf(wj, bf16_lo(v.w), acc[6]);
    acc[7] = fmaf(wj, bf16_hi(v.w), acc[7]);
  }
  out[i] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                      pack_bf16x2(acc[6], acc[7]));
}

int sm_count_glue() { return current_sm_count(); }

template <int kEPL>
cudaError_t launch_route_k(const void* logits, bool bf16, int64_t T, int E, int k, bool renorm, int32_t* ids,
                           float* wts, cudaStream_t s) {
  const int64_t want = (T + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sm_count_glue()) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  route_kernel<kEPL><<<grid, 256, 0, s>>>(logits, bf16, T, E, k, renorm, ids, wts);
  return cudaGetLastError();
}

}  // namespace

size_t moe_route_workspace_bytes(int64_t T, int32_t E) {
  const int64_t ntiles = (T + kTile - 1) / kTile;
  return static_cast<size_t>(ntiles) * static_cast<size_t>(E) * sizeof(int32_t);
}

cudaError_t launch_moe_route(const void* logits, bool bf16, int64_t T, int32_t E, int32_t k, bool renorm,
                             int32_t* ids, float* wts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                             void* workspace, cudaStream_t s) {
  cudaError_t e;
  if (E <= 32)
    e = launch_route_k<1>(logits, bf16, T, E, k, renorm, ids, wts, s);
  else if (E <= 64)
    e = launch_route_k<2>(logits, bf16, T, E, k, renorm, ids, wts, s);
  else if (E <= 128)
    e = launch_route_k<4>(logits, bf16, T, E, k, renorm, ids, wts, s);
  else if (E <= 256)
    e = launch_route_k<8>(logits, bf16, T, E, k, renorm, ids, wts, s);
  else if (E <= 512)
    e = launch_route_k<16>(logits, bf16, T, E, k, renorm, ids, wts, s);
  else
    e = launch_route_k<32>(logits, bf16, T, E, k, renorm, ids, wts, s);
  if (e != cudaSuccess) return e;
  const int ntiles = static_cast<int>((T + kTile - 1) / kTile);
  int32_t* tile_rows = static_cast<int32_t*>(workspace);
  const size_t smem_count = static_cast<size_t>(kTileWarps) * E * sizeof(uint32_t);
  const size_t smem_place = 2 * smem_count;
  e = cudaFuncSetAttribute(tile_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_count));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tile_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_place));
  if (e != cudaSuccess) return e;
  tile_kernel<false><<<ntiles, kTile, smem_count, s>>>(ids, T, k, E, tile_rows, nullptr, nullptr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scan_kernel<<<1, kScanThreads, 0, s>>>(tile_rows, ntiles, E, offsets);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tile_kernel<true><<<ntiles, kTile, smem_place, s>>>(ids, T, k, E, tile_rows, row_token, row_of);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_quant(const void* h, int64_t R, int64_t I, void* q, float* scale, void* act,
                                  cudaStream_t s) {
  const int I8 = static_cast<int>(I / 8);
  if (R == 0 || I8 == 0) return cudaSuccess;
  auto hp = static_cast<const uint4*>(h);
  auto qp = static_cast<uint2*>(q);
  auto ap = static_cast<uint4*>(act);
  // one warp per row for many short rows, one CTA per row otherwise (the same
  // trade as the per-token quantizer's)
  const int need = (I8 + 31) / 32;
  if (need <= 8 && R * I8 >= (int64_t{1} << 19)) {
    const dim3 grid(static_cast<unsigned>((R + kActRowsPerCta - 1) / kActRowsPerCta));
    constexpr int kT = 32 * kActRowsPerCta;
    switch (need) {
      case 1: silu_mul_quant_warp<1><<<grid, kT, 0, s>>>(hp, R, I8, qp, scale, ap); break;
      case 2: silu_mul_quant_warp<2><<<grid, kT, 0, s>>>(hp, R, I8, qp, scale, ap); break;
      case 3: silu_mul_quant_warp<3><<<grid, kT, 0, s>>>(hp, R, I8, qp, scale, ap); break;
      case 4: silu_mul_quant_warp<4><<<grid, kT, 0, s>>>(hp, R, I8, qp, scale, ap); break;
      case 5: case 6: silu_mul_quant_warp<6><<<grid, kT, 0, s>>>(hp, R, I8, qp, scale, ap); break;
      default: silu_mul_quant_warp<8><<<grid, kT, 0, s>>>(hp, R, I8, qp, scale, ap); break;
    }
    return cudaGetLastError();
  }
  int threads = ((I8 + 31) / 32) * 32;
  if (threads > kActThreads) threads = kActThreads;
  const int nch = (I8 + threads - 1) / threads;
  const dim3 grid(static_cast<unsigned>(R));
  switch (nch) {
    case 1: silu_mul_quant_kernel<1><<<grid, threads, 0, s>>>(hp, I8, qp, scale, ap); break;
    case 2: silu_mul_quant_kernel<2><<<grid, threads, 0, s>>>(hp, I8, qp, scale, ap); break;
    case 3: silu_mul_quant_kernel<3><<<grid, threads, 0, s>>>(hp, I8, qp, scale, ap); break;
    case 4: silu_mul_quant_kernel<4><<<grid, threads, 0, s>>>(hp, I8, qp, scale, ap); break;
    default: silu_mul_quant_kernel<0><<<grid, threads, 0, s>>>(hp, I8, qp, scale, ap); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_moe_combine(const void* y, int64_t R, int64_t H, const float* w, const int32_t* row_of, int64_t T,
                               int32_t k, void* out, unsigned int* status, cudaStream_t s) {
  const int H8 = static_cast<int>(H / 8);
  const int64_t n = T * H8;
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  combine_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(y), R, H8, w, row_of, T, k,
                                        static_cast<uint4*>(out), status);
  return cudaGetLastError();
}

}  // namespace w4
