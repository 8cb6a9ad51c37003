// W4A16 skinny GEMM for decode: y[M,N] = x[M,K] . W^T with W as GPTQ int4.
//
// vLLM API docs, inc.schemes.inc_w4a8_linear (class docstring): the W4A16
// path reads the same GPTQ "NT" qweight [K/8, N] as the W4A8 path.
// vllm-omni quantization/cpu_int4.py (module docstring): decode is a bandwidth
// problem -- the whole weight is read for one token, so bits per weight set
// the token rate -- and the weight is w = (q - 8) * scale + zero.
//
// Design (GB300):
//  * Persistent CTAs, at most one per SM. The output columns are cut into
//    strips of 32; a CTA owns whole strips across all of K, dealt round-robin,
//    so there is no cross-CTA reduction and the work per SM is within one
//    strip of even.
//  * One producer thread streams each strip as 16 KB TMA tiles (32 columns x
//    1024 k, 128-byte swizzle) through an up-to-8-deep shared-memory ring:
//    128 KB of weights in flight per SM, independent of registers. (Measured
//    on GB300: TMA streams at HBM rate from 16 KB tiles but only ~2.4 TB/s
//    from 8 KB and ~1.6 TB/s from 4 KB ones.)
//  * Programmatic dependent launch: the weights never depend on the previous
//    kernel, so the grid starts streaming them while the previous call on the
//    stream drains, and waits for it only before reading x and writing y.
//    A standalone 30 MB stream pays a ~4 us fixed cost per launch on GB300;
//    back-to-back decode calls hide most of it this way.
//  * Sixteen consumer warps, four per tile, each take 256 k of a tile, with
//    four independent MMA accumulator chains each. Swap-AB on the warp-level
//    tensor core (m16n8k16, fp16 in, fp32 accumulate): 16 output columns are
//    the MMA's rows, up to 8 tokens its columns.
//  * Nibbles enter the MMA with one AND per pair and no convert: a nibble in
//    bits 0-3 of an fp16 is the exact subnormal q * 2^-24, one in bits 4-7 is
//    16 q * 2^-24 (fp16 subnormal operands multiply exactly on the tensor
//    core). Nibbles i and i+4 of a word share one register. The activations
//    are staged once per CTA as fp16 2^e x, with 2^e a per-token power of two
//    that puts the token's largest |x| in [2^14, 2^15) so every 2^e x is an
//    exact fp16 (except ones below 2^-14 relative to that maximum, whose
//    rounding is far below the fp32 sums); the activations paired with the
//    16 q nibbles carry an extra 1/16.
//  * Per scale group the exact-product fp32 partial becomes
//    sum x (q - 8) = 2^24 acc - 8 sum(x), folded as
//    tot += s (2^24 acc - 8 sum x) + z sum x, with the token sums over 64-k
//    blocks computed once; the result is scaled back by 2^-e.
//  * The k order inside each 32-wide step is permuted consistently for both
//    operands; the word-row order (2c + step parity) makes the 16-byte
//    shared loads of a quarter-warp land in 8 distinct swizzled chunks.
//  * Partials of a strip are reduced across the consumer warps in shared
//    memory in a fixed order; the bias is added and y written once in bf16.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace w4 {
namespace {

constexpr int kStrip = 32;          // output columns per strip
constexpr int kStageRows = 128;     // word rows per stage (1024 k)
constexpr int kStageK = kStageRows * 8;
constexpr int kStageBytes = kStrip * kStageRows * 4;   // 16 KB
constexpr int kRingMax = 8;         // up to 128 KB of weights in flight
constexpr int kConsumers = 16;
constexpr int kPerStage = 4;        // consumer warps per stage, 32 word rows (256 k) each
constexpr int kQuarterRows = kStageRows / kPerStage;
constexpr int kProducerWarp = kConsumers;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kTok = 8;             // tokens per MMA column block
constexpr uint64_t kWaitNs = 2000000000ull;

struct Params {
  CUtensorMap tm_w;      // GPTQ words [K/8, N], box 32 x 128, 128-byte swizzle
  const uint16_t* x;     // bf16 [M, K]
  const uint16_t* sc;    // fp16 or bf16 [G, N]
  const uint16_t* zr;    // bf16 [G, N] or null
  const uint16_t* bias;  // bf16 [N] or null
  uint16_t* y;           // bf16 [M, N]
  int M, N, K, group;    // M <= 8 here
  int strips, stages;    // per strip: stages = ceil(K / 1024)
  int xstride;           // shared-memory row stride of x, in fp16 elements
  int ring;              // stages in the ring (<= kRingMax)
  unsigned int* status;
};

W4_DEV void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                    uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool kScaleBf16>
W4_DEV float scale_at(uint32_t bits16) {
  return kScaleBf16 ? __uint_as_float(bits16 << 16) : half_bits_to_f32(bits16);
}

W4_DEV uint2 ld4x16(const uint16_t* p, bool in) { return in ? ld_nc_v2(p) : make_uint2(0, 0); }

W4_DEV uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Shared-memory carve-up (byte offsets from the 1024-aligned base).
struct Layout {
  int red, bars, ex, xsum, xs, total;
  __host__ __device__ Layout(int nb64, int xchunks, int rows, int ring) {
    red = ring * kStageBytes;
    bars = red + 2 * kConsumers * kStrip * rows * 4;   // [2][kConsumers][rows * kStrip]
    ex = bars + 256;                      // 2 * kRingMax + 4 mbarriers + the abort flag
    xsum = ex + 2 * kTok * 4;             // per token: 2^e and 2^-e
    xs = (xsum + rows * nb64 * 4 + 15) & ~15;
    total = xs + rows * xchunks * 16;
  }
};

template <bool kScaleBf16, bool kZero, bool kBias>
__global__ void __launch_bounds__(kThreads, 1) w4a16_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  const int R = p.ring;
  const int nb64 = S * (kStageK / 64);       // 64-wide k blocks (padded to whole stages)
  const int xch = p.xstride / 8;             // 16-byte chunks per token row
  const Layout L(nb64, xch, p.M, R);
  const int red_n = p.M * kStrip;            // partial outputs per warp
  uint8_t* ring = smem;                                      // R x 16 KB, 1024-aligned
  float* red = reinterpret_cast<float*>(smem + L.red);       // [2][kConsumers][red_n]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kRingMax;
  uint64_t* red_full = empty + kRingMax;
  uint64_t* red_empty = red_full + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red_empty + 2);
  float* ex = reinterpret_cast<float*>(smem + L.ex);         // [kTok] 2^e, then [kTok] 2^-e
  float* xsum = reinterpret_cast<float*>(smem + L.xsum);     // [M][nb64]: sum of 2^e x over 64-k blocks
  uint4* xs = reinterpret_cast<uint4*>(smem + L.xs);         // [M][xch]: 2^e x as fp16, permuted

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // consumer warp w works on word rows [32 (w % 4), +32) of stages w / 4, w / 4 + 4, ...
  const int groups = kConsumers / kPerStage;
  const int act = (S < groups ? S : groups) * kPerStage;   // consumer warps with work in every strip
  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPerStage);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&red_full[i], act);
      mbar_init(&red_empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int my_strips = p.strips > (int)blockIdx.x ? (p.strips - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  // the next call on the stream may start now: its weight stream does not
  // depend on this call (it waits for this grid before touching x and y)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kProducerWarp) {
    // ---- stream this CTA's strips, stage by stage, through the ring; the
    // weights never depend on the previous kernel, so this starts at once ----
    if (lane == 0) {
      tc::prefetch_tmap(&p.tm_w);
      const int total = my_strips * S;
      for (int i = 0; i < total; ++i) {
        const int slot = i % R;
        if (!tc::wait(&empty[slot], ((i / R) & 1) ^ 1, abort_flag, p.status, kWaitNs)) break;
        const int strip = blockIdx.x + (i / S) * gridDim.x, st = i % S;
        mbar_arrive_expect_tx(&full[slot], kStageBytes);
        tc::tma_load_2d(ring + slot * kStageBytes, &p.tm_w, &full[slot], strip * kStrip, st * kStageRows);
      }
    }
  } else {
    const int M = p.M, K = p.K, N = p.N;
    // x (and y) may belong to the previous kernel on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // ---- prologue 1: per-token power-of-two scale 2^e with amax * 2^e in [2^14, 2^15),
    // so every 2^e x (and 2^e x / 16) below is an exact fp16 except negligibly small ones ----
    if (warp < M) {
      float a = 0.f;
      for (int k8 = lane * 8; k8 < K; k8 += 256) {
        const uint4 v = ld_nc_v4(p.x + (size_t)warp * K + k8);
        a = fmaxf(a, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))), fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
        a = fmaxf(a, fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))), fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      if (lane == 0) {
        int e = 0;
        if (a > 0.f) {
          int E;
          frexpf(a, &E);               // a = f * 2^E, f in [0.5, 1)
          e = min(max(15 - E, -100), 100);
        }
        ex[warp] = __int_as_float((e + 127) << 23);          // 2^e, exactly
        ex[kTok + warp] = __int_as_float((127 - e) << 23);   // 2^-e
      }
    }
    asm volatile("bar.sync 1, %0;" :: "n"(kConsumers * 32) : "memory");
    // ---- prologue 2: tokens to shared memory as fp16 2^e x, each 8-chunk in the order
    // (x0,x4) (x1/16,x5/16) (x2,x6) (x3/16,x7/16) that matches the nibble pairs; zero past K ----
    for (int i = threadIdx.x; i < M * xch; i += kConsumers * 32) {
      const int m = i / xch, k8 = (i % xch) * 8;
      uint4 o = make_uint4(0, 0, 0, 0);
      if (k8 < K) {
        const uint4 v = ld_nc_v4(p.x + (size_t)m * K + k8);
        const float sc = ex[m], sc16 = sc * 0.0625f;
        o.x = pack_f16x2(bf16_lo(v.x) * sc, bf16_lo(v.z) * sc);       // (x0, x4)
        o.y = pack_f16x2(bf16_hi(v.x) * sc16, bf16_hi(v.z) * sc16);   // (x1, x5) / 16
        o.z = pack_f16x2(bf16_lo(v.y) * sc, bf16_lo(v.w) * sc);       // (x2, x6)
        o.w = pack_f16x2(bf16_hi(v.y) * sc16, bf16_hi(v.w) * sc16);   // (x3, x7) / 16
      }
      xs[i] = o;
    }
    // ---- prologue 3: sums of 2^e x over 64-k blocks (for the -8 offset and the zeros) ----
    for (int i = threadIdx.x; i < M * nb64; i += kConsumers * 32) {
      const int m = i / nb64, k0 = (i % nb64) * 64;
      float sum = 0.f;
      for (int k8 = k0; k8 < k0 + 64 && k8 < K; k8 += 8) {
        const uint4 v = ld_nc_v4(p.x + (size_t)m * K + k8);
        sum += (bf16_lo(v.x) + bf16_hi(v.x)) + (bf16_lo(v.y) + bf16_hi(v.y)) + (bf16_lo(v.z) + bf16_hi(v.z)) +
               (bf16_lo(v.w) + bf16_hi(v.w));
      }
      xsum[i] = sum * ex[m];
    }
    asm volatile("bar.sync 1, %0;" :: "n"(kConsumers * 32) : "memory");

    const int r = lane >> 2, c = lane & 3;
    const int group = p.group;
    for (int su = 0; su < my_strips && !*abort_flag; ++su) {
      const int strip = blockIdx.x + su * gridDim.x;
      const int n0 = strip * kStrip + 4 * r;   // this lane's 4 columns n0..n0+3
      const bool n_in = n0 < N;
      float tot[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) tot[j][e] = 0.f;
      bool ok = true;
      // this warp's quarter of stages warp / 4, warp / 4 + groups, ... of the strip
      for (int st = warp / kPerStage; st < S; st += groups) {
        const int i = su * S + st, slot = i % R;
        if (!tc::wait(&full[slot], (i / R) & 1, abort_flag, p.status, kWaitNs, 500)) {
          ok = false;
          break;
        }
        const uint8_t* tile = ring + slot * kStageBytes + (warp % kPerStage) * kQuarterRows * 128;
        const int kst = st * kStageK + (warp % kPerStage) * kQuarterRows * 8;
        const int nsteps = max(0, min(kQuarterRows / 4, (K - kst) / 32));
        const uint4* xrow = xs + r * xch + kst / 8;
        // segments: the part of one scale group inside this quarter (even step counts)
        for (int t0 = 0; t0 < nsteps;) {
          const int g = (kst + t0 * 32) / group;
          const int t1 = min(nsteps, ((g + 1) * group - kst) / 32);
          float acc[4][4];   // [tile * 2 + k half]: four independent MMA chains
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
          const uint2 sv = ld4x16(p.sc + (size_t)g * N + n0, n_in);
          uint2 zv = make_uint2(0, 0);
          if (kZero) zv = ld4x16(p.zr + (size_t)g * N + n0, n_in);
          for (int t = t0; t < t1; ++t) {
            const int kb = 8 * (t >> 1) + 2 * c + (t & 1);      // word row inside the quarter
            const uint4 w = *reinterpret_cast<const uint4*>(tile + kb * 128 + ((r ^ (kb & 7)) << 4));
            const uint4 xv = (r < M) ? xrow[kb] : make_uint4(0, 0, 0, 0);
            // nibble pairs as fp16 subnormals: (i, i+4) at bits 0-3 -> q 2^-24,
            // at bits 4-7 -> 16 q 2^-24 (its activations carry the 1/16)
            const uint32_t xh = w.x >> 8, yh = w.y >> 8, zh = w.z >> 8, wh = w.w >> 8;
            // tile 0: rows r <-> n0, r+8 <-> n0+1; tile 1: rows r <-> n0+2, r+8 <-> n0+3
            mma_f16(acc[0], w.x & 0x000F000Fu, w.y & 0x000F000Fu, w.x & 0x00F000F0u, w.y & 0x00F000F0u, xv.x, xv.y);
            mma_f16(acc[1], xh & 0x000F000Fu, yh & 0x000F000Fu, xh & 0x00F000F0u, yh & 0x00F000F0u, xv.z, xv.w);
            mma_f16(acc[2], w.z & 0x000F000Fu, w.w & 0x000F000Fu, w.z & 0x00F000F0u, w.w & 0x00F000F0u, xv.x, xv.y);
            mma_f16(acc[3], zh & 0x000F000Fu, wh & 0x000F000Fu, zh & 0x00F000F0u, wh & 0x00F000F0u, xv.z, xv.w);
          }
          // fold: sum_k x (q - 8) = 2^24 acc - 8 sum(x) (all in units of 2^e x);
          // tot += s * that + z * sum(x)
          float x0 = 0.f, x1 = 0.f;
          for (int b = (kst + t0 * 32) / 64; b < (kst + t1 * 32) / 64; ++b) {
            if (2 * c < M) x0 += xsum[(2 * c) * nb64 + b];
            if (2 * c + 1 < M) x1 += xsum[(2 * c + 1) * nb64 + b];
          }
          const uint32_t sb[4] = {sv.x & 0xFFFFu, sv.x >> 16, sv.y & 0xFFFFu, sv.y >> 16};
          const uint32_t zb[4] = {zv.x & 0xFFFFu, zv.x >> 16, zv.y & 0xFFFFu, zv.y >> 16};
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float s_lo = scale_at<kScaleBf16>(sb[2 * j]), s_hi = scale_at<kScaleBf16>(sb[2 * j + 1]);
            const float z_lo = kZero ? __uint_as_float(zb[2 * j] << 16) : 0.f;
            const float z_hi = kZero ? __uint_as_float(zb[2 * j + 1] << 16) : 0.f;
            const float a_lo = s_lo * 16777216.f, a_hi = s_hi * 16777216.f;   // s * 2^24
            const float b_lo = fmaf(-8.f, s_lo, z_lo), b_hi = fmaf(-8.f, s_hi, z_hi);
            const float* p0 = acc[2 * j];
            const float* p1 = acc[2 * j + 1];
            tot[j][0] = fmaf(a_lo, p0[0] + p1[0], fmaf(b_lo, x0, tot[j][0]));
            tot[j][1] = fmaf(a_lo, p0[1] + p1[1], fmaf(b_lo, x1, tot[j][1]));
            tot[j][2] = fmaf(a_hi, p0[2] + p1[2], fmaf(b_hi, x0, tot[j][2]));
            tot[j][3] = fmaf(a_hi, p0[3] + p1[3], fmaf(b_hi, x1, tot[j][3]));
          }
          t0 = t1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);   // this quarter of the tile consumed
      }
      if (!ok || warp >= act) continue;
      // hand the partial to the reduction; warp 0 finishes the strip
      const int rb = su & 1;
      if (!tc::wait(&red_empty[rb], ((su >> 1) & 1) ^ 1, abort_flag, p.status, kWaitNs)) break;
      float* dst = red + (rb * kConsumers + warp) * red_n;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int nl = 4 * r + 2 * j;
        if (2 * c < M) {
          dst[(2 * c) * kStrip + nl] = tot[j][0];
          dst[(2 * c) * kStrip + nl + 1] = tot[j][2];
        }
        if (2 * c + 1 < M) {
          dst[(2 * c + 1) * kStrip + nl] = tot[j][1];
          dst[(2 * c + 1) * kStrip + nl + 1] = tot[j][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[rb]);
      if (warp == 0) {
        if (!tc::wait(&red_full[rb], (su >> 1) & 1, abort_flag, p.status, kWaitNs)) break;
        const float* src = red + rb * kConsumers * red_n;
        for (int o = lane; o < red_n; o += 32) {
          const int m = o / kStrip, n = strip * kStrip + o % kStrip;
          float v = 0.f;
          for (int w = 0; w < act; ++w) v += src[w * red_n + o];   // fixed order
          if (n < N) {
            v *= ex[kTok + m];                                     // undo 2^e (exact)
            if (kBias) v += __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16);
            p.y[(size_t)m * N + n] = static_cast<uint16_t>(f32_to_bf16_bits(v));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[rb]);
      }
    }
  }
  if (*abort_flag) {
    // let copies already issued land before the shared memory goes away
    const uint64_t t0 = tc::globaltimer_ns();
    while (tc::globaltimer_ns() - t0 < 1000000ull) {
    }
  }
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

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encode_weights(CUtensorMap* m, const void* qweight, int64_t N, int64_t K) {
  static EncodeTiled fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || f == nullptr) return cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiled>(f);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)(K / 8)};
  const cuuint64_t strides[1] = {(cuuint64_t)N * 4};
  const cuuint32_t box[2] = {kStrip, kStageRows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void*>(qweight), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int x_stride(int K) {
  const int stages = (K + kStageK - 1) / kStageK;
  return stages * kStageK + 8;   // +16 bytes: token rows start in different banks
}

size_t smem_bytes(int K, int rows, int ring) {
  const int stages = (K + kStageK - 1) / kStageK;
  return 1024 + static_cast<size_t>(Layout(stages * (kStageK / 64), x_stride(K) / 8, rows, ring).total);
}
constexpr size_t kSmemMax = 227 * 1024;

template <bool kScaleBf16, bool kZero, bool kBias>
cudaError_t launch_t(const Params& p, int grid, size_t smem, cudaStream_t s) {
  auto k = w4a16_kernel<kScaleBf16, kZero, kBias>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: this grid may start while the previous
  // kernel on the stream finishes; it waits for it before reading x
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace

size_t w4a16_smem_bytes(int64_t K, int32_t group) {
  (void)group;
  return smem_bytes(static_cast<int>(K), 1, 2);
}

cudaError_t launch_w4a16(const W4A16Args& a, cudaStream_t s) {
  Params p;
  memset(&p, 0, sizeof(p));
  cudaError_t e = encode_weights(&p.tm_w, a.qweight, a.N, a.K);
  if (e != cudaSuccess) return e;
  p.sc = static_cast<const uint16_t*>(a.w_scale);
  p.zr = static_cast<const uint16_t*>(a.zeros);
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.group = a.group;
  p.strips = (p.N + kStrip - 1) / kStrip;
  p.stages = (p.K + kStageK - 1) / kStageK;
  p.xstride = x_stride(p.K);
  p.status = a.status;
  // tokens in blocks of up to 8 beside a ring of at least 4 stages (deeper
  // when it fits); each block is one pass over the weights
  int block = kTok;
  while (block > 1 && smem_bytes(p.K, block, 4) > kSmemMax) --block;
  if (smem_bytes(p.K, block, 2) > kSmemMax) return cudaErrorInvalidValue;
  const int grid = p.strips < sm_count() ? p.strips : sm_count();
  const bool bf = a.scale_bf16, z = a.zeros != nullptr, b = a.bias != nullptr;
  for (int64_t m0 = 0; m0 < a.M; m0 += block) {
    p.x = static_cast<const uint16_t*>(a.x) + m0 * a.K;
    p.y = static_cast<uint16_t*>(a.y) + m0 * a.N;
    p.M = static_cast<int>(a.M - m0 < block ? a.M - m0 : block);
    p.ring = kRingMax;
    while (p.ring > 2 && smem_bytes(p.K, p.M, p.ring) > kSmemMax) --p.ring;
    const size_t smem = smem_bytes(p.K, p.M, p.ring);
    if (bf) {
      if (z) e = b ? launch_t<true, true, true>(p, grid, smem, s) : launch_t<true, true, false>(p, grid, smem, s);
      else e = b ? launch_t<true, false, true>(p, grid, smem, s) : launch_t<true, false, false>(p, grid, smem, s);
    } else {
      if (z) e = b ? launch_t<false, true, true>(p, grid, smem, s) : launch_t<false, true, false>(p, grid, smem, s);
      else e = b ? launch_t<false, false, true>(p, grid, smem, s) : launch_t<false, false, false>(p, grid, smem, s);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w4
