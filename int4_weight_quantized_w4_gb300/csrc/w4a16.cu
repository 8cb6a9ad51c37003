// W4A16 skinny GEMM for decode: y[M,N] = x[M,K] . W^T with W as GPTQ int4.
//
// vLLM API docs, inc.schemes.inc_w4a8_linear (class docstring): the W4A16
// path reads the same GPTQ "NT" qweight [K/8, N] as the W4A8 path.
// vllm-omni quantization/cpu_int4.py (module docstring): decode is a bandwidth
// problem -- the whole weight is read for one token, so bits per weight set
// the token rate -- and the weight is w = (q - 8) * scale + zero.
//
// Design (GB300):
//  * Two kernels per call, both with programmatic dependent launch. A one-warp
//    prefetch grid starts beside the previous call's GEMV (it needs no shared
//    memory), pulls this call's weights, scales and zeros into L2 and exits.
//    The GEMV grid that follows therefore streams its weights from L2 while
//    HBM already serves the next call's prefetch: back-to-back decode calls
//    keep HBM busy across the call boundary, and the conversion work per
//    weight (~1.8 us a call at 4096 x 14336 on 152 SMs) hides under it.
//    The GEMV's griddepcontrol.wait covers every prerequisite grid still in
//    flight, the previous call's GEMV included, so the prefetch grid itself
//    never waits (measured on GB300: one dependency hop of ~0.74 us instead
//    of two, ~1.68 us).
//  * GEMV: persistent CTAs, one per SM. The output columns are cut into
//    strips of 32; a CTA owns whole strips across all of K, dealt
//    round-robin, so there is no cross-CTA reduction.
//  * Each strip moves as 16 KB TMA tiles (32 columns x 1024 k, 128-byte
//    swizzle) with the scale (and zero) rows the tile's k range meets, all on
//    one mbarrier, through a ring of up to 8 stages. (A plain global load from
//    an SM with that much streaming in flight waits ~2 us on GB300, so the
//    consumer loop touches no global memory.) There is no producer warp: warp
//    w issues stage w of the initial fill, and the warp that finishes the last
//    unit of a stage refills its slot with the stage R later (a per-slot
//    shared counter elects it). Sixteen warps, four per SM sub-partition, get
//    120 registers each.
//  * The warps take 256-k units of a strip (four per stage): warp w gets
//    units w, w + 16, ..., so the four units of stage i always go to warp
//    group i % 4. The ring depth is a multiple of 4, so each warp sees every
//    phase of the slots it reads and the parity waits stay exact.
//  * Swap-AB on the warp-level tensor core (m16n8k16, fp16 in, fp32
//    accumulate): 16 output columns are the MMA rows, up to 8 tokens its
//    columns. Nibbles enter the MMA with one AND per pair and no convert: a
//    nibble in bits 0-3 of an fp16 is the exact subnormal q 2^-24, one in
//    bits 4-7 is 16 q 2^-24 (fp16 subnormal operands multiply exactly on the
//    tensor core, at full rate). Nibbles i and i+4 of a word share one
//    register. Each 256-k segment of a token's x is staged as fp16 2^e x, with
//    2^e a power of two per (token, segment) that puts the segment's largest
//    |x| in [2^14, 2^15), so every 2^e x is an exact fp16 (except ones below
//    2^-24 of that maximum, whose rounding is far below the fp32 sums); the
//    ones paired with the 16 q nibbles carry an extra 1/16.
//  * x segments have owner warps (segment u: warp u % 16): the owner
//    bulk-copies its segments right after the dependency wait, converts them
//    in place and signals a per-segment mbarrier, so no block-wide barrier
//    sits between the wait and the first MMA. At the common K = 4096 each
//    warp only ever reads its own segment.
//  * Per scale group the partial is folded as
//    tot += s 2^-e acc + (z - 8 s) X, X = 2^-24 sum x over the group's k
//    (since sum x (q - 8) = 2^24 2^-e acc - 8 sum x); tot is scaled by 2^24
//    at the end (exact). Fold points are compile-time for groups of 64, 128
//    and multiples of 256. For up to 4 tokens and groups of 128 the unit's
//    two groups go to two MMA columns per token (unused columns read a zero
//    row), so they accumulate side by side and the unit folds once (decode
//    chains measured 3-4% faster on GB300 at one token and 2% at four,
//    outputs bit-identical).
//  * The k order inside each 32-wide step is permuted consistently for both
//    operands; word rows 2c + (step parity) make the 16-byte shared loads of
//    a quarter-warp land in 8 distinct swizzled chunks.
//  * Each warp keeps its strip partial in registers and stores it once per
//    strip; after the last unit the block sums the partials in a fixed order,
//    adds the bias and writes y once in bf16.
//  * From page-locked host buffers (w4a16_gemm_host) the prefetch grid copies
//    x in and the GEMV writes y out as well, so such a call launches the same
//    two grids as a device call and chains with its neighbours the same way.
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
constexpr int kRingMax = 16;      // stage barriers: a ring of 4 or 8, or up to 16 resident stages
constexpr int kFirstFill = 8;     // stages of a refilled ring issued when the CTA starts
constexpr int kConsumers = 16;
constexpr int kUnitRows = 32;       // word rows per consumer unit (256 k, 8 steps)
constexpr int kUnitK = kUnitRows * 8;
constexpr int kUnitsPerStage = kStageRows / kUnitRows;
constexpr int kSegChunks = kUnitK / 8;   // 16-byte x chunks per 256-k segment (one per lane)
constexpr int kThreads = kConsumers * 32;
constexpr int kFirstRound = kConsumers / kUnitsPerStage;   // stages the first round of units reads
constexpr int kTok = 8;             // tokens per MMA column block
constexpr uint64_t kWaitNs = 2000000000ull;

struct Params {
  CUtensorMap tm_w;      // GPTQ words [K/8, N], box 32 x 128, 128-byte swizzle
  CUtensorMap tm_s;      // scales, fp16 or bf16 [G, N], box 32 x gh
  CUtensorMap tm_z;      // zeros, bf16 [G, N], box 32 x gh (when present)
  const uint16_t* x;     // bf16 [M, K]
  const uint16_t* bias;  // bf16 [N] or null
  uint16_t* y;           // bf16 [M, N]
  uint16_t* y_host;      // page-locked host copy of y (host entry point), or null
  int M, N, K, group;    // M <= 8 here
  int strips, stages;    // per strip: stages = ceil(K / 1024)
  int xstride;           // shared-memory row stride of x, in fp16 elements
  int ring;              // stage index -> slot i & (ring - 1): 4 or 8, or 16 when resident
  int slots;             // stage slots in shared memory (ring, or every stage of a CTA when resident)
  int resident;          // every stage of a CTA has its own slot: no slot is ever refilled
  int gh;                // scale rows per stage tile: most groups one stage's k range meets
  int zoff;              // byte offset of the zero rows inside a slot's scale area
  int scb;               // bytes of one slot's scale area (scales, then zeros)
  int pstrips;           // most strips one CTA owns
  int ring_shift;        // log2(ring)
  int group_shift;       // log2(group) when the group is a power of two, else -1
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

// One m16n8k16 MMA that starts from zero instead of accumulating.
W4_DEV void mma_f16_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

W4_DEV uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Shared-memory carve-up (byte offsets from the 1024-aligned base). The strip
// partials take [pstrips][kConsumers][rows][kStrip] floats, or with the
// partials in tensor memory only their per-quadrant sums, [pstrips][4][32
// lanes][8] floats.
struct Layout {
  int scl, red, bars, xrdy, exs, xsum, zro, xs, total;
  __host__ __device__ Layout(int nseg, int xchunks, int rows, int ring, int scb, int pstrips, bool tmem_red) {
    scl = ring * kStageBytes;             // ring x scb: scale (and zero) rows per slot
    red = scl + ring * scb;               // strip partials, or their quadrant sums
    bars = red + (tmem_red ? pstrips * 4 * 32 * 8 * 4 : pstrips * kConsumers * rows * kStrip * 4);
    // bars: full, per-warp x, slot counters, abort flag, the TMEM base
    xrdy = bars + 512;                    // [nseg] mbarriers: x segment converted
    exs = xrdy + nseg * 8;                // [nseg][kTok] 2^-e per segment and token
    xsum = exs + nseg * kTok * 4;         // [nseg * 4][kTok] 2^-24 sums of x over 64-k blocks
    zro = (xsum + nseg * 4 * kTok * 4 + 15) & ~15;   // 32 x 16 zero bytes (one token, one group of columns)
    xs = zro + 512;
    total = xs + rows * xchunks * 16;     // [rows][xchunks] x, converted in place
  }
};

// Pulls [base, base + bytes) into L2, this block's share of it, 16 KB at a
// time (base 16-byte aligned, bytes a multiple of 16).
W4_DEV void prefetch_share(const uint8_t* base, size_t bytes) {
  if (base == nullptr || bytes == 0) return;
  const size_t share = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
  const size_t lo = blockIdx.x * share;
  const size_t hi = lo + share < bytes ? lo + share : bytes;
  for (size_t o = lo; o < hi; o += 16384) {
    const uint32_t n = static_cast<uint32_t>(hi - o < 16384 ? hi - o : 16384);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(base + o), "r"(n) : "memory");
  }
}

// The L2 prefetch grid: one warp per SM, no shared memory, so it runs beside
// the previous call's GEMV. It lets its dependent (this call's GEMV) launch at
// once and touches nothing but L2, so it needs no dependency wait of its own:
// the GEMV's griddepcontrol.wait covers every prerequisite grid in flight.
// For the host entry point it also copies x (x16 16-byte words) from
// page-locked host memory into x: each thread reads its first word before
// the dependency wait (nothing before writes x_host) and writes after it (the
// kernels before may still read x). As a kernel, not a copy-engine job, the
// copy keeps consecutive calls chained (measured on GB300: a decode call from
// host buffers took ~24 us of stream time with cudaMemcpyAsync copies).
__global__ void __launch_bounds__(32) w4a16_prefetch_kernel(const uint8_t* w, size_t wb, const uint8_t* s,
                                                            size_t sb, const uint8_t* z, size_t zb,
                                                            const uint4* __restrict__ xh, uint4* __restrict__ x,
                                                            size_t x16) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    prefetch_share(w, wb);
    prefetch_share(s, sb);
    prefetch_share(z, zb);
  }
  if (x16 == 0) return;
  const size_t stride = static_cast<size_t>(gridDim.x) * 32;
  size_t i = static_cast<size_t>(blockIdx.x) * 32 + threadIdx.x;
  const uint4 first = i < x16 ? xh[i] : make_uint4(0, 0, 0, 0);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (i < x16) x[i] = first;
  for (i += stride; i < x16; i += stride) x[i] = xh[i];
}

// kSPF: steps (32 k each) per scale group inside a 256-k unit when the fold
// points are fixed -- 2 for group 64, 4 for group 128, 8 for groups that are
// multiples of 256 -- or 0 for any other group, whose fold points are found
// per unit.
// 120 registers a thread, not the 128 that 512 threads could have: a
// sub-partition then keeps room for the one-warp prefetch grid of the next
// call (4 x 32 x 120 + 768 <= 16384), which must run beside this grid.
// tot is set at every strip change before flush reads it; the compiler cannot
// see that through the lambda (a zero initializer measurably changes the
// register allocation of every instantiation, so the warning is silenced)
#pragma nv_diag_suppress 549
// kTmemRed: the warps' strip partials go to tensor memory instead of shared
// memory (at M = 5..8 the shared-memory partials would cost the ring half its
// depth); the block sums them per TMEM lane quadrant, then across quadrants.
template <bool kScaleBf16, bool kZero, int kSPF, bool kTmemRed, int kGC = 0>
__global__ void __maxnreg__(120) w4a16_kernel(const __grid_constant__ Params p) {
  // kGC (group columns, groups of 128): 1 for one token, 4 for two to four.
  // MMA column n holds token n / 2's sums over the unit's group n % 2, so the
  // unit folds once
  static_assert(kGC == 0 || (kSPF == 4 && !kTmemRed), "the group-column form folds two 128-k groups per unit");
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  const int R = p.ring;
  const int M = p.M;
  const int nseg = S * (kStageK / kUnitK);   // 256-k x segments (padded to whole stages)
  const int xch = p.xstride / 8;             // 16-byte chunks per token row
  const Layout L(nseg, xch, M, p.slots, p.scb, p.pstrips, kTmemRed);
  uint8_t* ring = smem;                                      // slots x 16 KB, 1024-aligned
  const uint8_t* scl = smem + L.scl;                         // slots x scb
  float* red = reinterpret_cast<float*>(smem + L.red);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* xbar = full + kRingMax;                          // [kConsumers] a warp's x copies landed
  unsigned int* done = reinterpret_cast<unsigned int*>(xbar + kConsumers);   // [kRingMax] units finished per slot
  volatile int* abort_flag = reinterpret_cast<volatile int*>(done + kRingMax);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.bars + 384);
  // TMEM columns: 8 per (local strip, warp / 4) in each lane quadrant
  uint32_t tmem_cols = 32;
  while (kTmemRed && tmem_cols < 32u * static_cast<uint32_t>(p.pstrips)) tmem_cols <<= 1;
  uint64_t* xrdy = reinterpret_cast<uint64_t*>(smem + L.xrdy);
  float* exs = reinterpret_cast<float*>(smem + L.exs);
  float* xsum = reinterpret_cast<float*>(smem + L.xsum);
  uint4* xs = reinterpret_cast<uint4*>(smem + L.xs);
  const uint4* zrow = reinterpret_cast<const uint4*>(smem + L.zro);
  if (kGC != 0 && threadIdx.x < 32) reinterpret_cast<uint4*>(smem + L.zro)[threadIdx.x] = make_uint4(0, 0, 0, 0);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      done[i] = 0u;
    }
    for (int i = 0; i < kConsumers; ++i) mbar_init(&xbar[i], 1);
    for (int i = 0; i < nseg; ++i) mbar_init(&xrdy[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (kTmemRed && warp == 0) tc::tmem_alloc(tmem_holder, tmem_cols);
  if (kTmemRed) tc::fence_before_sync();
  __syncthreads();
  if (kTmemRed) tc::fence_after_sync();

  const int my_strips = p.strips > (int)blockIdx.x ? (p.strips - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  // this warp's columns for local strip su, in its lane quadrant
  const uint32_t tmem = kTmemRed ? *tmem_holder : 0u;
  auto tcol = [&](int su) {
    return tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>((su * 4 + (warp >> 2)) * 8);
  };
  if (kTmemRed) {
    // zeros for the strips this warp contributes nothing to (fewer than 16
    // units a strip), written before any partial of the same columns
    const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    for (int su = 0; su < my_strips; ++su) tc::tmem_st8(tcol(su), zero);
    tc::tmem_wait_st();
  }

  // the next call on the stream may start now: its grids do not touch this
  // call's x or y before they wait for it
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int total = my_strips * S;            // stages this CTA streams
  const uint32_t tx = kStageBytes + (kZero ? 2 : 1) * p.gh * kStrip * 2;
  // stage i -> its ring slot (the weights never depend on the previous kernel)
  auto issue = [&](int i) {
    const int slot = i & (R - 1);
    const int col = (blockIdx.x + (i / S) * gridDim.x) * kStrip, st = i % S;
    const int gst = st * kStageK / p.group;   // first scale row the stage meets
    uint8_t* sdst = smem + L.scl + slot * p.scb;
    mbar_arrive_expect_tx(&full[slot], tx);
    tc::tma_load_2d(ring + slot * kStageBytes, &p.tm_w, &full[slot], col, st * kStageRows);
    tc::tma_load_2d(sdst, &p.tm_s, &full[slot], col, gst);
    if (kZero) tc::tma_load_2d(sdst + p.zoff, &p.tm_z, &full[slot], col, gst);
  };
  // initial fill: warp w issues stage w, so no one warp spends its start
  // issuing the whole ring (a TMA issue can stall while the copy engine is
  // busy). With resident stages only those the first round of units reads go
  // out when the CTA starts, and the rest after the x prologue, whose loads
  // would otherwise queue behind them. Measured on GB300, decode calls in a
  // chain: 8.6 -> 8.1 us a call. Fewer stages first, or the rest issued with
  // the x loads, measured slower, and so did the same split for a refilled
  // ring at M = 4 and 8.
  if (lane == 0 && warp < R && warp < (p.resident ? kFirstRound : kFirstFill) && warp < total) {
    tc::prefetch_tmap(&p.tm_w);
    tc::prefetch_tmap(&p.tm_s);
    if (kZero) tc::prefetch_tmap(&p.tm_z);
    issue(warp);
  }
  {
    const int K = p.K, group = p.group;
    // ---- prologue, per warp over the x segments it owns (u = warp, warp + 16,
    // ...): after the dependency wait each lane loads its 16 bytes of every
    // token row of the segment straight from global memory (a load through
    // L2, which sees what the previous kernel wrote; measured on GB300 it lands
    // ~1 us sooner than a bulk copy queued behind the weight tiles), finds each
    // token's largest exponent field E in the segment, which fixes 2^e,
    // e = 14 - (E - 127), and converts ----
    // x (and y) may belong to the previous kernel on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool x_ok = true;
    for (int u = warp; u < nseg && x_ok; u += kConsumers) {
      const int cc = u * kSegChunks + lane;
      uint4 xv8[kTok];   // every token's chunk in flight at once
#pragma unroll
      for (int m = 0; m < kTok; ++m)
        xv8[m] = (m < M && cc * 8 < K) ? ld_cg_v4(p.x + (size_t)m * K + cc * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int m = 0; m < kTok; ++m) {
        if (m >= M) break;
        const uint4 v = xv8[m];
        const uint32_t h = __vmaxu2(__vmaxu2(v.x & 0x7F807F80u, v.y & 0x7F807F80u),
                                    __vmaxu2(v.z & 0x7F807F80u, v.w & 0x7F807F80u));
        const uint32_t ef = __reduce_max_sync(0xffffffffu, max(h & 0xFFFFu, h >> 16));
        const int e = min(max(141 - static_cast<int>(ef >> 7), -120), 100);
        const float sc = __int_as_float((127 + e) << 23), sc16 = sc * 0.0625f;
        uint4 o;   // (x0,x4) (x1/16,x5/16) (x2,x6) (x3/16,x7/16): the nibble pair order
        o.x = pack_f16x2(bf16_lo(v.x) * sc, bf16_lo(v.z) * sc);
        o.y = pack_f16x2(bf16_hi(v.x) * sc16, bf16_hi(v.z) * sc16);
        o.z = pack_f16x2(bf16_lo(v.y) * sc, bf16_lo(v.w) * sc);
        o.w = pack_f16x2(bf16_hi(v.y) * sc16, bf16_hi(v.w) * sc16);
        xs[m * xch + cc] = o;
        // 2^-24 sums of x over 64-k blocks (8 neighbouring lanes)
        float sum = ((bf16_lo(v.x) + bf16_hi(v.x)) + (bf16_lo(v.y) + bf16_hi(v.y))) +
                    ((bf16_lo(v.z) + bf16_hi(v.z)) + (bf16_lo(v.w) + bf16_hi(v.w)));
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        if ((lane & 7) == 0) xsum[(u * 4 + lane / 8) * kTok + m] = sum * 5.9604644775390625e-8f;
        if (lane == 0) exs[u * kTok + m] = __int_as_float((127 - e) << 23);   // 2^-e, exactly
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xrdy[u]);   // releases this warp's writes of the segment
    }

    if (p.resident && lane == 0 && warp >= kFirstRound && warp < total) issue(warp);

    // ---- main loop over this warp's 256-k units ----
    const int r = lane >> 2, c = lane & 3;
    const int units = kUnitsPerStage * S;                // per strip
    const int total_units = x_ok ? my_strips * units : 0;
    // lane offsets of the two word rows a step reads (even / odd step), swizzled
    const int w_off_e = (2 * c) * 128 + ((r ^ (2 * c)) << 4);
    const int w_off_o = (2 * c + 1) * 128 + ((r ^ (2 * c + 1)) << 4);
    const uint4* xrow = xs + min(r, M - 1) * xch;        // tokens past M: any finite data, discarded
    float tot[2][4];
    int cur = -1;                                        // strip whose partial tot holds
    bool ok = true;
    auto flush = [&](int su) {
      if constexpr (kTmemRed) {
        const uint32_t v[8] = {__float_as_uint(tot[0][0]), __float_as_uint(tot[0][1]), __float_as_uint(tot[0][2]),
                               __float_as_uint(tot[0][3]), __float_as_uint(tot[1][0]), __float_as_uint(tot[1][1]),
                               __float_as_uint(tot[1][2]), __float_as_uint(tot[1][3])};
        tc::tmem_st8(tcol(su), v);
        return;
      }
      float* dst = red + (su * kConsumers + warp) * M * kStrip;
      if constexpr (kGC == 4) {   // lane (r, c) holds token c's two outputs of each tile
        if (c < M)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            dst[c * kStrip + 4 * r + 2 * j] = tot[j][0];
            dst[c * kStrip + 4 * r + 2 * j + 1] = tot[j][2];
          }
      } else {
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
      }
    };
    // unit v is unit u of strip su (v = su * units + u); kept incrementally
    int su = warp / units, u = warp % units;
    for (int v = warp; v < total_units; v += kConsumers, u += kConsumers) {
      while (u >= units) {
        u -= units;
        ++su;
      }
      const int st = u / kUnitsPerStage, qu = u % kUnitsPerStage;
      if (su != cur) {
        if (cur >= 0) flush(cur);
        cur = su;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) tot[j][e] = 0.f;
      }
      const int i = su * S + st, slot = i & (R - 1), phase = (i >> p.ring_shift) & 1;
      const int kunit = st * kStageK + qu * kUnitK;
      const int seg = u;                                   // kunit / 256
      const int nsteps = min(kUnitRows / 4, max(0, (K - kunit) / 32));   // even: K % 64 == 0
      if (!tc::wait(&xrdy[seg], 0, abort_flag, p.status, kWaitNs) ||
          !tc::wait(&full[slot], phase, abort_flag, p.status, kWaitNs, 500)) {
        ok = false;
        break;
      }
      if (nsteps > 0) {
        const uint8_t* wbase = ring + slot * kStageBytes + qu * (kUnitRows * 128);
        const uint8_t* we = wbase + w_off_e;
        const uint8_t* wo = wbase + w_off_o;
        const uint4* xe = xrow + kunit / 8 + 2 * c;
        // group columns: MMA column r takes token r / 2's x over the unit's
        // first 128-k group (r even) or its second (r odd), zeros elsewhere, so
        // both groups accumulate side by side and the unit folds once
        const uint4* xg = kGC == 4 ? xs + min(r >> 1, M - 1) * xch + kunit / 8 + 2 * c : xe;
        const uint4* xe0 = kGC == 1 ? (r != 0 ? zrow + 2 * c : xe)
                                    : ((r & 1) != 0 || (r >> 1) >= M ? zrow + 2 * c : xg);
        const uint4* xe1 = kGC == 1 ? (r != 1 ? zrow + 2 * c : xe)
                                    : ((r & 1) != 1 || (r >> 1) >= M ? zrow + 2 * c : xg);
        const int ct = kGC == 4 ? c : 0;   // the token whose sums this lane folds
        const float* xb = xsum + (kunit / 64) * kTok + 2 * c;
        const float2 f = *reinterpret_cast<const float2*>(exs + seg * kTok + 2 * c);   // 2^-e, tokens 2c, 2c+1
        // scale rows of the slot: this unit's first group is row kunit / group - gst
        const uint8_t* sbase = scl + slot * p.scb + 8 * r;
        const int row0 = kSPF == 2   ? 4 * qu
                         : kSPF == 4 ? 2 * qu
                         : p.group_shift >= 0 ? (kunit >> p.group_shift) - ((st * kStageK) >> p.group_shift)
                                              : kunit / group - st * kStageK / group;
        // steps that end a scale group (or the unit's k range) fold the partial
        uint32_t fold_mask = 0;
        if (kSPF == 0) {
          fold_mask = 1u << (nsteps - 1);
          for (int t = (group - kunit % group) / 32 - 1; t < nsteps - 1; t += group / 32) fold_mask |= 1u << t;
        }
        float acc[4][4];   // [tile * 2 + nibble half]: four independent MMA chains
        if (kSPF == 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
        }
        float X0 = 0.f, X1 = 0.f;
        int gseg = 0;
        // tot += s 2^-e acc + (z - 8 s) X for the scale group that just ended;
        // with fixed fold points the row is clamped into the slot's scale area
        // (past K it meets only zero products)
        auto fold = [&](int row) {
          const uint2 sv = *reinterpret_cast<const uint2*>(sbase + row * (kStrip * 2));
          const uint2 zv = kZero ? *reinterpret_cast<const uint2*>(sbase + p.zoff + row * (kStrip * 2))
                                 : make_uint2(0, 0);
          const uint32_t sb[4] = {sv.x & 0xFFFFu, sv.x >> 16, sv.y & 0xFFFFu, sv.y >> 16};
          const uint32_t zb[4] = {zv.x & 0xFFFFu, zv.x >> 16, zv.y & 0xFFFFu, zv.y >> 16};
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float s_lo = kScaleBf16 ? __uint_as_float(sb[2 * j] << 16) : half_bits_to_f32(sb[2 * j]);
            const float s_hi = kScaleBf16 ? __uint_as_float(sb[2 * j + 1] << 16) : half_bits_to_f32(sb[2 * j + 1]);
            const float z_lo = kZero ? __uint_as_float(zb[2 * j] << 16) : 0.f;
            const float z_hi = kZero ? __uint_as_float(zb[2 * j + 1] << 16) : 0.f;
            const float b_lo = fmaf(-8.f, s_lo, z_lo), b_hi = fmaf(-8.f, s_hi, z_hi);
            const float s0 = s_lo * f.x, s1 = s_lo * f.y, s2 = s_hi * f.x, s3 = s_hi * f.y;
            const float* p0 = acc[2 * j];
            const float* p1 = acc[2 * j + 1];
            tot[j][0] = fmaf(s0, p0[0], fmaf(s0, p1[0], fmaf(b_lo, X0, tot[j][0])));
            tot[j][1] = fmaf(s1, p0[1], fmaf(s1, p1[1], fmaf(b_lo, X1, tot[j][1])));
            tot[j][2] = fmaf(s2, p0[2], fmaf(s2, p1[2], fmaf(b_hi, X0, tot[j][2])));
            tot[j][3] = fmaf(s3, p0[3], fmaf(s3, p1[3], fmaf(b_hi, X1, tot[j][3])));
          }
          X0 = X1 = 0.f;
        };
        // group columns: acc[.][0] and acc[.][2] (rows r, r+8) hold token ct's
        // first group, acc[.][1] and acc[.][3] its second (lanes past the
        // tokens hold zeros and are never stored)
        auto fold_gc = [&](int row_a, int row_b) {
          const float f0 = exs[seg * kTok + ct];
          const uint2 sa = *reinterpret_cast<const uint2*>(sbase + row_a * (kStrip * 2));
          const uint2 sb2 = *reinterpret_cast<const uint2*>(sbase + row_b * (kStrip * 2));
          const uint2 za = kZero ? *reinterpret_cast<const uint2*>(sbase + p.zoff + row_a * (kStrip * 2))
                                 : make_uint2(0, 0);
          const uint2 zb2 = kZero ? *reinterpret_cast<const uint2*>(sbase + p.zoff + row_b * (kStrip * 2))
                                  : make_uint2(0, 0);
          const uint32_t s_a[4] = {sa.x & 0xFFFFu, sa.x >> 16, sa.y & 0xFFFFu, sa.y >> 16};
          const uint32_t s_b[4] = {sb2.x & 0xFFFFu, sb2.x >> 16, sb2.y & 0xFFFFu, sb2.y >> 16};
          const uint32_t z_a[4] = {za.x & 0xFFFFu, za.x >> 16, za.y & 0xFFFFu, za.y >> 16};
          const uint32_t z_b[4] = {zb2.x & 0xFFFFu, zb2.x >> 16, zb2.y & 0xFFFFu, zb2.y >> 16};
          auto sf = [&](uint32_t b) { return kScaleBf16 ? __uint_as_float(b << 16) : half_bits_to_f32(b); };
          auto zf = [&](uint32_t b) { return kZero ? __uint_as_float(b << 16) : 0.f; };
#pragma unroll
          for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // h = 0: row r (column 4r + 2j), h = 1: row r + 8 (4r + 2j + 1)
              const float s_ga = sf(s_a[2 * j + h]), s_gb = sf(s_b[2 * j + h]);
              const float b_ga = fmaf(-8.f, s_ga, zf(z_a[2 * j + h])), b_gb = fmaf(-8.f, s_gb, zf(z_b[2 * j + h]));
              const float* p0 = acc[2 * j];
              const float* p1 = acc[2 * j + 1];
              float v = tot[j][2 * h];
              v = fmaf(s_ga * f0, p0[2 * h], fmaf(s_ga * f0, p1[2 * h], fmaf(b_ga, X0, v)));
              v = fmaf(s_gb * f0, p0[2 * h + 1], fmaf(s_gb * f0, p1[2 * h + 1], fmaf(b_gb, X1, v)));
              tot[j][2 * h] = v;
            }
          }
          X0 = X1 = 0.f;
        };
#pragma unroll
        for (int t = 0; t < kUnitRows / 4; ++t) {
          const uint4 w = *reinterpret_cast<const uint4*>((t & 1 ? wo : we) + (t >> 1) * 1024);
          const uint4* xsel = kGC != 0 ? (t < 4 ? xe0 : xe1) : xe;
          const uint4 xv = (t & 1 ? xsel + 1 : xsel)[(t >> 1) * 8];
          // nibble pairs as fp16 subnormals: (i, i+4) at bits 0-3 -> q 2^-24,
          // at bits 4-7 -> 16 q 2^-24 (its activations carry the 1/16)
          const uint32_t xh = w.x >> 8, yh = w.y >> 8, zh = w.z >> 8, wh = w.w >> 8;
          // tile 0: rows r <-> n0, r+8 <-> n0+1; tile 1: rows r <-> n0+2, r+8 <-> n0+3
          if (kGC != 0 ? t == 0 : (kSPF != 0 && t % (kSPF > 0 ? kSPF : 1) == 0)) {   // fresh accumulators
            mma_f16_first(acc[0], w.x & 0x000F000Fu, w.y & 0x000F000Fu, w.x & 0x00F000F0u, w.y & 0x00F000F0u, xv.x, xv.y);
            mma_f16_first(acc[1], xh & 0x000F000Fu, yh & 0x000F000Fu, xh & 0x00F000F0u, yh & 0x00F000F0u, xv.z, xv.w);
            mma_f16_first(acc[2], w.z & 0x000F000Fu, w.w & 0x000F000Fu, w.z & 0x00F000F0u, w.w & 0x00F000F0u, xv.x, xv.y);
            mma_f16_first(acc[3], zh & 0x000F000Fu, wh & 0x000F000Fu, zh & 0x00F000F0u, wh & 0x00F000F0u, xv.z, xv.w);
          } else {
            mma_f16(acc[0], w.x & 0x000F000Fu, w.y & 0x000F000Fu, w.x & 0x00F000F0u, w.y & 0x00F000F0u, xv.x, xv.y);
            mma_f16(acc[1], xh & 0x000F000Fu, yh & 0x000F000Fu, xh & 0x00F000F0u, yh & 0x00F000F0u, xv.z, xv.w);
            mma_f16(acc[2], w.z & 0x000F000Fu, w.w & 0x000F000Fu, w.z & 0x00F000F0u, w.w & 0x00F000F0u, xv.x, xv.y);
            mma_f16(acc[3], zh & 0x000F000Fu, wh & 0x000F000Fu, zh & 0x00F000F0u, wh & 0x00F000F0u, xv.z, xv.w);
          }
          if (kGC != 0 && (t & 1)) {
            // the token's x sums over the unit's two groups (X0: first, X1: second)
            const float bs = xsum[(kunit / 64 + (t >> 1)) * kTok + ct];
            if (t < 4) X0 += bs; else X1 += bs;
            if (t == kUnitRows / 4 - 1) fold_gc(min(row0, p.gh - 1), min(row0 + 1, p.gh - 1));
          } else if (t & 1) {
            // a 64-k block ends: add its x sums (tokens 2c, 2c+1)
            const float2 bs = *reinterpret_cast<const float2*>(xb + (t >> 1) * kTok);
            X0 += bs.x;
            X1 += bs.y;
            if (kSPF != 0) {
              if (t % (kSPF > 0 ? kSPF : 1) == kSPF - 1) fold(min(row0 + t / (kSPF > 0 ? kSPF : 1), p.gh - 1));
            } else if (fold_mask & (1u << t)) {
              fold(row0 + gseg);
              ++gseg;
#pragma unroll
              for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
            }
          }
        }
      }
      // this unit of the tile is consumed; the warp that finishes the stage's
      // last unit refills the slot with stage i + R (the counter only grows:
      // the last of the four units of round i / R reads 4 (i / R) + 3). Every
      // reading thread orders its generic-proxy reads of the slot before the
      // asynchronous copy that will overwrite it, before the warp counts the
      // unit done. Resident stages are never overwritten: nothing to count.
      if (p.resident) continue;
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        asm volatile("fence.acq_rel.cta;" ::: "memory");
        const unsigned int before = atomicAdd(&done[slot], 1u);
        if (before == kUnitsPerStage * static_cast<unsigned int>(i >> p.ring_shift) + kUnitsPerStage - 1 &&
            i + R < total) {
          asm volatile("fence.acq_rel.cta;" ::: "memory");
          tc::fence_proxy_async_smem();   // the warps' reads of the slot before the copy that overwrites it
          issue(i + R);
        }
      }
    }
    if (ok && cur >= 0) flush(cur);
    if (kTmemRed) {
      tc::tmem_wait_st();
      tc::fence_before_sync();
    }
    __syncthreads();
    if (kTmemRed && !*abort_flag) {
      // ---- the partials of the four warps of each TMEM lane quadrant, summed
      // in warp order: lane l holds (token 2c + i % 2, output 4r + 2j + i / 2)
      // in column 4j + i, r = l / 4, c = l % 4 ----
      tc::fence_after_sync();
      for (int su = warp >> 2; su < my_strips; su += 4) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>(su * 32), v);
        float* qd = red + ((su * 4 + (warp & 3)) * 32 + lane) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          qd[e] = ((__uint_as_float(v[e]) + __uint_as_float(v[8 + e])) + __uint_as_float(v[16 + e])) +
                  __uint_as_float(v[24 + e]);
      }
      tc::fence_before_sync();
      __syncthreads();
    }
    if (!*abort_flag) {
      // ---- sum the strip partials of the warps that worked on each strip in
      // a fixed order (with TMEM partials: the quadrant sums in order), scale
      // back, add the bias, write y ----
      const int nout = my_strips * M * kStrip;
      for (int o = threadIdx.x; o < nout; o += kConsumers * 32) {
        const int su = o / (M * kStrip), m = (o / kStrip) % M, nl = o % kStrip;
        const int n = (blockIdx.x + su * gridDim.x) * kStrip + nl;
        const int v0 = su * units, v1 = v0 + min(units, kConsumers);
        float s = 0.f;
        if constexpr (kTmemRed) {
          const int ln = 4 * (nl >> 2) + (m >> 1), e = 4 * ((nl >> 1) & 1) + 2 * (nl & 1) + (m & 1);
          for (int qq = 0; qq < 4; ++qq) s += red[((su * 4 + qq) * 32 + ln) * 8 + e];
        } else {
          for (int vv = v0; vv < v1; ++vv) s += red[((su * kConsumers + vv % kConsumers) * M + m) * kStrip + nl];
        }
        if (n < p.N) {
          s *= 16777216.f;                                       // undo 2^-24 (exact)
          if (p.bias != nullptr) s += __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16);
          const uint16_t yv = static_cast<uint16_t>(f32_to_bf16_bits(s));
          p.y[(size_t)m * p.N + n] = yv;
          if (p.y_host != nullptr) p.y_host[(size_t)m * p.N + n] = yv;
        }
      }
    }
  }
  if (kTmemRed && warp == 0) {
    // every TMEM load and store of the block completed before the last barrier
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
  if (*abort_flag) {
    // let copies already issued land before the shared memory goes away
    const uint64_t t0 = tc::globaltimer_ns();
    while (tc::globaltimer_ns() - t0 < 1000000ull) {
    }
  }
}

#pragma nv_diag_default 549

int sm_count() { return current_sm_count(); }

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder(cudaError_t* err) {
  // looked up once; a function-local static is initialised once even when
  // several host threads get here together
  static const EncodeTiled fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiled>(f);
  }();
  *err = fn == nullptr ? cudaErrorNotSupported : cudaSuccess;
  return fn;
}

// A row-major [rows, N] matrix of `esize`-byte elements, read as tiles of
// 32 columns x box_rows rows (swizzled for the weight words).
cudaError_t encode_rows(CUtensorMap* m, const void* base, int64_t N, int64_t rows, int esize, int box_rows,
                        bool swizzle) {
  cudaError_t e;
  EncodeTiled fn = encoder(&e);
  if (fn == nullptr) return e;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)N * esize};
  const cuuint32_t box[2] = {kStrip, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The most scale groups the k range of one stage meets.
int group_rows(int K, int group) {
  int h = 1;
  for (int k0 = 0; k0 < K; k0 += kStageK) {
    const int k1 = (k0 + kStageK < K ? k0 + kStageK : K) - 1;
    if (k1 / group - k0 / group + 1 > h) h = k1 / group - k0 / group + 1;
  }
  return h;
}

// Bytes of one slot's scale area: gh rows of 32 scales, then as many zeros.
int scale_area(int gh, bool zeros, int* zoff) {
  const int rows = (gh * kStrip * 2 + 127) & ~127;
  *zoff = rows;
  return zeros ? 2 * rows : rows;
}

int x_stride(int K) {
  const int stages = (K + kStageK - 1) / kStageK;
  return stages * kStageK + 8;   // +16 bytes: token rows start in different banks
}

size_t smem_bytes(int K, int rows, int ring, int scb, int pstrips, bool tmem_red = false) {
  const int stages = (K + kStageK - 1) / kStageK;
  return 1024 + static_cast<size_t>(
                    Layout(stages * (kStageK / kUnitK), x_stride(K) / 8, rows, ring, scb, pstrips, tmem_red).total);
}
constexpr size_t kSmemMax = 227 * 1024;

cudaLaunchConfig_t pdl_config(int grid, int block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // programmatic dependent launch: the grid may start while the previous
  // kernel on the stream finishes; it waits for it before reading x
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bool kScaleBf16, bool kZero, int kSPF>
cudaError_t launch_t(const Params& p, bool tmem_red, int grid, size_t smem, cudaStream_t s) {
  auto k = tmem_red ? w4a16_kernel<kScaleBf16, kZero, kSPF, true> : w4a16_kernel<kScaleBf16, kZero, kSPF, false>;
  if constexpr (kSPF == 4)
    if (!tmem_red && p.M <= 4)
      k = p.M == 1 ? w4a16_kernel<kScaleBf16, kZero, 4, false, 1> : w4a16_kernel<kScaleBf16, kZero, 4, false, 4>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(grid, kThreads, smem, s, attr);
  return cudaLaunchKernelEx(&cfg, k, p);
}

template <bool kScaleBf16>
cudaError_t launch_spf(const Params& p, bool z, int spf, bool tr, int grid, size_t smem, cudaStream_t s) {
  switch (spf) {
    case 2: return z ? launch_t<kScaleBf16, true, 2>(p, tr, grid, smem, s) : launch_t<kScaleBf16, false, 2>(p, tr, grid, smem, s);
    case 4: return z ? launch_t<kScaleBf16, true, 4>(p, tr, grid, smem, s) : launch_t<kScaleBf16, false, 4>(p, tr, grid, smem, s);
    case 8: return z ? launch_t<kScaleBf16, true, 8>(p, tr, grid, smem, s) : launch_t<kScaleBf16, false, 8>(p, tr, grid, smem, s);
    default: return z ? launch_t<kScaleBf16, true, 0>(p, tr, grid, smem, s) : launch_t<kScaleBf16, false, 0>(p, tr, grid, smem, s);
  }
}

}  // namespace

size_t w4a16_smem_bytes(int64_t N, int64_t K, int32_t group) {
  int zoff;
  const int scb = scale_area(group_rows(static_cast<int>(K), group), true, &zoff);
  const int64_t strips = (N + kStrip - 1) / kStrip;
  const int64_t grid = strips < sm_count() ? strips : sm_count();
  const int pstrips = static_cast<int>((strips + grid - 1) / (grid > 0 ? grid : 1));
  return smem_bytes(static_cast<int>(K), 1, 4, scb, pstrips);
}

cudaError_t launch_w4a16(const W4A16Args& a, cudaStream_t s) {
  Params p;
  memset(&p, 0, sizeof(p));
  const int G = static_cast<int>(a.K / a.group);
  p.gh = group_rows(static_cast<int>(a.K), a.group);
  p.scb = scale_area(p.gh, a.zeros != nullptr, &p.zoff);
  cudaError_t e = encode_rows(&p.tm_w, a.qweight, a.N, a.K / 8, 4, kStageRows, true);
  if (e == cudaSuccess) e = encode_rows(&p.tm_s, a.w_scale, a.N, G, 2, p.gh, false);
  if (e == cudaSuccess && a.zeros != nullptr) e = encode_rows(&p.tm_z, a.zeros, a.N, G, 2, p.gh, false);
  if (e != cudaSuccess) return e;
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.group = a.group;
  p.strips = (p.N + kStrip - 1) / kStrip;
  p.stages = (p.K + kStageK - 1) / kStageK;
  p.xstride = x_stride(p.K);
  p.group_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if (p.group == (1 << sh)) p.group_shift = sh;
  p.status = a.status;
  const int grid = p.strips < sm_count() ? p.strips : sm_count();
  p.pstrips = (p.strips + grid - 1) / grid;
  auto bytes = [&](int rows, int ring) { return smem_bytes(p.K, rows, ring, p.scb, p.pstrips); };
  // Tokens go in blocks of up to 8, each block one pass over the weights,
  // beside a ring of 8 stages when it fits, else 4.
  int block = kTok;
  while (block > 1 && bytes(block, 4) > kSmemMax) --block;
  if (bytes(block, 4) > kSmemMax) return cudaErrorInvalidValue;
  const bool z = a.zeros != nullptr;
  // fixed fold points for the common group sizes
  const int spf = p.group == 64 ? 2 : p.group == 128 ? 4 : p.group % 256 == 0 ? 8 : 0;
  {
    // this call's weights, scales and zeros on their way into L2 while the
    // kernel before it on the stream still runs
    const size_t wb = static_cast<size_t>(a.K / 8) * a.N * 4, sb = static_cast<size_t>(G) * a.N * 2;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(sm_count(), 32, 0, s, attr);
    e = cudaLaunchKernelEx(&cfg, w4a16_prefetch_kernel, static_cast<const uint8_t*>(a.qweight), wb,
                           static_cast<const uint8_t*>(a.w_scale), sb, static_cast<const uint8_t*>(a.zeros),
                           z ? sb : size_t(0), static_cast<const uint4*>(a.x_host),
                           static_cast<uint4*>(const_cast<void*>(a.x)),
                           a.x_host != nullptr ? static_cast<size_t>(a.M) * a.K * 2 / 16 : size_t(0));
    if (e != cudaSuccess) return e;
  }
  for (int64_t m0 = 0; m0 < a.M; m0 += block) {
    p.x = static_cast<const uint16_t*>(a.x) + m0 * a.K;
    p.y = static_cast<uint16_t*>(a.y) + m0 * a.N;
    p.y_host = a.y_host != nullptr ? static_cast<uint16_t*>(a.y_host) + m0 * a.N : nullptr;
    p.M = static_cast<int>(a.M - m0 < block ? a.M - m0 : block);
    p.ring = bytes(p.M, 8) <= kSmemMax ? 8 : 4;
    // when the shared-memory partials cost the ring half its depth, the
    // partials go to tensor memory (8 columns per strip and warp group:
    // at most 16 strips a CTA in its 512 columns)
    const bool tmem_red = p.ring == 4 && p.pstrips <= 16 && smem_bytes(p.K, p.M, 8, p.scb, p.pstrips, true) <= kSmemMax;
    if (tmem_red) p.ring = 8;
    p.slots = p.ring;
    p.resident = 0;
    // every stage of a CTA in its own slot when they fit: no slot is
    // refilled, so the units skip the per-unit release (fences, counter,
    // refill copy), which measured as long as a unit's math
    const int share = p.pstrips * p.stages;
    if (!tmem_red && share <= kRingMax && bytes(p.M, share) <= kSmemMax) {
      p.ring = share <= 8 ? 8 : kRingMax;
      p.slots = share;
      p.resident = 1;
    }
    p.ring_shift = p.ring == 16 ? 4 : p.ring == 8 ? 3 : 2;
    const size_t smem = smem_bytes(p.K, p.M, p.slots, p.scb, p.pstrips, tmem_red);
    e = a.scale_bf16 ? launch_spf<true>(p, z, spf, tmem_red, grid, smem, s)
                     : launch_spf<false>(p, z, spf, tmem_red, grid, smem, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w4
