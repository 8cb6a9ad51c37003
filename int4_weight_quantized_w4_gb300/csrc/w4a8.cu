// W4A8 and W4AFP8 GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// vLLM API docs, inc.schemes.inc_w4a8_linear, INCXPUW4A8LinearMethod
// (class docstring, apply_weights): int8 per-token activations times the GPTQ
// int4 weight [K/8, N] with fp16 group scales, keeping the GEMM on an 8-bit
// datapath for compute-bound token counts. vLLM API docs, quantization.w4afp8,
// W4AFP8Config: int4 group-128 routed experts with fp8 per-token activations,
// weights in the compressed-tensors layout [E, N, K/8].
//
// sm_103a has no integer tensor-core MMA, so the integer products run exactly
// on the fp16 path: every int8 activation and every weight value q - 8 is an
// exact fp16, every product is exact in fp32, and a group's partial sum
// (|P| <= 127 * 8 * 16384 < 2^24) is an integer the fp32 accumulator holds
// exactly. e4m3 activations are exact in fp16 too.
//
// Per output tile of 128 outputs (n) x 256 tokens:
//  * swap-AB: the weights are the MMA's M operand (TMEM lane = output n),
//    the tokens its N operand, so the per-group scale s[g, n] is one register
//    per epilogue thread;
//  * TMA streams the raw packed weight words into a ring in shared memory;
//    converter warps turn each 32-bit word (8 nibbles) into 8 exact fp16
//    values q - 8 with LOP3 + HSUB2/HFMA2 (the fp16 mantissa of 1024 + q) and
//    write them into the 128-byte-swizzled K-major operand tile;
//  * the activations were widened once per call to exact fp16 (see
//    widen_kernel) and TMA loads them straight into the swizzled layout;
//  * one thread issues tcgen05.mma (M=128, N=256, K=16) into a TMEM
//    accumulator per group; the accumulator is double-buffered so the
//    epilogue folds group g (T += s[g,n] * P) while group g+1 accumulates;
//  * the epilogue finally writes y = bf16(s_x[m] * T + bias[n]).
// Within every 8-wide chunk of k both operands use the order
// (k0,k4,k1,k5,k2,k6,k3,k7), the order the nibble pairs come out in.
// One CTA per SM walks its share of the tiles (persistent), every ring
// counting on across tiles; a k-stage is two 64-k swizzle rows, so the MMA
// thread's per-stage waits and commits serve eight MMAs.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace w4 {
namespace {

constexpr int BM = 128;          // outputs per tile (MMA M, TMEM lanes)
constexpr int BN = 256;          // tokens per tile (MMA N)
constexpr int SEG_MAX = 16384;   // longest accumulation before a drain (exactness bound)

constexpr int A_SUB = BM * 128;         // 16 KB per sub-tile: one 128-byte swizzle row per output
constexpr int B_SUB = BN * 128;         // 32 KB per sub-tile: one 128-byte swizzle row per token

// A sub-tile is one 128-byte swizzle row per operand row: 64 k of fp16 or
// 128 k of e4m3 (FP8, kind::f8f6f4). An MMA takes 32 bytes of k either way
// (16 fp16 or 32 e4m3 values), so the descriptor steps are the same and an
// fp8 stage covers twice the k of an fp16 stage in the same MMA time.
// A stage is SUBS sub-tiles; the MMA thread's per-stage waits, fence and
// commits are shared by 4 x SUBS MMAs. Measured on GB300: with the operand
// producers taken out entirely a 64-k fp16 stage still took ~0.8 us (its four
// MMAs alone ~0.25 us in isolation), and two sub-tiles per stage raised the
// dense GEMM 12-19%. Every configuration uses two (Cfg<2, *>).
template <int SUBS, bool FP8>
struct Cfg {
  static constexpr int KS = FP8 ? 128 : 64;               // k per sub-tile
  static constexpr int UMMA_K = FP8 ? 32 : 16;            // k per MMA
  static constexpr int BK = KS * SUBS;                     // k per stage
  static constexpr int A_STAGES = SUBS == 1 ? 3 : 2;       // converted weight tiles
  static constexpr int B_STAGES = SUBS == 1 ? 4 : 2;       // activation tiles; even: each copy warp keeps its slots
  static constexpr int RAW_STAGES = 2;                     // packed weight words, RAW_PER k-stages per slot
  static constexpr int RAW_PER = 256 / BK;                 // one 16 KB packed-word copy per 256 k
  static constexpr int A_BYTES = A_SUB * SUBS;
  static constexpr int B_BYTES = B_SUB * SUBS;
  static constexpr int RAW_BYTES = BM * 256 / 2;           // 16 KB: 32 word rows of 128 outputs
  static constexpr int SMEM = B_STAGES * B_BYTES + A_STAGES * A_BYTES + RAW_STAGES * RAW_BYTES + 2048 + 1024;
};
static_assert(Cfg<2, false>::RAW_PER * Cfg<2, false>::BK == 256 && Cfg<2, true>::RAW_PER * Cfg<2, true>::BK == 256,
              "a packed-word copy is 32 word rows in every configuration");
static_assert(Cfg<2, false>::SMEM <= 232448 && Cfg<2, true>::SMEM <= 232448, "shared memory per CTA");
static_assert(Cfg<2, false>::A_STAGES == Cfg<2, false>::B_STAGES && Cfg<2, true>::A_STAGES == Cfg<2, true>::B_STAGES,
              "one full and one empty barrier serve both operands of a stage");

// Warp roles, four warpgroups: 0-7 epilogue (warp w reads TMEM lane quadrant
// w % 4, token half w / 4), 8-11 converters, 12 weight-word TMA, 13 and 15
// activation TMA (even / odd k-stages), 14 MMA issuer (and TMEM owner).
// Copies are issued from two warps and packed words 256 k at a time because
// on GB300 the copies one thread issues complete about one per 0.5 us
// whatever their size (4-64 KB): one issuer would feed the 32 KB activation
// tile of a 0.25 us stage at half the rate the MMAs consume it.
constexpr int kEpiWarps = 8;
constexpr int kConvWarps = 4;
constexpr int kWarpConv0 = 8;
constexpr int kWarpLoadW = 12;
constexpr int kWarpLoadB = 13;   // activation copies of even k-stages
constexpr int kWarpLoadB2 = 15;  // activation copies of odd k-stages
constexpr int kWarpMma = 14;
constexpr int kThreads = 16 * 32;
constexpr uint32_t kTmemCols = 2 * BN;        // double-buffered accumulator
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr int kEpiCols = BN / 2;              // token columns per epilogue thread


enum Mode : int { kDenseY = 0, kDensePartials = 1, kExperts = 2 };

struct Params {
  CUtensorMap tm_act;      // fp16 activations [rows, K], widened and permuted
  CUtensorMap tm_w;        // raw weight words: GPTQ [K/8, N] or CT [E, N, K/8]
  const uint16_t* w_scale; // fp16 [G, N] or [E, N, G]
  const float* x_scale;    // [rows]
  const uint16_t* bias;    // bf16 [N] or null
  void* out;               // bf16 [rows, N] or int32 [rows, G, N]
  const int32_t* offsets;  // [E + 1] (experts)
  int E, M, N, K, group, mode;
  int raw_rows;            // word rows (k / 8) per packed-word copy: min(32, K / 8)
  int m_tiles;             // row tiles (dense: ceil(M / 256); experts: an upper bound over all segments)
  int splits, ksplit;      // dense y: the K range cut into `splits` parts of `ksplit` (the last may be shorter)
  float* part;             // splits > 1: fp32 partial sums [splits][M][N], before x_scale and bias
  // dense y, the last wave only: work items 0 .. full_tiles - 1 are whole tiles; item full_tiles + j is part
  // j % tail_splits (tail_ksplit of k) of tile full_tiles + j / tail_splits
  int full_tiles, tail_tiles, tail_splits, tail_ksplit;
  float* tail_part;        // tail_splits > 1: fp32 partial sums [tail tile][part][BN rows][BM outputs]
  int items;               // work items the persistent CTAs walk
  unsigned int* status;
};

// 8 nibbles (k0..k7 of one output) -> 8 exact fp16 values q - 8 in the order
// (k0,k4,k1,k5,k2,k6,k3,k7). 0x6400 | q is 1024 + q; 0x6400 | q << 4 is
// 1024 + 16 q, which one fp16 FMA maps to q - 8 exactly.
W4_DEV uint4 nibbles_to_f16(uint32_t w) {
  const uint32_t w8 = w >> 8;
  uint4 o;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o.x) : "r"(and_or(w, 0x000F000Fu, 0x64006400u)), "r"(0x64086408u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o.y) : "r"(and_or(w, 0x00F000F0u, 0x64006400u)), "r"(0x2C002C00u),
      "r"(0xD480D480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o.z) : "r"(and_or(w8, 0x000F000Fu, 0x64006400u)), "r"(0x64086408u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o.w) : "r"(and_or(w8, 0x00F000F0u, 0x64006400u)), "r"(0x2C002C00u),
      "r"(0xD480D480u));
  return o;
}

// 8 nibbles (k0..k7 of one output) -> the e4m3 codes of (q - 8) * 2^-9 in
// natural k order (byte j = k j), the order the caller's e4m3 activations
// come in. In the lowest binades of e4m3 the code of v * 2^-9 for an integer
// 0 <= v <= 15 is v itself (subnormals m * 2^-9 for v < 8, then exponent
// field 1, (8 + m) * 2^-9), so with the sign bit every weight value is one
// byte: q >= 8 -> q - 8 = q ^ 8; q < 8 -> 0x80 | (8 - q) = 0x88 - q. The
// epilogue multiplies the group scale by 2^9 (exact) to undo the 2^-9.
W4_DEV uint2 nibbles_to_e4m3(uint32_t w) {
  const uint32_t e = w & 0x0F0F0F0Fu;                // k0 k2 k4 k6, one per byte
  const uint32_t o = (w >> 4) & 0x0F0F0F0Fu;         // k1 k3 k5 k7
  const uint32_t me = prmt(w << 4, 0u, 0xBA98u);     // 0xFF in the bytes whose q >= 8 (the nibble's bit 3)
  const uint32_t mo = prmt(w, 0u, 0xBA98u);
  // bytewise, with no borrow between bytes (q <= 15 < 0x88)
  const uint32_t ce = select_bits(me, e ^ 0x08080808u, 0x88888888u - e);
  const uint32_t co = select_bits(mo, o ^ 0x08080808u, 0x88888888u - o);
  return make_uint2(prmt(ce, co, 0x5140u), prmt(ce, co, 0x7362u));   // k0 k1 k2 k3, k4 k5 k6 k7
}

W4_DEV void bar_sync_epilogue() { asm volatile("bar.sync 1, %0;" :: "n"(kEpiWarps * 32) : "memory"); }

// Output tile `tid` of the grid of tiles (N tiles fastest): outputs n0 .. n0 +
// BM, rows row0 .. row_end (of one expert's segment in expert mode). False if
// the tile holds no rows. Every role decodes the same tiles the same way.
struct Tile {
  int n0, row0, row_end, expert;
  int k0, k1, split;   // the tile's k range (all of K unless the GEMM is split along K)
  int tail;            // index among the last wave's split tiles, or -1
};
// Where a role's walk over the experts stands: expert e, and the row tiles of
// the experts before it. A role visits its tiles in increasing order, so the
// expert of its next tile is never before the current one: each role reads
// the offsets once per expert and once per tile, not once per expert per tile.
struct TileCursor {
  int e = 0, base = 0;
};
// kTail: the launch splits the last wave's tiles (a separate instantiation:
// the remapping below, in the decode every role runs, measured ~4% slower per
// tile on grouped shapes, so launches without it do not carry it).
template <bool kTail>
W4_DEV bool decode_tile(const Params& p, int tid, int n_tiles, Tile& t, TileCursor& cur) {
  t.tail = -1;
  int part = 0;
  if (kTail && tid >= p.full_tiles) {   // a K part of one of the last wave's tiles
    const int j = tid - p.full_tiles;
    t.tail = j / p.tail_splits;
    part = j - t.tail * p.tail_splits;
    tid = p.full_tiles + t.tail;
  }
  const int nx = tid % n_tiles;
  int yt = tid / n_tiles;
  t.n0 = nx * BM;
  t.expert = 0;
  t.row0 = 0;
  t.row_end = 0;
  t.split = 0;
  t.k0 = 0;
  t.k1 = p.K;
  if (p.splits > 1) {   // dense only: N tiles fastest, then row tiles, then splits
    t.split = yt / p.m_tiles;
    yt %= p.m_tiles;
    t.k0 = t.split * p.ksplit;
    t.k1 = min(p.K, t.k0 + p.ksplit);
  }
  if (kTail && t.tail >= 0) {
    t.split = part;
    t.k0 = part * p.tail_ksplit;
    t.k1 = min(p.K, t.k0 + p.tail_ksplit);
  }
  if (p.mode == kExperts) {
    for (; cur.e < p.E; ++cur.e) {
      const int a = p.offsets[cur.e], b = p.offsets[cur.e + 1];
      const int nt = b > a ? (b - a + BN - 1) / BN : 0;
      if (yt < cur.base + nt) {
        t.expert = cur.e;
        t.row0 = a + (yt - cur.base) * BN;
        t.row_end = min(t.row0 + BN, b);
        break;
      }
      cur.base += nt;
    }
    t.row0 = max(t.row0, 0);
    t.row_end = min(t.row_end, p.M);
  } else {
    t.row0 = yt * BN;
    t.row_end = min(t.row0 + BN, p.M);
  }
  return t.row0 < t.row_end;
}

// Persistent: one CTA per SM takes tiles blockIdx.x, blockIdx.x + gridDim.x,
// ... of the n_tiles x y_tiles grid. Every ring (packed words, operand A,
// operand B, the two TMEM accumulators) keeps counting across tiles, so the
// copies and conversions of the next tile run while this tile's last groups
// are multiplied and its output is written.
template <int SUBS, bool FP8, bool kTail>
__global__ void __launch_bounds__(kThreads, 1) w4a8_tc_kernel(const __grid_constant__ Params p, int n_tiles,
                                                              int y_tiles) {
  using C = Cfg<SUBS, FP8>;
  constexpr int KS = C::KS, UMMA_K = C::UMMA_K;
  constexpr int BK = C::BK, A_STAGES = C::A_STAGES, B_STAGES = C::B_STAGES, RAW_STAGES = C::RAW_STAGES;
  constexpr int RAW_PER = C::RAW_PER, A_BYTES = C::A_BYTES, B_BYTES = C::B_BYTES, RAW_BYTES = C::RAW_BYTES;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));

  uint8_t* b_base = smem;                                  // 1024-aligned
  uint8_t* a_base = b_base + B_STAGES * B_BYTES;           // 1024-aligned
  uint8_t* raw_base = a_base + A_STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw_base + RAW_STAGES * RAW_BYTES);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + RAW_STAGES;
  // one "stage full" barrier per k-stage (the converter warps' arrivals and
  // the activation copy's bytes) and one "stage empty" barrier (a single
  // commit of the stage's MMAs, waited on by both producers)
  uint64_t* st_full = raw_empty + RAW_STAGES;
  uint64_t* st_empty = st_full + A_STAGES;
  uint64_t* acc_full = st_empty + A_STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* xs_s = reinterpret_cast<float*>(tmem_holder + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < RAW_STAGES; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kConvWarps);
    }
    for (int i = 0; i < A_STAGES; ++i) {
      mbar_init(&st_full[i], kConvWarps + 1);
      mbar_init(&st_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tc::tmem_alloc(tmem_holder, kTmemCols);
  if (warp == kWarpLoadW && lane == 0) {
    tc::prefetch_tmap(&p.tm_w);
    tc::prefetch_tmap(&p.tm_act);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  const int K = p.K;
  const int group = p.group;
  // n_tiles * y_tiles, or (kTail) the whole tiles plus the last wave's K parts
  const int total_tiles = kTail ? p.items : n_tiles * y_tiles;

  if (warp >= kEpiWarps) {
  // producer warpgroups give registers to the epilogue warpgroups
  asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
  if (warp == kWarpLoadW) {
    // ---- raw packed weight words -> ring ----
    if (lane == 0) {
      int rg = 0;   // copies issued so far (all tiles)
      bool ok = true;
      TileCursor cur;
      for (int tid = blockIdx.x; tid < total_tiles && ok; tid += gridDim.x) {
        Tile t;
        if (!decode_tile<kTail>(p, tid, n_tiles, t, cur)) continue;
        const int nraw = ((t.k1 - t.k0 + BK - 1) / BK + RAW_PER - 1) / RAW_PER;
        for (int ri = 0; ri < nraw; ++ri, ++rg) {
          const int r = rg % RAW_STAGES;
          if (!tc::wait(&raw_empty[r], ((rg / RAW_STAGES) & 1) ^ 1, abort_flag, p.status, kWaitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[r], static_cast<uint32_t>(p.raw_rows * BM * 4));
          const int wrow = t.k0 / 8 + ri * RAW_PER * (BK / 8);   // first word row of the copy
          if (p.mode == kExperts)
            tc::tma_load_3d(raw_base + r * RAW_BYTES, &p.tm_w, &raw_full[r], wrow, t.n0, t.expert);
          else
            tc::tma_load_2d(raw_base + r * RAW_BYTES, &p.tm_w, &raw_full[r], t.n0, wrow);
        }
      }
    }
  } else if (warp == kWarpLoadB || warp == kWarpLoadB2) {
    // ---- widened activations -> ring; the two warps take alternate stages
    // (B_STAGES is even, so each keeps its own slots) ----
    if (lane == 0) {
      const int mine = warp == kWarpLoadB ? 0 : 1;
      int sg = 0;   // stages so far (all tiles)
      bool ok = true;
      TileCursor cur;
      for (int tid = blockIdx.x; tid < total_tiles && ok; tid += gridDim.x) {
        Tile t;
        if (!decode_tile<kTail>(p, tid, n_tiles, t, cur)) continue;
        const int nst = (t.k1 - t.k0 + BK - 1) / BK;
        for (int s = 0; s < nst; ++s, ++sg) {
          if ((sg & 1) != mine) continue;
          const int b = sg % B_STAGES;
          if (!tc::wait(&st_empty[b], ((sg / B_STAGES) & 1) ^ 1, abort_flag, p.status, kWaitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&st_full[b], B_BYTES);
#pragma unroll
          for (int u = 0; u < SUBS; ++u)   // sub-tiles past K land as zeros
            tc::tma_load_2d(b_base + b * B_BYTES + u * B_SUB, &p.tm_act, &st_full[b], t.k0 + s * BK + u * KS,
                            t.row0);
        }
      }
    }
  } else if (warp >= kWarpConv0 && warp < kWarpConv0 + kConvWarps) {
    // ---- nibbles -> fp16 operand A ----
    const int tr = threadIdx.x - kWarpConv0 * 32;  // output row within the tile
    int sg = 0, rg = 0;
    bool ok = true;
    TileCursor cur;
    for (int tid = blockIdx.x; tid < total_tiles && ok; tid += gridDim.x) {
      Tile t;
      if (!decode_tile<kTail>(p, tid, n_tiles, t, cur)) continue;
      const int nst = (t.k1 - t.k0 + BK - 1) / BK;
      for (int s = 0; s < nst; ++s, ++sg) {
        const int sub = s % RAW_PER;   // k-stage within its packed-word copy
        const int r = rg % RAW_STAGES, a = sg % A_STAGES;
        if (!tc::wait(&raw_full[r], (rg / RAW_STAGES) & 1, abort_flag, p.status, kWaitNs)) {
          ok = false;
          break;
        }
        const uint32_t* raw = reinterpret_cast<const uint32_t*>(raw_base + r * RAW_BYTES);
        constexpr int kWords = BK / 8;   // packed words of one output per stage
        uint32_t w[kWords];
        if (p.mode == kExperts) {  // box [128 outputs][raw_rows words]
          // 32-word rows arrive 128-byte swizzled: 16-byte chunk c of row tr
          // sits at chunk c ^ (tr % 8), so a quarter-warp's loads hit 8
          // distinct bank groups
          const int swz = p.raw_rows == 32 ? (tr & 7) : 0;
#pragma unroll
          for (int v4 = 0; v4 < kWords / 4; ++v4) {
            const int c = sub * (kWords / 4) + v4;
            const uint4 q4 = *reinterpret_cast<const uint4*>(raw + tr * p.raw_rows + 4 * (c ^ swz));
            w[4 * v4] = q4.x;
            w[4 * v4 + 1] = q4.y;
            w[4 * v4 + 2] = q4.z;
            w[4 * v4 + 3] = q4.w;
          }
        } else {  // box [raw_rows words][128 outputs]
#pragma unroll
          for (int kb = 0; kb < kWords; ++kb) w[kb] = raw[(sub * kWords + kb) * BM + tr];
        }
        // The next asynchronous (TMA) copy into this slot must land after
        // these generic-proxy reads of it: the proxy fence orders them before
        // the release below. Without it, expert tiles on two-sub-tile stages
        // were measured to convert words of the slot's next copy.
        tc::fence_proxy_async_smem();
        __syncwarp();
        // the copy's words are in registers once its last k-stage is read
        if (sub == RAW_PER - 1 || s == nst - 1) {
          if (lane == 0) mbar_arrive(&raw_empty[r]);
          ++rg;
        }
        if (!tc::wait(&st_empty[a], ((sg / A_STAGES) & 1) ^ 1, abort_flag, p.status, kWaitNs)) {
          ok = false;
          break;
        }
        uint8_t* arow = a_base + a * A_BYTES + tr * 128;
        if constexpr (FP8) {
#pragma unroll
          for (int kp = 0; kp < kWords / 2; ++kp) {   // words 2kp, 2kp+1: sub-tile kp / 8, chunk kp % 8
            const uint2 lo = nibbles_to_e4m3(w[2 * kp]), hi = nibbles_to_e4m3(w[2 * kp + 1]);
            *reinterpret_cast<uint4*>(arow + (kp >> 3) * A_SUB + (((kp & 7) ^ (tr & 7)) << 4)) =
                make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
        } else {
#pragma unroll
          for (int kb = 0; kb < kWords; ++kb)   // word kb: sub-tile kb / 8, 16-byte chunk kb % 8 of the row
            *reinterpret_cast<uint4*>(arow + (kb >> 3) * A_SUB + (((kb & 7) ^ (tr & 7)) << 4)) = nibbles_to_f16(w[kb]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&st_full[a]);
      }
    }
  } else if (warp == kWarpMma) {
    // ---- one thread issues the MMAs ----
    // One wait and two descriptors per stage, the MMAs from constant offsets.
    // The tensor pipe takes only a few MMAs ahead of the issuing thread, so
    // what that thread does between MMAs shows up as idle pipe: whole stages
    // whose accumulations can change only at the stage's start or middle
    // (groups that are multiples of the stage width, or half of it) run
    // straight-line, with no per-MMA checks; measured on GB300, that alone
    // took the grouped prefill GEMM from 855 to 1,148 TOPS. Stages at a tile's
    // ragged end and other group sizes (multiples of 16) take the general
    // loop. Every tile opens a new accumulation.
    if (lane == 0) {
      // e4m3 A and B under kind::f8f6f4 take the same format code (0) that
      // fp16 takes under kind::f16, so one instruction descriptor serves both
      constexpr uint32_t idesc = tc::idesc_f16_f32(BM, BN);
      const uint64_t adesc0 = tc::sdesc_sw128(smem_addr(a_base));
      const uint64_t bdesc0 = tc::sdesc_sw128(smem_addr(b_base));
      int seg = -1, buf = 0, sg = 0;
      // accumulations change only at stage starts or middles: group boundaries
      // there (SEG_MAX is a multiple of every stage width)
      const bool lean = group % BK == 0 || 2 * group == BK;
      bool ok = true;
      TileCursor cur;
      for (int tid = blockIdx.x; tid < total_tiles && ok; tid += gridDim.x) {
        Tile t;
        if (!decode_tile<kTail>(p, tid, n_tiles, t, cur)) continue;
        ++seg;
        buf = seg & 1;
        const int nst = (t.k1 - t.k0 + BK - 1) / BK;
        int seg_end = min(min((t.k0 / group + 1) * group, t.k0 + SEG_MAX), t.k1);
        uint32_t acc = 0;
        if (!tc::wait(&acc_empty[buf], ((seg >> 1) & 1) ^ 1, abort_flag, p.status, kWaitNs)) break;
        tc::fence_after_sync();
        for (int s = 0; s < nst && ok; ++s, ++sg) {
          const int a = sg % A_STAGES, b = sg % B_STAGES;
          if (!tc::wait(&st_full[a], (sg / A_STAGES) & 1, abort_flag, p.status, kWaitNs, 200)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t ad = adesc0 + static_cast<uint64_t>((a * A_BYTES) >> 4);
          const uint64_t bd = bdesc0 + static_cast<uint64_t>((b * B_BYTES) >> 4);
          const int kbase = t.k0 + s * BK;
          constexpr int kPerSub = KS / UMMA_K;
          if (lean && kbase + BK <= t.k1) {
            // a whole stage whose accumulations can only change at its start or
            // its middle (tiles start on stage boundaries): no per-MMA checks
            constexpr int kHalf = BK / UMMA_K / 2;
#pragma unroll
            for (int h = 0; h < 2 && ok; ++h) {
              const int kh = kbase + h * (BK / 2);
              if (seg_end == kh) {   // close this accumulation, open the next buffer
                tc::commit(&acc_full[buf]);
                ++seg;
                buf = seg & 1;
                seg_end = min(min((kh / group + 1) * group, kh + SEG_MAX), t.k1);
                if (!tc::wait(&acc_empty[buf], ((seg >> 1) & 1) ^ 1, abort_flag, p.status, kWaitNs)) {
                  ok = false;
                  break;
                }
                tc::fence_after_sync();
                acc = 0;
              }
              const uint32_t d = tmem + buf * BN;
#pragma unroll
              for (int i = 0; i < kHalf; ++i) {
                const int j = h * kHalf + i, u = j / kPerSub, jj = j % kPerSub;
                if constexpr (FP8)
                  tc::mma_f8(d, ad + ((u * A_SUB) >> 4) + 2 * jj, bd + ((u * B_SUB) >> 4) + 2 * jj, idesc,
                             i > 0 ? 1u : acc);
                else
                  tc::mma_f16(d, ad + ((u * A_SUB) >> 4) + 2 * jj, bd + ((u * B_SUB) >> 4) + 2 * jj, idesc,
                              i > 0 ? 1u : acc);
              }
              acc = 1;
            }
          } else {
#pragma unroll
          for (int j = 0; j < BK / UMMA_K; ++j) {
            // MMA j: sub-tile j / 4, 32-byte step j % 4 inside its swizzle rows
            const int k = kbase + j * UMMA_K;
            if (k < t.k1) {
              if (k == seg_end) {  // close this accumulation, open the next buffer
                tc::commit(&acc_full[buf]);
                ++seg;
                buf = seg & 1;
                const int g = k / group;
                seg_end = min(min((g + 1) * group, k + SEG_MAX), t.k1);
                if (!tc::wait(&acc_empty[buf], ((seg >> 1) & 1) ^ 1, abort_flag, p.status, kWaitNs)) {
                  ok = false;
                  break;
                }
                tc::fence_after_sync();
                acc = 0;
              }
              const int u = j / kPerSub, jj = j % kPerSub;
              if constexpr (FP8)
                tc::mma_f8(tmem + buf * BN, ad + ((u * A_SUB) >> 4) + 2 * jj, bd + ((u * B_SUB) >> 4) + 2 * jj, idesc,
                           acc);
              else
                tc::mma_f16(tmem + buf * BN, ad + ((u * A_SUB) >> 4) + 2 * jj, bd + ((u * B_SUB) >> 4) + 2 * jj,
                            idesc, acc);
              acc = 1;
            }
          }
          }
          if (!ok) break;
          tc::commit(&st_empty[a]);
        }
        if (ok) tc::commit(&acc_full[buf]);
      }
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    // ---- epilogue: warp w owns TMEM lanes 32(w%4).. (outputs), token half w/4 ----
    const int q = warp & 3, half = warp >> 2;
    const int N = p.N;
    const int G = K / group;
    const bool partials = p.mode == kDensePartials;
    const int c0 = half * kEpiCols;
    int seg = 0;   // accumulations drained so far (all tiles)
    // Every epilogue thread walks every tile and meets both named barriers of
    // each, even after a wait has run out (ok = false then skips the work):
    // threads that left the loop early would strand the others at bar.sync.
    bool ok = true;
    TileCursor cur;
    for (int tid = blockIdx.x; tid < total_tiles; tid += gridDim.x) {
      Tile t;
      if (!decode_tile<kTail>(p, tid, n_tiles, t, cur)) continue;
      const int n = t.n0 + 32 * q + lane;
      const bool n_ok = n < N;
      bar_sync_epilogue();   // the previous tile's output is written: xs_s may change
      if (!partials)
        for (int j = threadIdx.x; j < BN; j += kEpiWarps * 32)
          xs_s[j] = (t.row0 + j < t.row_end) ? p.x_scale[t.row0 + j] : 0.f;
      bar_sync_epilogue();

      float T[kEpiCols];
#pragma unroll
      for (int j = 0; j < kEpiCols; ++j) T[j] = 0.f;

      // the scales of this group and the next three, loaded ahead: with the TMA
      // pipes full a plain load takes ~1-2 us, a group's MMAs ~0.5 us
      auto ld_scale = [&](int gg) -> uint32_t {
        if (partials || !n_ok || gg >= G) return 0u;
        const size_t si = (p.mode == kExperts) ? ((size_t)t.expert * N + n) * G + gg : (size_t)gg * N + n;
        return p.w_scale[si];
      };
      const int g0 = t.k0 / group;
      uint32_t sr0 = ld_scale(g0), sr1 = ld_scale(g0 + 1), sr2 = ld_scale(g0 + 2), sr3 = ld_scale(g0 + 3);
      int cur_g = g0;
      for (int k0 = t.k0; ok && k0 < t.k1; ++seg) {
        const int g = k0 / group;
        if (g != cur_g) {   // segments walk k in order: the group advances by one
          sr0 = sr1;
          sr1 = sr2;
          sr2 = sr3;
          sr3 = ld_scale(g + 3);
          cur_g = g;
        }
        const int kend = min(min((g + 1) * group, k0 + SEG_MAX), t.k1);
        const int buf = seg & 1;
        if (!tc::wait(&acc_full[buf], (seg >> 1) & 1, abort_flag, p.status, kWaitNs)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * BN + c0;
        if (partials) {
          int32_t* out = static_cast<int32_t*>(p.out);
#pragma unroll 1
          for (int cc = 0; cc < kEpiCols / 32; ++cc) {
            uint32_t v[32];
            tc::tmem_ld32(taddr + cc * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int row = t.row0 + c0 + cc * 32 + j;
              if (n_ok && row < t.row_end)
                out[((size_t)row * G + g) * N + n] = __float2int_rn(__uint_as_float(v[j]));
            }
          }
        } else {
          // the fp8 path's weights are (q - 8) 2^-9: 2^9 goes into the scale (exact)
          const float sc = half_bits_to_f32(sr0) * (FP8 ? 512.f : 1.f);
#pragma unroll
          for (int cc = 0; cc < kEpiCols / 32; ++cc) {
            uint32_t v[32];
            tc::tmem_ld32(taddr + cc * 32, v);
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              fma2(T[cc * 32 + j], T[cc * 32 + j + 1], sc, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        k0 = kend;
      }

      if (kTail && ok && !partials && !*abort_flag && t.tail >= 0) {
        // a K part of a last-wave tile: its fp32 sums, every row and output of
        // the tile (rows and outputs past the matrix hold finite values the
        // reduce pass never reads), 128 contiguous bytes per warp and token
        float* pp = p.tail_part + ((size_t)(t.tail * p.tail_splits + t.split) * BN + c0) * BM + 32 * q + lane;
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) pp[(size_t)j * BM] = T[j];
      } else if (ok && !partials && !*abort_flag && p.splits > 1) {
        // this split's fp32 sums; the reduce pass adds the splits, x_scale and bias
        float* pp = p.part + ((size_t)t.split * p.M + t.row0 + c0) * N + n;
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j)
          if (n_ok && t.row0 + c0 + j < t.row_end) pp[(size_t)j * N] = T[j];
      } else if (ok && !partials && !*abort_flag) {
        // Lanes 2i and 2i+1 hold outputs n and n+1 of the same tokens. For each
        // pair of tokens (j, j+1) they swap halves, so that the even lane stores
        // (n, n+1) of token j and the odd lane (n, n+1) of token j+1: one 4-byte
        // store per two outputs. N is even, so n + 1 < N whenever n < N.
        const float bsv = (p.bias != nullptr && n_ok) ? __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16) : 0.f;
        const int odd = lane & 1;
        const uint32_t sel = odd ? 0x3276u : 0x5410u;
        const int row_b = t.row0 + c0 + odd;
        uint32_t* yp = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + (size_t)row_b * N + (n & ~1));
#pragma unroll
        for (int j = 0; j < kEpiCols; j += 2) {
          const float2 xs2 = *reinterpret_cast<const float2*>(xs_s + c0 + j);
          const uint32_t v = pack_bf16x2(fmaf(xs2.x, T[j], bsv), fmaf(xs2.y, T[j + 1], bsv));
          const uint32_t o = prmt(v, __shfl_xor_sync(0xffffffffu, v, 1), sel);
          if (n_ok && row_b + j < t.row_end) *yp = o;
          yp += N;   // two rows on
        }
      }
    }
  }

  // ---- teardown: every warp arrives here; waits above are bounded ----
  if (*abort_flag) {
    // let copies and MMAs already issued land before the shared memory goes away
    const uint64_t t0 = tc::globaltimer_ns();
    while (tc::globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// widening pass: 8-bit activations -> exact fp16, k permuted per 8-chunk
// ---------------------------------------------------------------------------

template <bool FP8>
__global__ void __launch_bounds__(256) widen_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                    size_t n16) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = ld_stream_v4(src + i);
    dst[2 * i] = FP8 ? widen_e4m3(v.x, v.y) : widen_i8(v.x, v.y);
    dst[2 * i + 1] = FP8 ? widen_e4m3(v.z, v.w) : widen_i8(v.z, v.w);
  }
}

// ---------------------------------------------------------------------------
// split-K: y = bf16(x_scale[m] * (sum of the splits' fp32 partials) + bias[n])
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) split_reduce_kernel(const float4* __restrict__ part, int splits, int64_t M,
                                                           int N4, const float* __restrict__ x_scale,
                                                           const uint16_t* __restrict__ bias, uint2* __restrict__ y) {
  const int64_t total = M * N4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t m = i / N4;
    const int n = static_cast<int>(i - m * N4) * 4;
    float4 acc = part[i];
    for (int sp = 1; sp < splits; ++sp) {   // splits in order
      const float4 v = part[(size_t)sp * total + i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const float xs = x_scale[m];
    float b[4] = {0.f, 0.f, 0.f, 0.f};
    if (bias != nullptr) {
      const uint2 bb = *reinterpret_cast<const uint2*>(bias + n);
      b[0] = bf16_lo(bb.x);
      b[1] = bf16_hi(bb.x);
      b[2] = bf16_lo(bb.y);
      b[3] = bf16_hi(bb.y);
    }
    y[i] = make_uint2(pack_bf16x2(fmaf(xs, acc.x, b[0]), fmaf(xs, acc.y, b[1])),
                      pack_bf16x2(fmaf(xs, acc.z, b[2]), fmaf(xs, acc.w, b[3])));
  }
}

// The last wave's tiles: y = bf16(x_scale[m] * (sum of the tile's K parts, in
// order) + bias[n]) for the outputs of tail tiles first_tile .. first_tile +
// tail_tiles - 1, four outputs a thread.
__global__ void __launch_bounds__(256) tail_reduce_kernel(const float4* __restrict__ part, int tail_tiles, int parts,
                                                          int first_tile, int n_tiles, int64_t M, int N,
                                                          const float* __restrict__ x_scale,
                                                          const uint16_t* __restrict__ bias, uint2* __restrict__ y) {
  constexpr int kRow4 = BM / 4;   // float4 per tile row
  const int64_t total = (int64_t)tail_tiles * BN * kRow4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int tt = static_cast<int>(i / (BN * kRow4));
    const int rem = static_cast<int>(i - (int64_t)tt * BN * kRow4);
    const int r = rem / kRow4, c4 = rem - r * kRow4;
    const int tile = first_tile + tt;
    const int64_t m = (int64_t)(tile / n_tiles) * BN + r;
    const int n = (tile % n_tiles) * BM + 4 * c4;
    if (m >= M || n >= N) continue;   // N is a multiple of 8: n < N puts all four in range
    const size_t base = ((size_t)tt * parts * BN + r) * kRow4 + c4;
    float4 acc = part[base];
    for (int sp = 1; sp < parts; ++sp) {   // parts in order
      const float4 v = part[base + (size_t)sp * BN * kRow4];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const float xs = x_scale[m];
    float b[4] = {0.f, 0.f, 0.f, 0.f};
    if (bias != nullptr) {
      const uint2 bb = *reinterpret_cast<const uint2*>(bias + n);
      b[0] = bf16_lo(bb.x);
      b[1] = bf16_hi(bb.x);
      b[2] = bf16_lo(bb.y);
      b[3] = bf16_hi(bb.y);
    }
    y[(m * N + n) / 4] = make_uint2(pack_bf16x2(fmaf(xs, acc.x, b[0]), fmaf(xs, acc.y, b[1])),
                                    pack_bf16x2(fmaf(xs, acc.z, b[2]), fmaf(xs, acc.w, b[3])));
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t get_encoder(EncodeTiled* fn) {
  // looked up once; a function-local static is initialised once even when
  // several host threads get here together
  static const EncodeTiled cached = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiled>(f);
  }();
  if (cached == nullptr) return cudaErrorNotSupported;
  *fn = cached;
  return cudaSuccess;
}

cudaError_t encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiled fn = nullptr;
  cudaError_t e = get_encoder(&fn);
  if (e != cudaSuccess) return e;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int sm_count_w4a8() { return current_sm_count(); }

cudaError_t widen(const void* src, void* dst, int64_t rows, int64_t K, bool fp8, cudaStream_t s) {
  const size_t n16 = (size_t)rows * (size_t)K / 16;
  if (n16 == 0) return cudaSuccess;
  const size_t want = (n16 + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 152 * 16 ? want : 152 * 16);
  if (fp8)
    widen_kernel<true><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  else
    widen_kernel<false><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

// Split along K when the output tiles fill the 152 SMs of a GB300 poorly.
// Two forms, priced against no split with a tile weight t = K * 11.7 ns, the
// fp32 partials' traffic at 6.8 TB/s and 2 us for the reduce launch. (t was a
// tile's time at ~0.45 of the bf16 peak; tiles now take ~8.7 ns per k, but
// re-pricing with that dropped last-wave splits that still measured faster,
// 1,152 against 1,071 TOPS at 4096 x 11008 x 4096, so the weight stays.)
//  * every tile in s parts (1 to 4, at least 512 k each): ceil(tiles s / 152)
//    / s waves of t, plus 8 s M N bytes;
//  * the last wave only, when it is at most half full: the whole waves as they
//    are, then each of its r tiles in s parts (2 to 16, at least 256 k each):
//    ceil(r s / 152) waves of t / s, plus 2 * 4 r s 128 * 256 bytes, plus the
//    measured costs of that kernel instantiation (below).
// Parts are cut on 128-k stages and on group boundaries. At 4096 x 11008 x
// 4096 the second form only just wins (the tenth wave's 8 tiles), at 16384 x
// 3072 x 3072 it splits the last 16 tiles, and at 512 x 4096 x 4096 the
// first form takes two parts. Fixed figures keep the choice, and the
// workspace it needs, the same on every device.
constexpr int kSplitSms = 152;
struct Split {
  int splits, ksplit;                // every tile
  int tail_splits, tail_ksplit;      // the last wave's tiles
  int64_t full_tiles, tail_tiles;
};
Split choose_split(int64_t M, int64_t N, int64_t K, int32_t group) {
  const int64_t tiles = ((M + BN - 1) / BN) * ((N + BM - 1) / BM);
  int64_t gran = 128;   // stages of the fp16 path; the cut must also fall on a group boundary
  if (group < K) {
    int64_t a = gran, b = group;
    while (b) {
      const int64_t t = a % b;
      a = b;
      b = t;
    }
    gran = gran / a * group;   // lcm(128, group)
  }
  const double t_tile = static_cast<double>(K) * 11.7e-9, launch = 2e-6;
  // the part size for s parts, or 0 when the cut does not give exactly s parts
  auto part_k = [&](int sp) -> int64_t {
    const int64_t ks = ((K + sp - 1) / sp + gran - 1) / gran * gran;
    return (K + ks - 1) / ks == sp ? ks : 0;
  };
  const Split none{1, static_cast<int>(K), 0, 0, tiles, 0};
  const double none_t = static_cast<double>((tiles + kSplitSms - 1) / kSplitSms) * t_tile;
  Split best = none;
  double best_t = 1e30;   // the cheapest split; taken only if clearly cheaper than none
  for (int sp = 2; sp <= 4; ++sp) {
    if (K / sp < 512) break;
    const int64_t ks = part_k(sp);
    if (ks == 0) continue;
    const double waves = static_cast<double>((tiles * sp + kSplitSms - 1) / kSplitSms) / sp;
    const double t = waves * t_tile + 8.0 * sp * static_cast<double>(M) * static_cast<double>(N) / 6.8e12 + launch;
    if (t < best_t) {
      best_t = t;
      best = Split{sp, static_cast<int>(ks), 0, 0, tiles, 0};
    }
  }
  const int64_t r = tiles % kSplitSms;
  if (tiles > kSplitSms && r > 0 && 2 * r <= kSplitSms) {
    const int64_t full = tiles - r;
    // measured on GB300: the instantiation that splits the last wave runs its
    // whole tiles ~4% slower when the group is smaller than K, and the short
    // items' fill, drain and the reduce cost ~8 us in all
    const double slow = group < K ? 1.04 : 1.0, fixed = 8e-6;
    for (int sp = 2; sp <= 16; ++sp) {
      if (K / sp < 256) break;
      const int64_t ks = part_k(sp);
      if (ks == 0) continue;
      const double t = static_cast<double>(full / kSplitSms) * t_tile * slow +
                       static_cast<double>((r * sp + kSplitSms - 1) / kSplitSms) * t_tile / sp +
                       2.0 * 4.0 * r * sp * BM * BN / 6.8e12 + fixed;
      if (t < best_t) {
        best_t = t;
        best = Split{1, static_cast<int>(K), sp, static_cast<int>(ks), full, r};
      }
    }
  }
  return best_t < none_t * 0.97 ? best : none;   // a clear gain only
}

// Workspace bytes of the split partials for a plan.
size_t split_bytes(const Split& sp, int64_t M, int64_t N) {
  if (sp.splits > 1) return (size_t)sp.splits * M * N * 4;
  if (sp.tail_splits > 1) return (size_t)sp.tail_tiles * sp.tail_splits * BM * BN * 4;
  return 0;
}

template <bool FP8>
cudaError_t run_t(const W4A8Args& a, int mode, cudaStream_t s) {
  using C = Cfg<2, FP8>;
  // set on every call: the attribute belongs to the current device, and a
  // once-per-process flag would race between host threads
  cudaError_t e = cudaFuncSetAttribute(w4a8_tc_kernel<2, FP8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM);
  if (e != cudaSuccess) return e;
  const bool experts = mode == kExperts;
  // the activation operand TMA reads: the e4m3 codes themselves (fp8 path),
  // or the 8-bit codes widened once to exact fp16 in the workspace
  const void* act = a.act;
  if (!FP8) {
    e = a.prewidened ? cudaSuccess : widen(a.act, a.workspace, a.M, a.K, experts, s);
    if (e != cudaSuccess) return e;
    act = a.workspace;
  }

  const int n_tiles = static_cast<int>((a.N + BM - 1) / BM);

  Params p;
  memset(&p, 0, sizeof(p));
  // packed-word copies cover RAW_PER k-stages, or all of a short K (expert
  // mode needs K % 32 == 0, so its copy width is a multiple of 16 bytes)
  p.raw_rows = static_cast<int>(a.K / 8 < 32 ? a.K / 8 : 32);   // RAW_PER * BK / 8 = 32 in every configuration
  {
    // one sub-tile: 128 bytes of k (64 fp16 or 128 e4m3 values) x 256 rows
    const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)a.K * (FP8 ? 1 : 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(C::KS), BN};
    e = encode(&p.tm_act, FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, act, dims, strides,
               box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  if (experts) {
    // rows of 32 words (128 bytes) come 128-byte swizzled, so that the
    // converter threads, one output row each, read them without bank conflicts
    const cuuint64_t dims[3] = {(cuuint64_t)a.K / 8, (cuuint64_t)a.N, (cuuint64_t)a.E};
    const cuuint64_t strides[2] = {(cuuint64_t)a.K / 8 * 4, (cuuint64_t)a.N * (a.K / 8) * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(p.raw_rows), BM, 1};
    e = encode(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, a.qweight, dims, strides, box,
               p.raw_rows == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.K / 8};
    const cuuint64_t strides[1] = {(cuuint64_t)a.N * 4};
    const cuuint32_t box[2] = {BM, static_cast<cuuint32_t>(p.raw_rows)};
    e = encode(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, a.qweight, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (e != cudaSuccess) return e;
  p.w_scale = static_cast<const uint16_t*>(a.w_scale);
  p.x_scale = a.x_scale;
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.out = a.out;
  p.offsets = a.expert_offsets;
  p.E = a.E;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.group = a.group;
  p.mode = mode;
  p.status = a.status;

  // tile rows: dense, one per 256 rows; experts, an upper bound on the tiles
  // of all segments together (each expert's last tile may be partial)
  p.m_tiles = static_cast<int>(experts ? (a.M + BN - 1) / BN + a.E : (a.M + BN - 1) / BN);
  p.splits = 1;
  p.ksplit = p.K;
  p.tail_splits = 0;
  if (mode == kDenseY) {
    // split along K when the workspace holds the partial sums after the activations
    const Split sp = choose_split(a.M, a.N, a.K, a.group);
    const size_t extra = split_bytes(sp, a.M, a.N);
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + w4a8_workspace_bytes(a.M, a.K));
    if (extra > 0 && a.workspace_bytes >= w4a8_workspace_bytes(a.M, a.K) + extra) {
      if (sp.splits > 1) {
        p.splits = sp.splits;
        p.ksplit = sp.ksplit;
        p.part = part;
      } else {
        p.tail_splits = sp.tail_splits;
        p.tail_ksplit = sp.tail_ksplit;
        p.full_tiles = static_cast<int>(sp.full_tiles);
        p.tail_tiles = static_cast<int>(sp.tail_tiles);
        p.tail_part = part;
      }
    }
  }
  const long long y_tiles = (long long)p.m_tiles * p.splits;
  const long long total = p.tail_splits > 1 ? (long long)p.full_tiles + (long long)p.tail_tiles * p.tail_splits
                                            : y_tiles * n_tiles;
  if (total > INT32_MAX || y_tiles * n_tiles > INT32_MAX) return cudaErrorInvalidConfiguration;
  p.items = static_cast<int>(total);
  // persistent: one CTA per SM (the shared-memory rings fill an SM)
  const long long grid = total < sm_count_w4a8() ? total : sm_count_w4a8();
  if (p.tail_splits > 1) {
    if constexpr (!FP8) {   // dense only
      e = cudaFuncSetAttribute(w4a8_tc_kernel<2, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
      if (e != cudaSuccess) return e;
      w4a8_tc_kernel<2, false, true><<<static_cast<unsigned>(grid), kThreads, C::SMEM, s>>>(p, n_tiles,
                                                                                          static_cast<int>(y_tiles));
    }
  } else {
    w4a8_tc_kernel<2, FP8, false><<<static_cast<unsigned>(grid), kThreads, C::SMEM, s>>>(p, n_tiles,
                                                                                        static_cast<int>(y_tiles));
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.tail_splits > 1) {
    const int64_t n4 = (int64_t)p.tail_tiles * BN * (BM / 4);
    const int64_t want = (n4 + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(want < sm_count_w4a8() * 8 ? want : sm_count_w4a8() * 8);
    tail_reduce_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(p.tail_part), p.tail_tiles,
                                              p.tail_splits, p.full_tiles, n_tiles, a.M, static_cast<int>(a.N),
                                              a.x_scale, static_cast<const uint16_t*>(a.bias),
                                              static_cast<uint2*>(a.out));
    return cudaGetLastError();
  }
  if (p.splits == 1) return e;
  const int64_t n4 = a.M * (a.N / 4);
  const int64_t want = (n4 + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < sm_count_w4a8() * 8 ? want : sm_count_w4a8() * 8);
  split_reduce_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(p.part), p.splits, a.M,
                                             static_cast<int>(a.N / 4), a.x_scale,
                                             static_cast<const uint16_t*>(a.bias), static_cast<uint2*>(a.out));
  return cudaGetLastError();
}

cudaError_t run(const W4A8Args& a, int mode, cudaStream_t s) {
  return (mode == kExperts && a.fp8_act) ? run_t<true>(a, mode, s) : run_t<false>(a, mode, s);
}

}  // namespace

size_t w4a8_workspace_bytes(int64_t rows, int64_t K) { return static_cast<size_t>(rows) * static_cast<size_t>(K) * 2; }

size_t w4a8_workspace_bytes_split(int64_t M, int64_t N, int64_t K, int32_t group) {
  return w4a8_workspace_bytes(M, K) + split_bytes(choose_split(M, N, K, group), M, N);
}

cudaError_t launch_w4a8_dense(const W4A8Args& a, cudaStream_t s) {
  return run(a, a.partials ? kDensePartials : kDenseY, s);
}

cudaError_t launch_w4afp8_experts(const W4A8Args& a, cudaStream_t s) { return run(a, kExperts, s); }

bool w4afp8_fp8_path(int32_t group) { return group % 32 == 0; }

}  // namespace w4
