// Device-side helpers shared by the kernels of the int4-weight linear layer.
// sm_103a only: every helper is plain CUDA or inline PTX for that target.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "w4.h"

#define W4_DEV __device__ __forceinline__

namespace w4 {

// ---------------------------------------------------------------------------
// device status word (bounded waits record W4_ERR_TIMEOUT here)
// ---------------------------------------------------------------------------

// Sets *status to `code` once (the first error wins).
W4_DEV void report(unsigned int* status, unsigned int code) {
  if (status != nullptr) atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------------------
// bit helpers
// ---------------------------------------------------------------------------

W4_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & b) | c as one LOP3.
W4_DEV uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// (a & b) ^ c as one LOP3.
W4_DEV uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// m ? a : b, bit by bit, as one LOP3.
W4_DEV uint32_t select_bits(uint32_t m, uint32_t a, uint32_t b) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
  return d;
}

// d0 += a * b0 and d1 += a * b1, two fp32 FMAs (round to nearest) in one
// packed instruction.
W4_DEV void fma2(float& d0, float& d1, float a, float b0, float b1) {
  asm("{.reg .b64 d, x, y; mov.b64 d, {%0, %1}; mov.b64 x, {%2, %2}; mov.b64 y, {%3, %4}; "
      "fma.rn.f32x2 d, x, y, d; mov.b64 {%0, %1}, d;}"
      : "+f"(d0), "+f"(d1) : "f"(a), "f"(b0), "f"(b1));
}

W4_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
W4_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// fp32 -> bf16 bits, round to nearest even (finite inputs).
W4_DEV uint32_t f32_to_bf16_bits(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

W4_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

W4_DEV float half_bits_to_f32(uint32_t h16) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(static_cast<uint16_t>(h16)));
  return f;
}

// ---------------------------------------------------------------------------
// 8-bit activation codes -> exact fp16, k permuted per 8-chunk
// (the operand layout of the W4A8 tensor-core kernel)
// ---------------------------------------------------------------------------

// int8 bytes b0..b7 -> fp16 (b0,b4,b1,b5,b2,b6,b3,b7). (b ^ 0x80) in the low
// mantissa byte of 1024 is 1152 + b; subtracting 1152 leaves b exactly.
W4_DEV uint32_t i8pair(uint32_t u0, uint32_t u1, uint32_t sel) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(and_xor(prmt(u0, u1, sel), 0x00FF00FFu, 0x64806480u)),
      "r"(0x64806480u));
  return d;
}

W4_DEV uint4 widen_i8(uint32_t u0, uint32_t u1) {
  return make_uint4(i8pair(u0, u1, 0x0400u), i8pair(u0, u1, 0x0501u), i8pair(u0, u1, 0x0602u),
                    i8pair(u0, u1, 0x0703u));
}

W4_DEV uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t d;
  asm("{.reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t;}" : "=r"(d) : "r"(two_codes));
  return d;
}

// e4m3 codes b0..b7 -> fp16 (b0,b4,b1,b5,b2,b6,b3,b7), exactly.
W4_DEV uint4 widen_e4m3(uint32_t u0, uint32_t u1) {
  const uint32_t a = prmt(u0, u1, 0x5140u), b = prmt(u0, u1, 0x7362u);
  return make_uint4(e4m3x2_to_f16x2(a & 0xFFFFu), e4m3x2_to_f16x2(a >> 16), e4m3x2_to_f16x2(b & 0xFFFFu),
                    e4m3x2_to_f16x2(b >> 16));
}

// ---------------------------------------------------------------------------
// per-token quantization: the codes of the IEEE quotient fl(x / s)
// ---------------------------------------------------------------------------

W4_DEV uint32_t e4m3x2_rn(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

// Packed fp32 pairs: one f32x2 instruction for two results, round to nearest.
W4_DEV void mul2(float& d0, float& d1, float a0, float a1, float b) {
  asm("{.reg .b64 d, x, y; mov.b64 x, {%2, %3}; mov.b64 y, {%4, %4}; mul.rn.f32x2 d, x, y; mov.b64 {%0, %1}, d;}"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b));
}
W4_DEV void add2(float& d0, float& d1, float a0, float a1, float b) {
  asm("{.reg .b64 d, x, y; mov.b64 x, {%2, %3}; mov.b64 y, {%4, %4}; add.rn.f32x2 d, x, y; mov.b64 {%0, %1}, d;}"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b));
}

// Halfwise larger magnitude of two words of two 16-bit floats (bf16, or fp16
// with kF16); the sign bits of the result carry no meaning.
template <bool kF16>
W4_DEV uint32_t absmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  if (kF16)
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The codes of the IEEE quotient fl(x / s). With r = fl(1 / s) and the two
// per-row factors rlo = fl(r (1 - 2^-20)), rhi = fl(r (1 + 2^-20)), the products
// fl(x rlo) and fl(x rhi) are (x / s)(1 -+ 2^-20)(1 + e) with |e| < 3.1 * 2^-24,
// while fl(x / s) = (x / s)(1 + e'), |e'| <= 2^-24: fl(x / s) lies between the
// two products (a tiny x whose products underflow lies with them below every
// rounding boundary). Rounding onto the int8 or e4m3 grid is monotone, so
// where both products give the same code, that is the code of fl(x / s). An
// 8-element chunk in which some element's ends differ takes the IEEE divide
// for all 8: a value within about 2^-20 of a rounding boundary, or a
// near-exact tie, which bf16 inputs make common (0.2 to 0.3% of elements:
// x / amax is a ratio of two 8-bit mantissas). Measured on GB300 against a
// test per pair of elements, and against a per-chunk test with per-pair
// divides inside: one test per chunk is fastest on activations with outlier
// channels and within 5% on tie-heavy rows without them.
//
// A subnormal s (amax below 2^-126 times the code maximum) breaks the relative
// bounds and may overflow 1 / s: there rlo = 0 and rhi = inf, whose ends differ
// on every element, so such rows are quantized with the divide throughout.
struct QuotientBracket {
  float s, rlo, rhi;
};

W4_DEV QuotientBracket quotient_bracket(float s) {
  if (s < 1.17549435e-38f) return {s, 0.f, __int_as_float(0x7f800000)};
  const float r = __frcp_rn(s);
  return {s, r * 0.99999904632568359375f, r * 1.00000095367431640625f};
}

// Activation halves of a word as fp32 (exact): bf16, or fp16 (kF16).
template <bool kF16>
W4_DEV float act_lo(uint32_t w) {
  return kF16 ? half_bits_to_f32(w & 0xFFFFu) : bf16_lo(w);
}
template <bool kF16>
W4_DEV float act_hi(uint32_t w) {
  return kF16 ? half_bits_to_f32(w >> 16) : bf16_hi(w);
}

// The int8 codes clamp(rne(fl(x / s)), -127, 127) of the 8 activations of a
// 16-byte chunk, element i in byte i. Adding 1.5 * 2^23 rounds a value below
// 2^22 in magnitude to an integer (round to nearest even) and leaves that
// integer in the low bits of the sum, its low byte the two's-complement code.
// On the bracket path |x / s| <= 127 (1 + 2^-22) (s normal, |x| <= amax), so
// no code leaves [-127, 127] and no clamp is needed there.
template <bool kF16>
W4_DEV uint2 quant_int8_chunk(const uint4& v, const QuotientBracket& b) {
  constexpr float kMagic = 12582912.f;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[8];
  uint32_t diff = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float xl = act_lo<kF16>(w[i]), xh = act_hi<kF16>(w[i]);
    float l0, l1, h0, h1;
    mul2(l0, l1, xl, xh, b.rlo);
    mul2(h0, h1, xl, xh, b.rhi);
    add2(l0, l1, l0, l1, kMagic);
    add2(h0, h1, h0, h1, kMagic);
    c[2 * i] = __float_as_uint(l0);
    c[2 * i + 1] = __float_as_uint(l1);
    diff |= (c[2 * i] ^ __float_as_uint(h0)) | (c[2 * i + 1] ^ __float_as_uint(h1));
  }
  if (diff != 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float ql = fmaxf(-127.f, fminf(127.f, __fdiv_rn(act_lo<kF16>(w[i]), b.s)));
      const float qh = fmaxf(-127.f, fminf(127.f, __fdiv_rn(act_hi<kF16>(w[i]), b.s)));
      c[2 * i] = __float_as_uint(ql + kMagic);
      c[2 * i + 1] = __float_as_uint(qh + kMagic);
    }
  }
  return make_uint2(prmt(prmt(c[0], c[1], 0x0040u), prmt(c[2], c[3], 0x0040u), 0x5410u),
                    prmt(prmt(c[4], c[5], 0x0040u), prmt(c[6], c[7], 0x0040u), 0x5410u));
}

// The e4m3 codes (satfinite, round to nearest even) of fl(x / s) for the 8
// activations of a 16-byte chunk, element i in byte i.
template <bool kF16>
W4_DEV uint2 quant_e4m3_chunk(const uint4& v, const QuotientBracket& b) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t p[4];
  uint32_t diff = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float xl = act_lo<kF16>(w[i]), xh = act_hi<kF16>(w[i]);
    float l0, l1, h0, h1;
    mul2(l0, l1, xl, xh, b.rlo);
    mul2(h0, h1, xl, xh, b.rhi);
    p[i] = e4m3x2_rn(l0, l1);
    diff |= p[i] ^ e4m3x2_rn(h0, h1);
  }
  if (diff != 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      p[i] = e4m3x2_rn(__fdiv_rn(act_lo<kF16>(w[i]), b.s), __fdiv_rn(act_hi<kF16>(w[i]), b.s));
  }
  return make_uint2(prmt(p[0], p[1], 0x5410u), prmt(p[2], p[3], 0x5410u));
}

// ---------------------------------------------------------------------------
// global memory access
// ---------------------------------------------------------------------------

// 16-byte streaming load that bypasses L1 (each weight byte is read once).
W4_DEV uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

W4_DEV uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// 16-byte load cached in L2 only: sees data another grid wrote, even one
// that finished while this grid was already running.
W4_DEV uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

W4_DEV uint2 ld_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// mbarrier with bounded waits
// ---------------------------------------------------------------------------

W4_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

W4_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count));
}

W4_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

W4_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("{.reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0];}" :: "r"(smem_addr(bar)) : "memory");
}

W4_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{.reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;}"
               :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

W4_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, polling at most `limit`
// times. Returns false (after recording W4_ERR_TIMEOUT) if it never does.
W4_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit, unsigned int* status) {
  for (long long i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  report(status, W4_ERR_TIMEOUT);
  return false;
}

}  // namespace w4
