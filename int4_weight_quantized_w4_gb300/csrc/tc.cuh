// Inline-PTX wrappers for the Blackwell tensor-core path (sm_103a):
// TMA tile loads, tcgen05 TMEM allocation / MMA / commit / loads, the fences
// that order them, and a time-bounded mbarrier wait.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace w4 {
namespace tc {

W4_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar`. Gives up after `limit_ns` of wall time,
// or as soon as another thread of the CTA has raised *abort; on its own
// timeout it records W4_ERR_TIMEOUT and raises *abort. Returns true when the
// phase completed.
// One poll that lets the hardware suspend the thread for up to `hint_ns`
// (it resumes as soon as the phase completes), so waiting warps do not take
// issue slots from the warps that do the work.
W4_DEV bool try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p;}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

W4_DEV bool wait(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned int* status,
                 uint64_t limit_ns, uint32_t hint_ns = 1000) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (try_wait_suspend(bar, parity, hint_ns)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      report(status, W4_ERR_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion counted on an mbarrier)
// ---------------------------------------------------------------------------

W4_DEV void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

W4_DEV void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      :: "r"(smem_addr(smem_dst)), "l"(tmap), "r"(smem_addr(bar)), "r"(c0), "r"(c1) : "memory");
}

W4_DEV void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(smem_addr(smem_dst)), "l"(tmap), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

// Contiguous global -> shared copy of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completion counted on `bar`.
W4_DEV void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_addr(smem_dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// Starts moving a tile into L2 without a shared-memory destination or a
// completion to wait for (a later tma_load_2d of it then hits in L2).
W4_DEV void tma_prefetch_l2_2d(const void* tmap, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               :: "l"(tmap), "r"(c0), "r"(c1) : "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads its operands through it).
W4_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ---------------------------------------------------------------------------

// Whole warp: allocate `ncols` TMEM columns; the base address lands in *dst.
W4_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_addr(dst)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

W4_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// Eight 32-bit columns of a warp's TMEM lane quadrant, one value per lane
// and column; tmem_wait_st waits until the thread's stores have completed.
W4_DEV void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
W4_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

W4_DEV void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
W4_DEV void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout: rows of 128 bytes, 8-row atoms of 1024 bytes (stride between atoms
// 1024 B), 16-byte chunks XOR-swizzled by row % 8. The atom base must be
// 1024-byte aligned; advancing K inside the atom adds bytes/16 to the start.
W4_DEV uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);   // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading-dim offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride-dim offset
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                   // swizzle: 128 B
  return d;
}

// Instruction descriptor with fp32 accumulator, both operands K-major, shape
// M x N, A and B format code 0: fp16 under kind::f16, e4m3 under
// kind::f8f6f4.
constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                                // D format: f32
         | (0u << 7) | (0u << 10)                 // A, B format: f16
         | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}

W4_DEV void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{.reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// The same MMA on 8-bit floats (kind::f8f6f4; the formats come from idesc):
// M x N x 32 per instruction, fp32 accumulator.
W4_DEV void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{.reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive (once) on `bar` when every tcgen05 op this thread issued so far is done.
W4_DEV void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_addr(bar)) : "memory");
}

// Warp-wide: 32 lanes x 32 consecutive 32-bit columns from TMEM. The wait is
// in the same asm statement so no use of v can be scheduled before it.
W4_DEV void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr) : "memory");
}

}  // namespace tc
}  // namespace w4
