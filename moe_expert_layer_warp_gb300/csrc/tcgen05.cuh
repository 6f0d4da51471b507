// tcgen05.cuh — inline-PTX helpers for the 5th-generation tensor cores on
// sm_103a: shared-memory matrix descriptors, the instruction descriptor of a
// bf16 × bf16 → fp32 MMA, tcgen05.mma / commit, tensor-memory (TMEM)
// allocation and loads.
//
// Operand layout used throughout: K-major tiles of rows × 64 bf16 (128 bytes
// per row) written by TMA with the 128-byte swizzle, tile base 1024-byte
// aligned; 8-row groups are 1024 bytes apart. A K-step of 16 elements is
// selected by advancing the descriptor's start address by 32 bytes.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace moe {
namespace umma {

// Shared-memory descriptor of a K-major, 128-byte-swizzled operand tile.
MOE_DEV uint64_t desc_sw128(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_byte_addr >> 4) & 0x3FFFu);  // start address, 16-byte units
  d |= (uint64_t)1 << 16;                            // leading-dim offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                  // stride between 8-row groups
  d |= (uint64_t)1 << 46;                            // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                            // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with A = B = bf16, D = fp32, both K-major,
// M × N tile (M = 128; N a multiple of 16 up to 256).
MOE_DEV uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                        // D format: fp32
         | (1u << 7)                      // A format: bf16
         | (1u << 10)                     // B format: bf16
         | ((uint32_t)(N >> 3) << 17)     // N / 8
         | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// D[tmem] (+)= A[smem] · B[smem]ᵀ; accumulate when `acc` != 0. One thread.
MOE_DEV void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed (its shared-memory reads done, its TMEM writes visible).
MOE_DEV void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Warp-wide: allocate `ncols` TMEM columns (power of two ≥ 32); the base
// address is written to *dst in shared memory.
MOE_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

MOE_DEV void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

MOE_DEV void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide: thread t receives TMEM lane (lane_base + t), 16 consecutive
// 32-bit columns starting at the address's column. lane_base must be the
// warp's quadrant, 32·(warp % 4), encoded in the address's upper 16 bits.
MOE_DEV void ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

MOE_DEV void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace umma
}  // namespace moe
