// Fifth-generation tensor core (tcgen05) and tensor memory (TMEM) building
// blocks for sm_100-family GPUs (sm_103a here), as inline PTX:
//   * TMEM allocation by one warp, released before the CTA exits;
//   * tcgen05.mma kind::f16 (bf16 x bf16 -> fp32 accumulators in TMEM), its
//     shared-memory matrix descriptors (K-major operands in the 128-byte
//     swizzle that a TMA tile load writes) and its instruction descriptor;
//   * tcgen05.commit (an mbarrier arrival once the issued MMAs are done)
//     and tcgen05.ld of accumulator columns into registers.
#pragma once

#include <cstdint>

#include "tma.cuh"

namespace gq {
namespace tc {

// Allocate `ncols` TMEM columns (a power of two, 32..512) for the CTA; the
// base address is written to *dst (shared memory).  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations against thread synchronisation.
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory descriptor of a K-major operand tile stored as TMA writes it
// with the 128-byte swizzle: rows of 128 bytes (64 bf16 along K), 8-row
// atoms of 1024 bytes one after another along M/N.  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (bits 16-29; unused for
// swizzled K-major layouts, 1), stride byte offset >> 4 (bits 32-45: 1024
// bytes between 8-row atoms), descriptor version 1 (bits 46-47), base offset
// 0 (bits 49-51: atoms 1024-byte aligned), layout type 2 = 128-byte swizzle
// (bits 61-63).  The K-th 16-element slice of the 64-element row starts 32 K
// bytes further (start address + 2 K).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3
// in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D (TMEM) = A * B^T (+ D when accumulate != 0), issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread has
// completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane (warp
// w of a warpgroup reads lanes 32 (w % 4) .. 32 (w % 4) + 31; taddr holds
// that lane base in bits 16-31 and the first column in bits 0-15).  Whole
// warp; the values are valid after wait_ld.
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace gq
