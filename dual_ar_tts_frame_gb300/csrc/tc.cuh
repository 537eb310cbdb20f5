// PTX wrappers for the 5th-generation tensor cores (tcgen05: MMA with the
// accumulator in tensor memory) and for tiled tensor copies (TMA), sm_103a.
//
// Descriptor formats follow the PTX ISA's tcgen05 chapter:
//  * shared-memory matrix descriptor (64 bits): start address >> 4 in bits
//    0-13, leading-dimension byte offset >> 4 in bits 16-29, stride-dimension
//    byte offset >> 4 in bits 32-45, the fixed version 1 in bits 46-47, base
//    offset 0 (1024-byte aligned swizzle atoms) in bits 49-51, the swizzle
//    mode in bits 61-63 (2 = 128-byte swizzle);
//  * instruction descriptor for kind::f16 (32 bits): D format in bits 4-5
//    (1 = f32), A and B formats in bits 7-9 and 10-12 (1 = bf16), A/B major
//    in bits 15/16 (0 = K-major), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace dualar {

// ---- descriptors --------------------------------------------------------------
// K-major operand tile whose rows are 128 bytes (64 bf16), written by a TMA
// copy with 128-byte swizzle: 8-row atoms of 1024 bytes, one after another.
DEVI uint64_t smem_desc_sw128(const void* tile) {
  const uint32_t a = smem_addr(tile);
  uint64_t d = 0;
  d |= static_cast<uint64_t>((a & 0x3FFFFu) >> 4);          // start address
  d |= static_cast<uint64_t>(16u >> 4) << 16;                // leading byte offset (unused for this layout)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;              // stride byte offset: one 8-row atom
  d |= static_cast<uint64_t>(1) << 46;                       // version
  d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ---- tensor memory ---------------------------------------------------------------
// Executed by one whole warp.  The allocated column base is written to *dst.
DEVI void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
DEVI void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major; issued by one thread.
DEVI void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// The mbarrier receives one arrival once every MMA this thread issued so far
// has completed (its shared-memory operands may then be overwritten).
DEVI void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 32 lanes x 16 columns of 32-bit values: lane i of the warp gets row
// (lane base + i), columns col .. col+15.
DEVI void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// The same without the wait: registers are valid after tmem_wait_ld().
DEVI void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
DEVI void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- tiled tensor copies (TMA) -----------------------------------------------------
// 2-D tile global -> shared, completing on an mbarrier.  x (innermost, in
// elements) must keep x * element size a multiple of 16 bytes.
DEVI void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
DEVI void tma_load_2d_hint(void* dst, const void* tmap, int x, int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 3-D tile shared -> global (bulk async group); the source must stay
// untouched until the group has been waited for.
DEVI void tma_store_3d(const void* tmap, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
               "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
DEVI void tma_store_3d_hint(const void* tmap, const void* src, int x, int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(tmap),
      "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}
DEVI void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until this thread's committed bulk stores have completed (written).
DEVI void tma_store_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Request a 2-D tile of the tensor into L2 only (no completion to wait for).
DEVI void tma_prefetch_l2_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
               : "memory");
}

DEVI void tma_prefetch_l2_2d_hint(const void* tmap, int x, int y, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile.L2::cache_hint [%0, {%1, %2}], %3;" ::"l"(tmap),
               "r"(x), "r"(y), "l"(policy)
               : "memory");
}

}  // namespace dualar
