// Fifth-generation tensor core (tcgen05) helpers for sm_103a: tensor-memory
// allocation, shared-memory matrix descriptors, instruction descriptors, the
// f16 MMA with f32 accumulation in TMEM, completion commits and TMEM loads.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace moe {

// ---- tensor memory -------------------------------------------------------------
// One warp allocates `ncols` columns (a power of two >= 32) of the CTA's TMEM; the
// base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_addr(smem_dst)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- ordering between threads and the tensor core --------------------------------
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy writes to shared memory become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- descriptors -------------------------------------------------------------------
// Shared-memory matrix descriptor, K-major operand without swizzling: the operand
// is made of 8-row x 16-byte core matrices (8 f16 along K per row, rows 16 bytes
// apart); `lbo` is the byte distance between core matrices adjacent along K and
// `sbo` the distance between core matrices adjacent along M (or N).
__device__ __forceinline__ uint64_t smem_desc(const void* p, uint32_t lbo, uint32_t sbo) {
  const uint32_t a = smem_addr(p);
  uint64_t d = 0;
  d |= (uint64_t)((a & 0x3FFFFu) >> 4);           // bits 0-13: start address / 16
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;   // bits 16-29: leading-dimension byte offset / 16
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;   // bits 32-45: stride-dimension byte offset / 16
  d |= (uint64_t)1 << 46;                          // bits 46-48: fixed 0b001
  // bits 49-51 base offset 0, bit 52 relative offsets, bits 61-63 no swizzle
  return d;
}
// Instruction descriptor of kind::f16 with f16 A and B, f32 accumulator, both
// operands K-major, shape M x N (M = 64 or 128, N a multiple of 16 up to 256).
__host__ __device__ __forceinline__ uint32_t idesc_f16_f32(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                          // accumulator format: f32
  // A format (bits 7-9) and B format (bits 10-12): f16 = 0; K-major A and B (bits 15, 16) = 0
  d |= (uint32_t)(N >> 3) << 17;         // bits 17-22: N / 8
  d |= (uint32_t)(M >> 4) << 24;         // bits 24-28: M / 16
  return d;
}

// ---- MMA and completion ----------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T over K = 16; one thread issues it.
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u) : "memory");
}
// Arrive once on the mbarrier when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_addr(bar)) : "memory");
}

// ---- TMEM -> registers -------------------------------------------------------------------
// Warp w (w % 4 = q) reads TMEM lanes 32q .. 32q + 31, 16 consecutive 32-bit columns
// starting at column `col`: thread l gets lane 32q + l.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace moe
