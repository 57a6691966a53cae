// msa_tcgen05.cuh -- inline PTX for the 5th-generation tensor core (tcgen05) on
// sm_103a: tensor-memory (TMEM) allocation, shared-memory matrix descriptors,
// the single-thread MMA, its completion commit to an mbarrier, and TMEM loads.
#pragma once

#include <stdint.h>

namespace msa {
namespace tc {

// ---- TMEM allocation (executed by one whole warp) ---------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_slot))),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// ---- ordering -----------------------------------------------------------------

__device__ __forceinline__ void fence_before_thread_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_thread_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Makes generic-proxy shared-memory writes visible to the async proxy (the
// tensor core reads its shared-memory operands through the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- descriptors ---------------------------------------------------------------

// Shared-memory matrix descriptor of a K-major operand stored with 128-byte
// swizzling: rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte
// offset), leading byte offset unused for this layout; descriptor version 1;
// layout type 2 = 128B swizzle.  `smem_addr` is a shared-window byte address
// (the base of the operand's first row, advanced by 32 bytes per K step).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  const uint64_t start = (smem_addr & 0x3FFFFu) >> 4;
  const uint64_t lbo = 16u >> 4;
  const uint64_t sbo = 1024u >> 4;
  return start | (lbo << 16) | (sbo << 32) | (1ull << 46) | (2ull << 61);
}

// Shared-memory matrix descriptor of an MN-major 8-bit operand stored with
// 128-byte swizzling, as a TMA tile of [K rows x 128 B] leaves it: each
// 128-byte row holds 128 consecutive M (or N) elements of one k, and 8-row
// groups along K are 1024 bytes apart.  The operand spans a single 128-byte
// atom along M, so both offsets can carry the K-group stride (the field that
// strides along M is then never used).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
  const uint64_t start = (smem_addr & 0x3FFFFu) >> 4;
  const uint64_t lbo = 1024u >> 4;
  const uint64_t sbo = 1024u >> 4;
  return start | (lbo << 16) | (sbo << 32) | (1ull << 46) | (2ull << 61);
}

// Shared-memory matrix descriptor of an MN-major 8-bit operand without
// swizzling: 8 x 16 B core matrices (8 consecutive k, 16 consecutive M or N
// elements each, 128 contiguous bytes), `k_stride` bytes apart along K
// (leading byte offset) and `mn_stride` bytes apart along M or N (stride byte
// offset).
__device__ __forceinline__ uint64_t interleave_mnmajor_desc(uint32_t smem_addr, uint32_t k_stride,
                                                            uint32_t mn_stride) {
  const uint64_t start = (smem_addr & 0x3FFFFu) >> 4;
  const uint64_t lbo = k_stride >> 4;
  const uint64_t sbo = mn_stride >> 4;
  return start | (lbo << 16) | (sbo << 32) | (1ull << 46) | (0ull << 61);
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B, fp32 accumulate,
// both operands K-major, shape M x N (M = 128, N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7)                                 // A format: E4M3
         | (0u << 10)                                // B format: E4M3
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// As idesc_e4m3_f32, with both A and B MN-major (bits 15 and 16).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32_mn(int M, int N) {
  return idesc_e4m3_f32(M, N) | (1u << 15) | (1u << 16);
}

// ---- MMA -----------------------------------------------------------------------

// D[tmem] (+)= A[smem] * B[smem]^T, issued by a single thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
      : "memory");
}

// ---- TMEM -> registers -------------------------------------------------------------

// 16 consecutive 32-bit columns of this thread's TMEM lane (the warp reads
// lanes 32*(warp%4) .. +31).
__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- registers -> TMEM -------------------------------------------------------------

// 32 consecutive 32-bit columns of this thread's TMEM lane (the warp writes
// lanes 32*(warp%4) .. +31).
__device__ __forceinline__ void st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
        "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
        "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
        "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace msa
