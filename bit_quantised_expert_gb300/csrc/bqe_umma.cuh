// bqe_umma.cuh — thin wrappers for the 5th-generation tensor core path of
// sm_100/sm_103 (tcgen05): tensor-memory allocation, shared-memory matrix
// descriptors, the bf16 MMA with fp32 accumulation in tensor memory, commit
// to an mbarrier, and tensor-memory loads for the epilogue.
//
// Operand layout used throughout: K-major tiles of 64 bf16 per row (128 B),
// rows in groups of 8 forming 1024-byte atoms, the 16-byte chunks of row r
// stored at chunk position (c XOR (r mod 8)) — the 128-byte swizzle.  Tiles
// start on 1024-byte boundaries.
#pragma once

#include <stdint.h>

#include "bqe_internal.cuh"

namespace bqe {

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a swizzled K-major tile.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t c) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

#ifdef __CUDACC__
// Shared-memory matrix descriptor (tcgen05): start address >> 4 in bits 0-13,
// leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45,
// descriptor version 1 in bits 46-47, base offset 0, swizzle mode in 61-63
// (2 = 128-byte swizzle).  For K-major 128B-swizzled tiles the stride between
// 8-row atoms is 1024 bytes; the leading offset is unused (one atom spans K).
__device__ __forceinline__ uint64_t umma_desc_sw128(const void* smem_tile) {
  const uint32_t a = smem_u32(smem_tile);
  uint64_t d = 0;
  d |= (uint64_t)((a >> 4) & 0x3FFFu);
  d |= (uint64_t)(16u >> 4) << 16;     // leading byte offset (ignored for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;   // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B
// of one type (bits 7-9 and 10-12: 0 fp16, 1 bf16), both K-major (bits 15,
// 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ __forceinline__ uint32_t umma_idesc_f16(int M, int N, bool bf16) {
  const uint32_t t = bf16 ? 1u : 0u;
  return (1u << 4) | (t << 7) | (t << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N) { return umma_idesc_f16(M, N, true); }

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction (M x N x 16), fp16 or bf16
// operands as the instruction descriptor says.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory writes by ordinary stores become visible to the tensor core
// (async proxy) after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 lanes x 16 columns of fp32 from tensor memory, waiting for the load in
// the same statement: thread = lane (row), v[i] = column (taddr's column) + i.
// The warp may only address its own quarter of the lanes (32 * (warp % 4)).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
#endif

}  // namespace bqe
