// Inline-PTX helpers for the 5th-generation tensor cores of sm_103a (tcgen05): tensor-memory
// allocation, shared-memory matrix descriptors, the kind::f16 instruction descriptor, the MMA, its
// commit to an mbarrier, and tensor-memory loads and stores.
//
// Operand layouts used here (16-bit elements, E = elements per swizzle row: 64 with the 128-byte
// swizzle, 32 with the 64-byte swizzle):
//   K-major (rows = M or N, K contiguous): K is cut into atoms of E elements; atom u of an R-row
//     operand is a region of R rows x (2 E) bytes, row r at r * 2E, its 16-byte chunk c stored at
//     chunk c ^ ((r % 8) for 128 B, (r / 2) % 4 for 64 B), i.e. the byte offset's bits [4..] XORed
//     with its bits [7..].  Groups of 8 rows are SBO = 16 E bytes apart; one MMA reads 16 K
//     elements (32 bytes), so K step k starts at atom (16 k) / E, byte (32 k) % (2 E).
//   MN-major (K rows, N contiguous; the V operand): N is cut into atoms of E elements, each a
//     region of K rows x 2E bytes laid out like the K-major atom (a row is one k); N-atoms are
//     LBO = region bytes apart, groups of 8 k rows SBO = 16 E bytes apart; K step k starts 16 k
//     rows on (32 E k bytes).
// Both are the layouts the tensor-memory-access copies produce with the matching swizzle for a
// box whose inner extent is E elements.  Region bases are 1024-byte aligned.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace pkv {
namespace tc {

constexpr uint32_t kLayoutSwizzle128 = 2;
constexpr uint32_t kLayoutSwizzle64 = 4;

// Shared-memory matrix descriptor: start address, leading and stride byte offsets (16-byte units),
// descriptor version 1 (bit 46), base offset 0 (atoms aligned to the swizzle repeat), layout type.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)(layout & 7u) << 61);
}

// Swizzle layout type for atoms of E elements.
__host__ __device__ constexpr uint32_t layout_for(int E) { return E == 64 ? kLayoutSwizzle128 : kLayoutSwizzle64; }

// Byte offset of element (r, k) inside a K-major operand of R rows (atoms of E elements), and of the
// 16-byte chunk holding elements k..k+7 (k a multiple of 8).
__host__ __device__ constexpr uint32_t kmajor_offset(int R, int E, int r, int k) {
  const uint32_t o = (uint32_t)(r * E * 2 + (k % E) * 2);
  const uint32_t mask = E == 64 ? 7u : 3u;
  return (uint32_t)((k / E) * R * E * 2) + (o ^ (((o >> 7) & mask) << 4));
}

// Instruction descriptor of kind::f16: fp16 A and B, fp32 accumulator, dense; A K-major, B K-major
// or MN-major; N >> 3 in bits 17..22, M >> 4 in bits 24..28.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M rows = lanes, K along the columns, two 16-bit elements per
// 32-bit column, the lower K index in the low half) read from tensor memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Allocate `ncols` (a power of two >= 32) tensor-memory columns; the whole warp executes it and the
// base address lands in *dst (shared memory).
__device__ __forceinline__ void alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive 32-bit columns of the calling thread's lane (the warp reads lanes
// 32 * (warp % 4) .. + 31; taddr carries the lane in bits 16..31 and the column in bits 0..15).
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// 16 consecutive 32-bit columns (x16 shape), as ld32/st32.
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

}  // namespace tc
}  // namespace pkv
