// tcgen05 (5th-generation tensor core) primitives for sm_103a, as inline PTX:
// tensor-memory (TMEM) allocation, shared-memory matrix descriptors, the
// instruction descriptor of kind::f16 MMAs, MMA issue with operand A from
// shared memory or from TMEM, completion tracking through mbarriers, and the
// 32x32b TMEM load / store shapes (thread t of a warp <-> TMEM lane
// 32 * (warp % 4) + t).
#pragma once

#include <stdint.h>

namespace lrkv {
namespace tc {

// ------------------------------------------------------------ descriptors
// Swizzle codes of the shared-memory descriptor (bits 61..63) for rows of
// `span` bytes laid out as the TMA writes them (8-row swizzle atoms).
__host__ __device__ constexpr uint32_t swizzle_code(int span) {
  return span == 128 ? 2u : span == 64 ? 4u : span == 32 ? 6u : 0u;
}

// Shared-memory matrix descriptor: start address, leading-dimension and
// stride-dimension byte offsets (all >> 4), descriptor version 1, swizzle.
// K-major operands: SBO = bytes between 8-row groups, LBO unused (16).
// MN-major operands: LBO = bytes between swizzle-atom columns along M/N,
// SBO = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t swz) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swz) << 61;
  return d;
}

// Instruction descriptor of a kind::f16 MMA with fp32 accumulation:
// A/B fp16 (ab_bf16 = false) or bf16, K-major (false) or MN-major operands.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool ab_bf16, bool a_mn, bool b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(ab_bf16) << 7) | (static_cast<uint32_t>(ab_bf16) << 10) |
         (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, issued by one thread.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with operand A read from TMEM (16-bit elements packed two per column).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the mbarrier when every MMA issued so far by this thread
// has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// ---------------------------------------------------------- TMEM alloc
// Warp-wide: allocates `ncols` columns (power of two >= 32) and writes the
// base address to shared memory at `slot`.
__device__ __forceinline__ void alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// ------------------------------------------------------- TMEM load/store
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

#define LRKV_R8(a, o) "=r"(a[o + 0]), "=r"(a[o + 1]), "=r"(a[o + 2]), "=r"(a[o + 3]), \
                      "=r"(a[o + 4]), "=r"(a[o + 5]), "=r"(a[o + 6]), "=r"(a[o + 7])
#define LRKV_W8(a, o) "r"(a[o + 0]), "r"(a[o + 1]), "r"(a[o + 2]), "r"(a[o + 3]), \
                      "r"(a[o + 4]), "r"(a[o + 5]), "r"(a[o + 6]), "r"(a[o + 7])

// 32 lanes x N consecutive 32-bit columns: thread t gets lane t, columns
// taddr.col .. +N-1 in v[0..N-1].
__device__ __forceinline__ void ld_x2(uint32_t taddr, uint32_t (&v)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];\n"
               : "=r"(v[0]), "=r"(v[1])
               : "r"(taddr));
}
__device__ __forceinline__ void ld_x4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr));
}
__device__ __forceinline__ void ld_x8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : LRKV_R8(v, 0)
               : "r"(taddr));
}
__device__ __forceinline__ void ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : LRKV_R8(v, 0), LRKV_R8(v, 8)
      : "r"(taddr));
}
__device__ __forceinline__ void ld_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : LRKV_R8(v, 0), LRKV_R8(v, 8), LRKV_R8(v, 16), LRKV_R8(v, 24)
      : "r"(taddr));
}
__device__ __forceinline__ void st_x2(uint32_t taddr, const uint32_t (&v)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};\n" ::"r"(taddr), "r"(v[0]), "r"(v[1])
               : "memory");
}
__device__ __forceinline__ void st_x4(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3])
               : "memory");
}
__device__ __forceinline__ void st_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr),
               LRKV_W8(v, 0)
               : "memory");
}
__device__ __forceinline__ void st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      LRKV_W8(v, 0), LRKV_W8(v, 8)
      : "memory");
}
__device__ __forceinline__ void st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      LRKV_W8(v, 0), LRKV_W8(v, 8), LRKV_W8(v, 16), LRKV_W8(v, 24)
      : "memory");
}
#undef LRKV_R8
#undef LRKV_W8

// N consecutive columns, N in {2, 4, 8, 16, 32}.
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, uint32_t (&v)[N]) {
  if constexpr (N == 2) ld_x2(taddr, v);
  else if constexpr (N == 4) ld_x4(taddr, v);
  else if constexpr (N == 8) ld_x8(taddr, v);
  else if constexpr (N == 16) ld_x16(taddr, v);
  else ld_x32(taddr, v);
}
template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
  if constexpr (N == 2) st_x2(taddr, v);
  else if constexpr (N == 4) st_x4(taddr, v);
  else if constexpr (N == 8) st_x8(taddr, v);
  else if constexpr (N == 16) st_x16(taddr, v);
  else st_x32(taddr, v);
}

}  // namespace tc
}  // namespace lrkv
