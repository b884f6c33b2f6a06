// Device-side helpers shared by the lrkv kernels (sm_103a): mbarrier / TMA
// primitives with bounded waits, the TMA swizzle address map, and the RoPE angle evaluation.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lrkv.h"

namespace lrkv {

constexpr int kBlock = 16;  // tokens per paged block

// ----------------------------------------------------------------- status
__device__ __forceinline__ void report(int32_t* st, int code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

// ------------------------------------------------------------- bf16 packs
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float f16_lo(uint32_t u) { return __half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xffffu))); }
__device__ __forceinline__ float f16_hi(uint32_t u) { return __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16))); }
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// bf16 pair -> fp16 pair (exact for values inside the fp16 range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  return pack_f16(bf16_lo(u), bf16_hi(u));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ warp MMA
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// --------------------------------------------------------- TMA swizzle
// Byte offset of (row, byte) inside a tile written by a TMA load whose rows
// are `row_bytes` long, under the tensor map's swizzle mode. The swizzle XORs
// the 16-byte chunk index (bits 4..) with address bits 7.. ; the tile base
// must be aligned to the swizzle atom (8 rows x span).
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t byte) {
  const uint32_t off = row * ROW_BYTES + byte;
  if constexpr (ROW_BYTES >= 128) return off ^ (((off >> 7) & 7u) << 4);
  else if constexpr (ROW_BYTES == 64) return off ^ (((off >> 7) & 3u) << 4);
  else if constexpr (ROW_BYTES == 32) return off ^ (((off >> 7) & 1u) << 4);
  else return off;
}

// ------------------------------------------------------- mbarrier / TMA
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of an mbarrier; gives up after ~`limit` polls
// (each try_wait already blocks for a hardware-defined slice), stores
// LRKV_ERR_TIMEOUT and returns false. Never spins forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* st,
                                          uint32_t limit = (1u << 22)) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  report(st, LRKV_ERR_TIMEOUT);
  return false;
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// 3-D tiled TMA load global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            int32_t c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// In-register Walsh-Hadamard transform of 32 values (Sylvester order,
// unnormalised). The d-point transform, d = 32 m, is H_m (x) H_32: group g of
// H_d v is fwht32 of sum_k (-1)^popc(g & k) v[32 k .. 32 k + 31].
__device__ __forceinline__ void fwht32(float* z) {
#pragma unroll
  for (int len = 1; len < 32; len <<= 1)
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if ((i & len) == 0) {
        const float a = z[i], b = z[i + len];
        z[i] = a + b;
        z[i + len] = a - b;
      }
}

// sqrt(d) of the compressed pool's value scale ||v|| / sqrt(d), d = 64 or 128
template <int D>
constexpr float kSqrtD = D == 128 ? 11.313708498984760f : 8.0f;

// Bits 0-3 of x moved to bits 0, 8, 16, 24 (x < 16).
__device__ __forceinline__ uint32_t spread4(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }

// Plain (untiled) bulk copy global -> shared: both addresses 16-byte aligned,
// `bytes` a multiple of 16, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// 4-D tiled TMA load global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------------ RoPE
// cos / sin of the rotary angle t * theta for integer positions t < 2^20.
// theta is given as an unevaluated sum th_hi + th_lo of two floats (the
// double-precision theta split on the host). The product t * th_hi is kept
// exactly as p + e (Dekker's two-product via FMA); the multiple of 2*pi is
// removed with a two-constant Cody-Waite reduction (Cody & Waite, "Software
// Manual for the Elementary Functions", 1980) whose first product is exact
// for |n| < 2^18. The reduced argument lies in about [-pi, pi] with an
// absolute error near 3e-7 rad; sincosf then evaluates it.
__device__ __forceinline__ float2 rope_cos_sin(int32_t t, float th_hi, float th_lo) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr float kC1 = static_cast<float>(kTwoPi);
  constexpr float kC2 = static_cast<float>(kTwoPi - static_cast<double>(kC1));
  constexpr float kInv = static_cast<float>(1.0 / kTwoPi);
  const float tf = static_cast<float>(t);
  const float p = tf * th_hi;
  float e = fmaf(tf, th_hi, -p);
  e = fmaf(tf, th_lo, e);
  const float n = rintf(p * kInv);
  float r = fmaf(-n, kC1, p);
  r = fmaf(-n, kC2, r);
  r += e;
  float s, c;
  sincosf(r, &s, &c);
  return make_float2(c, s);
}

// Same reduction, then the hardware sine/cosine approximation (absolute error
// near 2^-21 on [-pi, pi]); used where the result feeds fp16 arithmetic.
__device__ __forceinline__ float2 rope_cos_sin_fast(int32_t t, float th_hi, float th_lo) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr float kC1 = static_cast<float>(kTwoPi);
  constexpr float kC2 = static_cast<float>(kTwoPi - static_cast<double>(kC1));
  constexpr float kInv = static_cast<float>(1.0 / kTwoPi);
  const float tf = static_cast<float>(t);
  const float p = tf * th_hi;
  float e = fmaf(tf, th_hi, -p);
  e = fmaf(tf, th_lo, e);
  const float n = rintf(p * kInv);
  float r = fmaf(-n, kC1, p);
  r = fmaf(-n, kC2, r);
  r += e;
  float s, c;
  __sincosf(r, &s, &c);
  return make_float2(c, s);
}

// Per-launch RoPE frequencies theta_j = base^(-2j/d), j < d/2, split hi/lo.
struct RopeFreqs {
  float hi[64];
  float lo[64];
};

}  // namespace lrkv
