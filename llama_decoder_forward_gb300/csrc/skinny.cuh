// skinny.cuh - pieces shared by the decode-sized projections (M = B <= 64):
// mma.sync m16n8k16 and ldmatrix wrappers and the weight-row order of a
// narrow output unit for each epilogue.
#pragma once

#include "common.cuh"

namespace smol {

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

// Weight rows of unit u: NT groups of 8 consecutive rows, group g starting
// at unit_wrow(u, g).  The epilogues read the columns in this order.
template <int EPI, int NT>
__device__ __forceinline__ int unit_wrow(int u, int g) {
  if constexpr (EPI == kEpiQkvRope) {
    // head u/4, rotation pairs i0 .. i0+7 (i0 = 8*(u%4)): rows i0.. and 32+i0..
    return (u >> 2) * 64 + (u & 3) * 8 + g * 32;
  } else if constexpr (EPI == kEpiSwiglu) {
    // act columns a0 .. a0+15 (NT = 4) or a0 .. a0+7 (NT = 2): gate rows, then
    // up rows, of the 64-row block pair
    const int a0 = u * (NT * 4), blk = a0 >> 6, off = a0 & 63;
    return blk * 128 + (g / (NT / 2)) * 64 + off + (g % (NT / 2)) * 8;
  } else {
    return (u * NT + g) * 8;                        // output columns u*8*NT ..
  }
}

}  // namespace smol
