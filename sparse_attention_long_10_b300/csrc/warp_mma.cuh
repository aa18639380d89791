// warp_mma.cuh -- warp-level tensor-core helpers (mma.sync m16n8k16, bf16 in,
// fp32 accumulate) and ldmatrix loads from 128-byte-swizzled TMA tiles.
//
// Used by the decode kernels, whose contractions have only 16 rows (the query
// heads of one GQA group against one query token): a 16 x 8 x 16 warp MMA
// fits that shape exactly, and those kernels are bound by HBM, not by the
// tensor pipe.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace nsa {

// D += A * B;  A: 16x16 bf16 row-major fragment, B: 16x8 bf16 "col" fragment.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices; lane l supplies the row address of matrix l/8.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Same, each matrix transposed on the way into registers.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Shared address of the 16-byte unit ``unit`` (0..7) of row ``row`` of a
// 64-column (128-byte) bf16 box stored with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_addr(uint32_t box_base, int row, int unit) {
  return box_base + (uint32_t)row * 128u + ((uint32_t)(unit ^ (row & 7)) << 4);
}

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// Barrier over the first ``nthreads`` threads of the CTA (named barrier id).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace nsa
