// Warp-level bf16 tensor-core helpers (mma.sync m16n8k16, fp32 accumulate).
//
// Fragment ownership of m16n8k16 (lane = 4*r + m, r = lane/4, m = lane%4):
//   A (16x16, row-major): a0 = A[r][2m..2m+1],   a1 = A[r+8][2m..2m+1],
//                         a2 = A[r][2m+8..2m+9], a3 = A[r+8][2m+8..2m+9]
//   B (16x8, k-major):    b0 = B[2m..2m+1][r],   b1 = B[2m+8..2m+9][r]
//   C (16x8):             c0,c1 = C[r][2m..2m+1], c2,c3 = C[r+8][2m..2m+1]
// (the lower k index sits in the lower 16 bits of a register).
//
// The k dimension of a product is a sum, so its order is free.  The kernels
// use that freedom so that one 16-byte load of 8 consecutive channels feeds
// two k-steps directly: for chunk c = 4s + m of a row (channels 8c..8c+7),
//   k-step 2s   takes channels 8c+0,1 as slots 2m,2m+1 and 8c+2,3 as 2m+8,2m+9
//   k-step 2s+1 takes channels 8c+4,5 and 8c+6,7 the same way,
// i.e. the 16-byte vector {x, y, z, w} gives {x, y} to k-step 2s and {z, w}
// to k-step 2s+1, for A rows and B columns alike.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace sls {

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// max(x, 0) and min(x, 0) of two packed bf16 values (exact).
__device__ __forceinline__ uint32_t bf16x2_relu(uint32_t w) {
  uint32_t r = w;
  if (w & 0x00008000u) r &= 0xffff0000u;
  if (w & 0x80000000u) r &= 0x0000ffffu;
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_negpart(uint32_t w) {
  uint32_t r = w;
  if (!(w & 0x00008000u)) r &= 0xffff0000u;
  if (!(w & 0x80000000u)) r &= 0x0000ffffu;
  return r;
}

}  // namespace sls
