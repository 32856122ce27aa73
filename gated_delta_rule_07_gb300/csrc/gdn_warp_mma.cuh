// gdn_warp_mma.cuh -- warp-level tensor-core helpers (ldmatrix, mma.sync m16n8k16 with fp16
// operands and fp32 accumulation) and the XOR-swizzled 16-bit tile addressing they read.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace warp_mma {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Four 8 x 8 matrices of 16-bit values to shared memory; lanes 8m .. 8m + 7 give the row
// addresses of matrix m, and lane l's register m holds its row l / 4, columns 2 (l % 4) and
// 2 (l % 4) + 1 (the layout ldmatrix returns).
__device__ __forceinline__ void stsm_x4(uint32_t addr, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}

// D = A * B + D, m16n8k16, A row-major, B column-major, fp16 in, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ swizzled 16-bit tiles
//
// A tile is `rows` x RL 16-bit values, row-major, with the 16-byte chunks of each row XOR-
// permuted by (row & 7) so that the eight row addresses of an ldmatrix hit eight different
// bank groups.  For RL = 64 this is the 128-byte-swizzle layout the tcgen05 kernels use.

template <int RL>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {  // c: multiple of 8
  return (uint32_t)(r * RL * 2) + ((((uint32_t)c >> 3) ^ ((uint32_t)r & 7u)) << 4);
}

// A fragment (16 x 16 at m0, k0) from a tile stored [m][k].
template <int RL>
__device__ __forceinline__ void load_a(uint32_t base, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31;
  ldsm_x4(base + tile_off<RL>(m0 + (l & 15), k0 + ((l >> 4) << 3)), a);
}

// A fragment (16 x 16 at m0, k0) from a tile stored [k][m] (the transpose).
template <int RL>
__device__ __forceinline__ void load_a_t(uint32_t base, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31, mi = l >> 3, rr = l & 7;
  ldsm_x4_t(base + tile_off<RL>(k0 + rr + ((mi >> 1) << 3), m0 + ((mi & 1) << 3)), a);
}

// B fragments of two n8 tiles (k0..k0+15, n0..n0+15) from a tile stored [k][n]:
// b[0], b[1] for columns n0..n0+7 and b[2], b[3] for n0+8..n0+15.
template <int RL>
__device__ __forceinline__ void load_b_kn(uint32_t base, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, mi = l >> 3, rr = l & 7;
  ldsm_x4_t(base + tile_off<RL>(k0 + rr + ((mi & 1) << 3), n0 + ((mi >> 1) << 3)), b);
}

// Same from a tile stored [n][k].
template <int RL>
__device__ __forceinline__ void load_b_nk(uint32_t base, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, mi = l >> 3, rr = l & 7;
  ldsm_x4(base + tile_off<RL>(n0 + rr + ((mi >> 1) << 3), k0 + ((mi & 1) << 3)), b);
}


}  // namespace warp_mma
}  // namespace gdn
