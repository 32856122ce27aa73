// gdn_tc5_util.cuh -- device and host helpers shared by the tcgen05 kernels: named barriers
// that tolerate divergent arrivals, TMA and bulk copies, packed 16-bit conversions, and the
// TMA descriptor of a [T, heads, 128] bf16 tensor.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace tc5u {

constexpr float kHalfMax = 65504.f;

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Named barriers over `n` threads (whole warps).  A lane may arrive after divergent work of its
// own (one lane issuing bulk copies, or waiting for them), so each warp first reconverges and
// the barrier is the form that does not require a converged warp; the warp leaves converged, as
// the tcgen05.ld / st that follow require.
__device__ __forceinline__ void named_bar(int id, int n) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
  __syncwarp();
}
// Barrier over `n` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
  uint32_t r;
  __syncwarp();
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbarrier.red.and.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  __syncwarp();
  return r != 0;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ bool fits_half(float x) { return fabsf(x) <= kHalfMax; }

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
// One 64 x 64 box of a [T, heads, 128] bf16 tensor (128-byte swizzle) into shared memory;
// completion is counted in bytes on the mbarrier.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int head,
                                        int t0, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(head), "r"(t0), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile(
      "{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
          mbar),
      "r"(bytes)
      : "memory");
}

// NB 16-byte chunks of bf16 at src + 1024 k to fp16 at dst + 1024 k; with SCALED the values of
// chunk k are multiplied by e[8 k] (chunks 1024 bytes apart lie 8 rows apart in a tile of
// 128-byte rows, and swizzling permutes chunks within a row only).  Returns the largest
// magnitude written, or m if larger.  All loads are issued before the first store: the compiler
// cannot tell src and dst apart and would otherwise wait for each store before the next load.
template <int NB, bool SCALED>
__device__ __forceinline__ float to_half_chunks(const uint8_t* src, uint8_t* dst, const float* e,
                                                float m) {
  uint4 x[NB];
#pragma unroll
  for (int k = 0; k < NB; ++k) x[k] = *reinterpret_cast<const uint4*>(src + 1024 * k);
  float mk[2] = {m, 0.f};
#pragma unroll
  for (int k = 0; k < NB; ++k) {
    const float sc = SCALED ? e[8 * k] : 1.f;
    uint32_t* w = reinterpret_cast<uint32_t*>(&x[k]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
      if (SCALED) {
        f.x *= sc;
        f.y *= sc;
      }
      mk[k & 1] = fmaxf(mk[k & 1], fmaxf(fabsf(f.x), fabsf(f.y)));
      w[i] = pack_h2(f.x, f.y);
    }
    *reinterpret_cast<uint4*>(dst + 1024 * k) = x[k];
  }
  return fmaxf(mk[0], mk[1]);
}

// Bulk copies (no tensor map): global -> shared completing on an mbarrier, and shared ->
// global in a bulk group.  Sizes are multiples of 16 bytes, addresses 16-byte aligned.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {  // sources of earlier bulk stores reusable
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {  // earlier bulk stores complete
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against libcuda).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled encode_fn() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// [T, heads, 128] bf16 tensor read as 64 (features) x 1 (head) x 64 (tokens) boxes with the
// 128-byte swizzle; tokens past T read as zeros.
inline cudaError_t make_map(CUtensorMap* m, const void* base, int64_t T, int heads) {
  EncodeTiled fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)(T > 0 ? T : 1)};
  const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  static const uint16_t dummy[64] __attribute__((aligned(16))) = {};
  void* addr = const_cast<void*>(base ? base : static_cast<const void*>(dummy));
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, addr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tc5u
}  // namespace gdn
