// gdn_common.cuh -- device helpers shared by the kernels of libgdn (not by the oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;  // C: tokens per chunk

// I/O element conversion.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Records the first error code in a device status word (no-op for a null word).
__device__ __forceinline__ void set_status(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

// Token range [b, e) of sequence n.  A null table means one sequence [0, T).  Returns false
// (and records GDN_ERR_DEVICE_INPUT) when the table is inconsistent, so that no kernel ever
// indexes outside [0, T) whatever the caller passed.
__device__ __forceinline__ bool seq_bounds(const int32_t* cu, int n, int64_t T, int32_t* st,
                                           int64_t& b, int64_t& e) {
  if (cu == nullptr) {
    b = 0;
    e = T;
    return true;
  }
  const int64_t x = cu[n], y = cu[n + 1];
  if (x < 0 || y < x || y > T) {
    set_status(st, GDN_ERR_DEVICE_INPUT);
    return false;
  }
  b = x;
  e = y;
  return true;
}

// Chunk range [c0, c1) of segment r of a sequence of L tokens: Nc = ceil(L / C) chunks split
// into P contiguous segments, the first (Nc mod P) one chunk longer.
__device__ __forceinline__ void segment_chunks(int64_t L, int P, int r, int64_t& c0,
                                               int64_t& c1) {
  const int64_t nc = (L + kChunk - 1) / kChunk;
  const int64_t base = nc / P, extra = nc % P;
  c0 = (int64_t)r * base + ((int64_t)r < extra ? r : extra);
  c1 = c0 + base + ((int64_t)r < extra ? 1 : 0);
}

// Chunk "slots" enumerate every (sequence, chunk) pair without a prefix sum: sequence n owns
// slots [floor(cu[n]/C) + n, floor(cu[n]/C) + n + Nc_n), disjoint for a valid table, and all
// slots lie below floor(T/C) + N.  Maps a slot to (n, chunk); false if the slot is unused.
__device__ __forceinline__ bool slot_to_chunk(const int32_t* cu, int N, int64_t T, int64_t slot,
                                              int& n_out, int64_t& chunk_out) {
  int n = 0;
  if (cu != nullptr) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {  // largest n with cu[n]/C + n <= slot
      const int mid = (lo + hi + 1) >> 1;
      const int64_t base = (int64_t)(cu[mid] < 0 ? 0 : cu[mid]) / kChunk + mid;
      if (base <= slot) lo = mid; else hi = mid - 1;
    }
    n = lo;
  }
  const int64_t b = cu ? (int64_t)(cu[n] < 0 ? 0 : cu[n]) : 0;
  const int64_t e = cu ? (int64_t)cu[n + 1] : T;
  const int64_t c = slot - (b / kChunk + n);
  if (c < 0 || e < b || c >= (e - b + kChunk - 1) / kChunk) return false;
  n_out = n;
  chunk_out = c;
  return true;
}

}  // namespace gdn
