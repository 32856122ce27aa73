// Test-only probe of the library's tcgen05 building blocks (gdn_sm100.cuh): runs one
// 128 x N x K MMA with the operand layouts the chunk kernels use and writes D to global
// memory, so a test can compare it with a plain matrix product.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_sm100.cuh"

using namespace gdn::sm100;

struct ProbeCase {
  int N, K;
  int a_src;        // 0 smem K-major, 1 smem MN-major, 2 TMEM
  int b_mn;         // 0 K-major, 1 MN-major
  int a_cap, b_cap;  // rows per 64-wide column block of the stored A / B tile
  int b_roff;       // row offset of B inside its tile
};

// A_log [128][K] and B_log [K][N] are plain row-major fp16; D [128][N] fp32.
__global__ void __launch_bounds__(128) probe_kernel(ProbeCase pc, const __half* A_log,
                                                    const __half* B_log, float* D,
                                                    int* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint32_t tmem_base;
  __shared__ __align__(8) uint64_t mbar;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int M = 128, N = pc.N, K = pc.K;
  // swizzle atoms must start on a 1024-byte boundary
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* sa = smem;           // 64 KB region for A
  unsigned char* sb = smem + 65536;   // 64 KB region for B
  // lay A out
  if (pc.a_src == 0) {
    for (int e = tid; e < M * K; e += 128) {
      const int m = e / K, k = e % K;
      *reinterpret_cast<__half*>(sa + sw128_offset(pc.a_cap, m, k)) = A_log[m * K + k];
    }
  } else if (pc.a_src == 1) {
    for (int e = tid; e < M * K; e += 128) {
      const int m = e / K, k = e % K;
      *reinterpret_cast<__half*>(sa + sw128_offset(pc.a_cap, k, m)) = A_log[m * K + k];
    }
  }
  for (int e = tid; e < K * N; e += 128) {
    const int k = e / N, n = e % N;
    const uint32_t off = pc.b_mn ? sw128_offset(pc.b_cap, pc.b_roff + k, n)
                                 : sw128_offset(pc.b_cap, pc.b_roff + n, k);
    *reinterpret_cast<__half*>(sb + off) = B_log[k * N + n];
  }
  if (warp == 0) {
    tmem_alloc((uint32_t)__cvta_generic_to_shared(&tmem_base), 512);
    tmem_relinquish();
  }
  if (tid == 0) mbar_init((uint32_t)__cvta_generic_to_shared(&mbar), 1);
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = tmem_base;
  const uint32_t d_t = tbase;            // columns [0, N)
  const uint32_t a_t = tbase + 256;      // columns [256, 256 + K/2)
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  if (pc.a_src == 2) {
    const int m = tid;  // this thread's TMEM lane
    for (int c0 = 0; c0 < K / 2; c0 += 16) {
      uint32_t r[16];
      for (int j = 0; j < 16; ++j) {
        __half2 p = __halves2half2(A_log[m * K + 2 * (c0 + j)], A_log[m * K + 2 * (c0 + j) + 1]);
        r[j] = *reinterpret_cast<uint32_t*>(&p);
      }
      tmem_st16(a_t + lane_off + c0, r);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
  }
  const uint32_t mb = (uint32_t)__cvta_generic_to_shared(&mbar);
  if (tid == 0) {
    const uint32_t sa_addr = (uint32_t)__cvta_generic_to_shared(sa);
    const uint32_t sb_addr = (uint32_t)__cvta_generic_to_shared(sb);
    const uint32_t id = idesc_f16(M, N, pc.a_src == 1, pc.b_mn);
    for (int ks = 0; ks < K / 16; ++ks) {
      uint64_t bdesc;
      if (pc.b_mn)
        bdesc = sdesc(sb_addr + pc.b_roff * 128 + ks * 2048, pc.b_cap * 128, 1024);
      else
        bdesc = sdesc(sb_addr + (ks >> 2) * pc.b_cap * 128 + pc.b_roff * 128 + (ks & 3) * 32,
                      16, 1024);
      if (pc.a_src == 2) {
        mma_ts(d_t, a_t + ks * 8, bdesc, id, ks > 0);
      } else {
        uint64_t adesc = pc.a_src == 1
            ? sdesc(sa_addr + ks * 2048, pc.a_cap * 128, 1024)
            : sdesc(sa_addr + (ks >> 2) * pc.a_cap * 128 + (ks & 3) * 32, 16, 1024);
        mma_ss(d_t, adesc, bdesc, id, ks > 0);
      }
    }
    mma_commit(mb);
  }
  const bool ok = mbar_wait(mb, 0, 1u << 24);
  fence_after_sync();
  if (!ok) {
    if (tid == 0) atomicExch(status, 5);
  } else {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tmem_ld32(d_t + lane_off + c0, v);
      for (int j = 0; j < 32; ++j) D[tid * N + c0 + j] = v[j];
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

extern "C" int probe_run(int N, int K, int a_src, int b_mn, int a_cap, int b_cap, int b_roff,
                         const void* A, const void* B, void* D, void* status) {
  if (N != 64 && N != 128) return -1;
  if (K != 64 && K != 128) return -1;
  if (a_cap < 128 || b_cap < 64 || b_roff + (b_mn ? K : N) > b_cap) return -1;
  ProbeCase pc{N, K, a_src, b_mn, a_cap, b_cap, b_roff};
  const int smem = 131072 + 1024;
  cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  probe_kernel<<<1, 128, smem>>>(pc, static_cast<const __half*>(A),
                                  static_cast<const __half*>(B), static_cast<float*>(D),
                                  static_cast<int*>(status));
  if (cudaGetLastError() != cudaSuccess) return -2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
