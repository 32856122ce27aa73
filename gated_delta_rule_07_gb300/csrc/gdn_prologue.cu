// gdn_prologue.cu -- the layer-side steps ahead of the recurrence: the causal depthwise conv over
// the q | k | v channels, q and k L2-normalised per head, and g, beta from their projections.
//
// Page "Add context parallelism to the Gated Delta Net", section "Implementation" (layer-side
// bullets): a causal depthwise conv whose halo is conv_kernel_dim - 1 tokens.  Page "RFC(qwen35):
// TP Phase2", section "Partition Contract": a per-request conv state of qkv_dim x
// (conv_kernel_dim - 1) inputs.  Readings where the pages are silent: an optional SiLU after the
// conv, q and k divided by their L2 norm (floored at 1e-6) per (token, head), g = -exp(A_log)
// softplus(a + dt_bias) and beta = sigmoid(b) per value head.
//
//   y_t[c] = sum_{i < W} w[c][i] x_{t - W + 1 + i}[c], with inputs before a sequence's start taken
//   from its conv state (oldest first) or zero.
//
// HBM-bound elementwise work: one CTA per (block of 64 tokens, head slice of the channels), one
// thread per channel that slides the conv window through the block in registers; the block's
// outputs are staged in shared memory so that q and k can be normalised per token.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kTB = 64;       // tokens per CTA
constexpr int kPThreads = 512;  // 128 channels x 4 quarters of the token block

__device__ __forceinline__ float ld_x(const void* p, int64_t i, bool bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
              : static_cast<const float*>(p)[i];
}
__device__ __forceinline__ void st_x(void* p, int64_t i, float x, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else
    static_cast<float*>(p)[i] = x;
}

// sequence of token t: the largest n with cu[n] <= t (cu null: one sequence)
__device__ __forceinline__ int seq_of(const int32_t* cu, int N, int64_t t) {
  if (!cu) return 0;
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr int kHalo = 3;       // inputs before a block's first token that its conv can read
constexpr int kRow = 128 + 1;  // padded row of a staged tile (floats)

// eight consecutive I/O elements (16-byte aligned in bf16, 32-byte in fp32) as fp32
__device__ __forceinline__ void ld8x(const void* p, int64_t i, bool bf16, float* dst) {
  if (bf16) {
    const uint4 x = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p) + i);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 f = __bfloat1622float2(h2[m]);
      dst[2 * m] = f.x;
      dst[2 * m + 1] = f.y;
    }
  } else {
    const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    const float4 u = f[0], w = f[1];
    dst[0] = u.x; dst[1] = u.y; dst[2] = u.z; dst[3] = u.w;
    dst[4] = w.x; dst[5] = w.y; dst[6] = w.z; dst[7] = w.w;
  }
}
__device__ __forceinline__ void st8x(void* p, int64_t i, bool bf16, const float* v) {
  if (bf16) {
    uint4 x;
    __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&x);
#pragma unroll
    for (int m = 0; m < 4; ++m) h2[m] = __floats2bfloat162_rn(v[2 * m], v[2 * m + 1]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p) + i) = x;
  } else {
    float4* f = reinterpret_cast<float4*>(static_cast<float*>(p) + i);
    f[0] = make_float4(v[0], v[1], v[2], v[3]);
    f[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

struct ProSmem {
  float xs[kTB + kHalo][kRow];  // inputs of tokens t0 - 3 .. t1 - 1 (rows before 0 are zero);
                                // row t + 3 then receives token t's conv output
  float inv[kTB];
  int64_t sb[kTB];              // start of each token's sequence
  int seq[kTB];                 // and its index
  int inside[kTB];              // 1: the token's whole conv window lies in its sequence
};

// grid: (token blocks, 2 hk + hv head slices).  The block's input tile is staged in shared memory
// with 16-byte loads, the conv reads it (or, before a sequence's start, the sequence's conv
// state), and the outputs leave with 16-byte stores.
__global__ void __launch_bounds__(kPThreads) prologue_kernel(PrologueArgs a) {
  extern __shared__ __align__(16) uint8_t praw[];
  ProSmem& sm = *reinterpret_cast<ProSmem*>(praw);
  const int blk = blockIdx.y, tid = threadIdx.x;
  const bool is_q = blk < a.hk, is_k = !is_q && blk < 2 * a.hk;
  const int hd = is_q ? blk : is_k ? blk - a.hk : blk - 2 * a.hk;  // head within its kind
  const int width = (is_q || is_k) ? a.K : a.V;
  const int64_t ch = is_q ? (int64_t)hd * a.K
                   : is_k ? (int64_t)a.hk * a.K + (int64_t)hd * a.K
                          : 2LL * a.hk * a.K + (int64_t)hd * a.V;  // first channel of the slice
  const int64_t Ch = 2LL * a.hk * a.K + (int64_t)a.hv * a.V;
  const int64_t t0 = (int64_t)blockIdx.x * kTB;
  const int64_t t1 = (t0 + kTB < a.T) ? t0 + kTB : a.T;
  const int nt = (int)(t1 - t0), W = a.W, g8 = width / 8;
  // ---- stage the tile; each token's sequence
  for (int e = tid; e < (nt + kHalo) * g8; e += kPThreads) {
    const int r = e / g8, c8 = 8 * (e % g8);
    const int64_t t = t0 - kHalo + r;
    if (t >= 0) ld8x(a.x, t * Ch + ch + c8, a.bf16, &sm.xs[r][c8]);
    else
#pragma unroll
      for (int m = 0; m < 8; ++m) sm.xs[r][c8 + m] = 0.f;
  }
  for (int t = tid; t < nt; t += kPThreads) {
    const int n = seq_of(a.cu, a.N, t0 + t);
    const int64_t sb = a.cu ? a.cu[n] : 0;
    sm.seq[t] = n;
    sm.sb[t] = sb;
    sm.inside[t] = t0 + t - (W - 1) >= sb;
  }
  __syncthreads();
  // ---- the conv (and SiLU), a channel per thread: the window slides through the staged tile in
  // registers; a token whose window crosses its sequence's start reads the conv state instead
  const int cl = tid & 127, qt = tid >> 7;  // channel, quarter of the block's tokens
  const bool act = cl < width;
  const int64_t c = ch + cl;
  const int tq = 16 * qt;  // the quarter's first token; its window = tokens tq - 3 .. tq - 1
  float w[4] = {0.f, 0.f, 0.f, 0.f}, x0 = 0.f, x1 = 0.f, x2 = 0.f;
  if (act) {
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = i < W ? a.conv_w[c * W + i] : 0.f;
    x0 = sm.xs[tq][cl];
    x1 = sm.xs[tq + 1][cl];
    x2 = sm.xs[tq + 2][cl];
  }
  __syncthreads();  // every window is read before any output overwrites an input row
  if (act) {
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int t = tq + jj;
      if (t >= nt) break;
      const float x3 = sm.xs[t + kHalo][cl];
      float y;
      if (sm.inside[t]) {  // the whole window lies in the token's sequence
        y = W == 4 ? fmaf(w[0], x0, fmaf(w[1], x1, fmaf(w[2], x2, w[3] * x3)))
          : W == 3 ? fmaf(w[0], x1, fmaf(w[1], x2, w[2] * x3))
          : W == 2 ? fmaf(w[0], x2, w[1] * x3)
                   : w[0] * x3;
      } else {  // the window crosses the sequence's start: earlier inputs from its conv state
        const int64_t tt = t0 + t, sb = sm.sb[t];
        y = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i < W) {
            const int64_t s = tt - (W - 1) + i;  // the input this tap reads
            const int wi = 4 - W + i;            // the window register holding it
            float x = 0.f;
            if (s >= sb) x = wi == 0 ? x0 : wi == 1 ? x1 : wi == 2 ? x2 : x3;
            else if (a.state_in) x = ld_x(a.state_in, ((int64_t)sm.seq[t] * Ch + c) * (W - 1) + (s - sb + W - 1), a.bf16);
            y = fmaf(w[i], x, y);
          }
        }
      }
      x0 = x1;
      x1 = x2;
      x2 = x3;
      if (a.silu) y = __fdividef(y, 1.f + __expf(-y));  // (the divisor is >= 1)
      sm.xs[t + kHalo][cl] = y;
    }
  }
  __syncthreads();
  if (is_q || is_k) {  // 1 / max(|y|, 1e-6) per token: a warp per token in turn
    const int warp = tid >> 5, lane = tid & 31;
    for (int t = warp; t < nt; t += kPThreads / 32) {
      float s2 = 0.f;
      for (int c = lane; c < width; c += 32) s2 = fmaf(sm.xs[t + kHalo][c], sm.xs[t + kHalo][c], s2);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      if (lane == 0) sm.inv[t] = rsqrtf(fmaxf(s2, 1e-12f));
    }
    __syncthreads();
  }
  // ---- outputs, eight channels a store
  {
    void* dst = is_q ? a.q : is_k ? a.k : a.v;
    const int heads = (is_q || is_k) ? a.hk : a.hv;
    for (int e = tid; e < nt * g8; e += kPThreads) {
      const int t = e / g8, c8 = 8 * (e % g8);
      const float sc = (is_q || is_k) ? sm.inv[t] : 1.f;
      float v8[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) v8[m] = sm.xs[t + kHalo][c8 + m] * sc;
      st8x(dst, ((t0 + t) * heads + hd) * (int64_t)width + c8, a.bf16, v8);
    }
  }
  if (!is_q && !is_k && tid < nt) {  // g, beta of this value head
    const int64_t t = t0 + tid;
    const float av = ld_x(a.a, t * a.hv + hd, a.bf16), bv = ld_x(a.b, t * a.hv + hd, a.bf16);
    const float z = av + a.dt_bias[hd];
    const float sp = z > 20.f ? z : log1pf(__expf(z));  // softplus
    a.g[t * a.hv + hd] = -__expf(a.A_log[hd]) * sp;
    a.beta[t * a.hv + hd] = 1.f / (1.f + __expf(-bv));
  }
}

// new conv state: the last W - 1 inputs of each sequence; when a sequence is shorter, the older
// state entries shift in (entry j = the input W - 1 - j positions before the sequence's end).
__global__ void prologue_state_kernel(PrologueArgs a) {
  const int64_t Ch = 2LL * a.hk * a.K + (int64_t)a.hv * a.V;
  const int n = blockIdx.y;
  const int W1 = a.W - 1;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < Ch;
       c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t sb = a.cu ? a.cu[n] : 0, se = a.cu ? a.cu[n + 1] : a.T, L = se - sb;
    float vals[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      float x = 0.f;
      if (j < W1) {
        if (L + j >= W1) x = ld_x(a.x, (se - W1 + j) * Ch + c, a.bf16);
        else if (a.state_in) x = ld_x(a.state_in, ((int64_t)n * Ch + c) * W1 + (L + j), a.bf16);
      }
      vals[j] = x;
    }
#pragma unroll
    for (int j = 0; j < 3; ++j)
      if (j < W1) st_x(a.state_out, ((int64_t)n * Ch + c) * W1 + j, vals[j], a.bf16);
  }
}

}  // namespace

cudaError_t prologue(const PrologueArgs& a, cudaStream_t s) {
  if (a.T > 0) {
    cudaError_t e = cudaFuncSetAttribute(prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(ProSmem));
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((a.T + kTB - 1) / kTB), (unsigned)(2 * a.hk + a.hv));
    prologue_kernel<<<grid, kPThreads, sizeof(ProSmem), s>>>(a);
  }
  if (a.state_out && a.W > 1) {
    const dim3 grid(64, (unsigned)a.N);
    prologue_state_kernel<<<grid, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
