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
constexpr int kPThreads = 128;

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

// grid: (token blocks, 2 hk + hv head slices); thread = channel within the slice
__global__ void __launch_bounds__(kPThreads) prologue_kernel(PrologueArgs a) {
  __shared__ float ys[kTB][kPThreads + 1];
  __shared__ float inv[kTB];
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
  const int W = a.W;
  if (tid < width) {
    const int64_t c = ch + tid;
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = i < W ? a.conv_w[c * W + i] : 0.f;
    // win[i] = x_{t - W + 1 + i} for i < W - 1 (the carried inputs), refilled at sequence starts
    int n = seq_of(a.cu, a.N, t0);
    int64_t sb = a.cu ? a.cu[n] : 0;
    float win[3] = {0.f, 0.f, 0.f};
    auto fill = [&](int64_t t) {  // the W - 1 inputs before token t of sequence n
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int64_t s = t - (W - 1) + i;
        float x = 0.f;
        if (i < W - 1) {
          if (s >= sb) x = ld_x(a.x, s * Ch + c, a.bf16);
          else if (a.state_in) x = ld_x(a.state_in, ((int64_t)n * Ch + c) * (W - 1) + (s - sb + W - 1), a.bf16);
        }
        win[i] = x;
      }
    };
    fill(t0);
    int64_t next = (a.cu && n + 1 <= a.N) ? a.cu[n + 1] : a.T;
    for (int64_t t = t0; t < t1; ++t) {
      while (t >= next && n + 1 < a.N) {  // a new sequence starts at t
        ++n;
        sb = a.cu[n];
        next = a.cu[n + 1];
        fill(t);
      }
      const float xt = ld_x(a.x, t * Ch + c, a.bf16);
      float y = (W == 4 ? w[3] : W == 3 ? w[2] : W == 2 ? w[1] : w[0]) * xt;
#pragma unroll
      for (int i = 0; i < 3; ++i)
        if (i < W - 1) y = fmaf(w[i], win[i], y);
      win[0] = W == 2 ? xt : win[1];  // shift the window (constant indices: registers)
      win[1] = W == 3 ? xt : win[2];
      win[2] = xt;
      if (a.silu) y = y / (1.f + __expf(-y));
      ys[t - t0][tid] = y;
    }
  }
  __syncthreads();
  const int nt = (int)(t1 - t0);
  if (is_q || is_k) {  // 1 / max(|y|, 1e-6) per token: a warp per token in turn
    const int warp = tid >> 5, lane = tid & 31;
    for (int t = warp; t < nt; t += kPThreads / 32) {
      float s = 0.f;
      for (int c = lane; c < width; c += 32) s = fmaf(ys[t][c], ys[t][c], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) inv[t] = rsqrtf(fmaxf(s, 1e-12f));
    }
    __syncthreads();
  }
  if (tid < width) {
    void* dst = is_q ? a.q : is_k ? a.k : a.v;
    const int heads = (is_q || is_k) ? a.hk : a.hv;
    for (int t = 0; t < nt; ++t) {
      const float y = (is_q || is_k) ? ys[t][tid] * inv[t] : ys[t][tid];
      st_x(dst, ((t0 + t) * heads + hd) * (int64_t)width + tid, y, a.bf16);
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
    const dim3 grid((unsigned)((a.T + kTB - 1) / kTB), (unsigned)(2 * a.hk + a.hv));
    prologue_kernel<<<grid, kPThreads, 0, s>>>(a);
  }
  if (a.state_out && a.W > 1) {
    const dim3 grid(64, (unsigned)a.N);
    prologue_state_kernel<<<grid, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
