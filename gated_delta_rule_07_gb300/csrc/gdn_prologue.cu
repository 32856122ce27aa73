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
// HBM-bound elementwise work, streamed through registers: a thread owns four consecutive channels
// of one head and walks a run of 64 tokens, its conv window held in registers and the next four
// tokens' inputs already in flight; q and k are normalised by a shuffle reduction over the lanes
// that hold the head.  No shared memory, no block barrier.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

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

// sequence of token t: the largest n < N with cu[n] <= t (cu null: one sequence)
__device__ __forceinline__ int seq_of(const int32_t* cu, int N, int64_t t) {
  if (!cu) return 0;
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr int kSThreads = 256;  // threads of a CTA
constexpr int kLoadBytes = 16;  // bytes of one token a thread loads: its consecutive channels
constexpr int kRing = 8;        // tokens in a thread's shared-memory ring (kRing - 1 in flight)
template <typename IO>
__host__ __device__ constexpr int cpt() { return kLoadBytes / (int)sizeof(IO); }  // channels a thread owns

constexpr int kWords = kLoadBytes / 4;
static_assert(kLoadBytes == 16, "one 16-byte copy per token and thread");
struct Raw {  // one token's channels of a thread, as loaded
  uint32_t u[kWords];
};
__device__ __forceinline__ Raw raw_load(const void* p) {
  const uint4 v = __ldg(static_cast<const uint4*>(p));
  Raw r;
  r.u[0] = v.x; r.u[1] = v.y; r.u[2] = v.z; r.u[3] = v.w;
  return r;
}
__device__ __forceinline__ void raw_store(void* p, const Raw& r) {
  *static_cast<uint4*>(p) = make_uint4(r.u[0], r.u[1], r.u[2], r.u[3]);
}
template <typename IO>
__device__ __forceinline__ Raw raw_at(const void* base, int64_t i) {
  return raw_load(static_cast<const IO*>(base) + i);
}
// to fp32 (a bf16 is the top half of an fp32) and back
template <typename IO>
__device__ __forceinline__ void unpack(const Raw& r, float* f) {
#pragma unroll
  for (int i = 0; i < kWords; ++i) {
    if constexpr (sizeof(IO) == 2) {
      f[2 * i] = __uint_as_float(r.u[i] << 16);
      f[2 * i + 1] = __uint_as_float(r.u[i] & 0xffff0000u);
    } else {
      f[i] = __uint_as_float(r.u[i]);
    }
  }
}
template <typename IO>
__device__ __forceinline__ Raw pack(const float* f) {
  Raw r;
#pragma unroll
  for (int i = 0; i < kWords; ++i) {
    if constexpr (sizeof(IO) == 2) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      r.u[i] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      r.u[i] = __float_as_uint(f[i]);
    }
  }
  return r;
}

// how the channel slots of a token map onto threads: a head of width w occupies the next power
// of two >= w / cpt<IO>() lanes (aligned), q heads then k heads then v heads
struct SlotMap {
  int lphk, lphv;    // lanes per q / k head, per v head
  int qk_slots;      // 2 hk lphk
  int slots;         // qk_slots + hv lphv
  int cpr;           // CTAs per token range (each a slice of the channel slots)
  int ranges;        // token ranges (the grid is ranges x cpr CTAs, all resident at once)
};

// SiLU y sigmoid(y).  fp32 I/O: y / (1 + e^-y).  bf16 I/O: h + h tanh(h) with h = y / 2 on the
// hardware tanh approximation (absolute error ~2.5e-4 |y|, below the bf16 rounding of the result
// where it matters, and one special-function op instead of two)
template <typename IO>
__device__ __forceinline__ float silu(float y) {
  if constexpr (sizeof(IO) == 2) {
    const float h = 0.5f * y;
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(h));
    return fmaf(h, th, h);
  } else {
    return __fdividef(y, 1.f + __expf(-y));  // (the divisor is >= 1)
  }
}
// one 16-byte copy global -> shared of this thread's (no bytes read, zero filled, when !ok), as
// its own commit group
__device__ __forceinline__ void ring_copy(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// g, beta of every (token, value head)
__device__ void gate_maps(const PrologueArgs& a) {
  const int64_t n = a.T * a.hv, stride = (int64_t)gridDim.x * kSThreads;
  for (int64_t e = (int64_t)blockIdx.x * kSThreads + threadIdx.x; e < n; e += stride) {
    const int h = (int)(e % a.hv);
    const float av = ld_x(a.a, e, a.bf16), bv = ld_x(a.b, e, a.bf16);
    const float z = av + a.dt_bias[h];
    const float sp = z > 20.f ? z : log1pf(__expf(z));  // softplus
    a.g[e] = -__expf(a.A_log[h]) * sp;
    a.beta[e] = 1.f / (1.f + __expf(-bv));
  }
}

// one input of a window read the slow way (only where the window reaches before its sequence's
// start): token u from x inside the sequence that starts at sb, before it the sequence's conv
// state (oldest entry first), zero past the state
template <typename IO>
__device__ __forceinline__ void window_input(const PrologueArgs& a, int64_t Ch, int64_t c,
                                             int64_t u, int64_t sb, int seq, float* f) {
  if (u >= sb && u >= 0) {
    unpack<IO>(raw_at<IO>(a.x, u * Ch + c), f);
    return;
  }
  const int W1 = a.W - 1;
  const int64_t j = W1 - (sb - u);
  const int64_t base = ((int64_t)seq * Ch + c) * W1 + j;
#pragma unroll
  for (int m = 0; m < cpt<IO>(); ++m)
    f[m] = (a.state_in && j >= 0) ? ld_x(a.state_in, base + m * W1, a.bf16) : 0.f;
}

// grid: m.ranges x m.cpr CTAs, as many as are resident at once: CTA (range r, part p) walks the
// tokens of range r through the channels of part p, then takes its share of the g, beta maps.
// Taps are padded to four, y_t = w0 x_{t-3} + w1 x_{t-2} + w2 x_{t-1} + w3 x_t, summed in that
// fixed order.  LPHK = m.lphk (lanes per q / k head), fixed at compile time for the norms.
template <typename IO, int LPHK>
__global__ void __launch_bounds__(kSThreads, 2) prologue_kernel(PrologueArgs a, SlotMap m) {
  constexpr int kCPT = cpt<IO>();
  const int range = (int)blockIdx.x / m.cpr;
  const int slot = ((int)blockIdx.x % m.cpr) * kSThreads + (int)threadIdx.x;
  // this thread's head and lanes
  const bool qk = slot < m.qk_slots;
  const int lph = qk ? LPHK : m.lphv;
  const int rel = qk ? slot : slot - m.qk_slots;
  const int hh = rel / lph, l = rel % lph;  // head (q heads then k heads, or v head), lane
  const int width = qk ? a.K : a.V;
  const bool act = slot < m.slots && kCPT * l < width;
  const int64_t Ch = 2LL * a.hk * a.K + (int64_t)a.hv * a.V;
  const int64_t c = (qk ? (int64_t)hh * a.K : 2LL * a.hk * a.K + (int64_t)hh * a.V) + kCPT * l;
  const int head = qk && hh >= a.hk ? hh - a.hk : hh, heads = qk ? a.hk : a.hv;
  const int64_t drow = (int64_t)heads * width;
  const bool warp_qk = ((slot & ~31) < m.qk_slots);  // the warp holds some q / k head
  const int W = a.W;
  float w[kCPT][4];
#pragma unroll
  for (int ch = 0; ch < kCPT; ++ch)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[ch][i] = (act && i >= 4 - W) ? a.conv_w[(c + ch) * W + i - (4 - W)] : 0.f;

  // token indices fit in 32 bits (the API caps the token count at INT32_MAX)
  const int t0 = (int)(a.T * range / m.ranges), t1 = (int)(a.T * (range + 1) / m.ranges);
  int n = seq_of(a.cu, a.N, t0);
  int s0 = a.cu ? a.cu[n] : 0, s1 = a.cu ? a.cu[n + 1] : (int)a.T;  // the sequence's bounds

  // window slots: token t0 + i lives in slot i mod 4; slots 1, 2, 3 start with the three tokens
  // ahead of the range (replaced from the conv state where a window reaches before its
  // sequence's start)
  float xw[4][kCPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int ch = 0; ch < kCPT; ++ch) xw[i][ch] = 0.f;
  if (act && t0 >= 3) {
    unpack<IO>(raw_at<IO>(a.x, (t0 - 3) * Ch + c), xw[1]);
    unpack<IO>(raw_at<IO>(a.x, (t0 - 2) * Ch + c), xw[2]);
    unpack<IO>(raw_at<IO>(a.x, (t0 - 1) * Ch + c), xw[3]);
  }
  // the thread's ring of inputs in flight: token t0 + i in slot i mod kRing, at ring[slot][thread]
  extern __shared__ __align__(16) uint4 ring[];
  const uint32_t ring0 = (uint32_t)__cvta_generic_to_shared(ring + threadIdx.x);
  // (a copy that reads nothing still names x's first element, an address inside the tensor)
  const IO* x0 = static_cast<const IO*>(a.x);
  const IO* xc = x0 + c;
#pragma unroll
  for (int r = 0; r < kRing - 1; ++r) {
    const bool ok = act && t0 + r < t1;
    ring_copy(ring0 + r * kSThreads * 16, ok ? xc + (int64_t)(t0 + r) * Ch : x0, ok);
  }
  const IO* xn = xc + (int64_t)(t0 + kRing - 1) * Ch;  // the next token to copy (used when in range)
  IO* dp = static_cast<IO*>(qk ? (hh < a.hk ? a.q : a.k) : a.v) + (int64_t)head * width +
           kCPT * l + t0 * drow;
  static_assert(kRing % 4 == 0, "ring slots advance four tokens at a time");
  for (int tb = t0; tb < t1; tb += 4) {
    const int rb = (tb - t0) % kRing;
#pragma unroll
    for (int J = 0; J < 4; ++J) {
      const int t = tb + J;
      if (t >= t1) break;
      {  // token t + kRing - 1 into the slot that token t - 1 used; then token t has landed
        const bool ok = act && t + kRing - 1 < t1;
        ring_copy(ring0 + ((rb + J + kRing - 1) % kRing) * kSThreads * 16, ok ? xn : x0, ok);
        xn += Ch;
        asm volatile("cp.async.wait_group %0;\n" ::"n"(kRing - 1) : "memory");
      }
      if (t >= s1 || t - 3 < s0) {  // (uniform: every thread of the CTA walks the same tokens)
        while (n < a.N - 1 && t >= s1) {
          ++n;
          s0 = s1;
          s1 = a.cu[n + 1];
        }
        if (t - 3 < s0 && act) {  // the window reaches before the sequence's start
          window_input<IO>(a, Ch, c, t - 3, s0, n, xw[(J + 1) & 3]);
          window_input<IO>(a, Ch, c, t - 2, s0, n, xw[(J + 2) & 3]);
          window_input<IO>(a, Ch, c, t - 1, s0, n, xw[(J + 3) & 3]);
        }
      }
      {
        const uint4 v = ring[(rb + J) * kSThreads + threadIdx.x];
        Raw r;
        r.u[0] = v.x; r.u[1] = v.y; r.u[2] = v.z; r.u[3] = v.w;
        unpack<IO>(r, xw[J]);
      }
      float o[kCPT], s2 = 0.f;
#pragma unroll
      for (int ch = 0; ch < kCPT; ++ch) {
        float y = fmaf(w[ch][0], xw[(J + 1) & 3][ch],
                       fmaf(w[ch][1], xw[(J + 2) & 3][ch],
                            fmaf(w[ch][2], xw[(J + 3) & 3][ch], w[ch][3] * xw[J][ch])));
        if (a.silu) y = silu<IO>(y);
        o[ch] = y;
        s2 = fmaf(y, y, s2);
      }
      if (warp_qk) {  // 1 / max(|y|, 1e-6) over the head's lanes (aligned groups of LPHK)
#pragma unroll
        for (int off = 1; off < LPHK; off <<= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        if (qk) {
          const float inv = rsqrtf(fmaxf(s2, 1e-12f));
#pragma unroll
          for (int ch = 0; ch < kCPT; ++ch) o[ch] *= inv;
        }
      }
      if (act) raw_store(dp, pack<IO>(o));
      dp += drow;
    }
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  gate_maps(a);
}

template <typename IO, int LPHK>
cudaError_t launch_prologue(const PrologueArgs& a, SlotMap m, cudaStream_t s) {
  const int smem = kRing * kSThreads * 16;
  const auto kern = prologue_kernel<IO, LPHK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, smem);
  if (e != cudaSuccess) return e;
  // one wave: the token ranges split the resident CTAs between them (at least 16 tokens each)
  const int64_t resident = (int64_t)(per_sm > 0 ? per_sm : 1) * sms;
  int64_t ranges = resident / m.cpr;
  if (ranges > (a.T + 15) / 16) ranges = (a.T + 15) / 16;
  m.ranges = (int)(ranges > 1 ? ranges : 1);
  const int64_t ctas = (int64_t)m.ranges * m.cpr;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kSThreads, smem, s>>>(a, m);
  return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_prologue_io(const PrologueArgs& a, const SlotMap& m, cudaStream_t s) {
  switch (m.lphk) {
    case 1: return launch_prologue<IO, 1>(a, m, s);
    case 2: return launch_prologue<IO, 2>(a, m, s);
    case 4: return launch_prologue<IO, 4>(a, m, s);
    case 8: return launch_prologue<IO, 8>(a, m, s);
    case 16: return launch_prologue<IO, 16>(a, m, s);
    default: return launch_prologue<IO, 32>(a, m, s);
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
    auto pow2 = [](int x) { int p = 1; while (p < x) p <<= 1; return p; };
    SlotMap m;
    const int cp = kLoadBytes / (a.bf16 ? 2 : 4);
    m.lphk = pow2(a.K / cp);
    m.lphv = pow2(a.V / cp);
    m.qk_slots = 2 * a.hk * m.lphk;
    m.slots = m.qk_slots + a.hv * m.lphv;
    m.cpr = (m.slots + kSThreads - 1) / kSThreads;
    cudaError_t e = a.bf16 ? launch_prologue_io<__nv_bfloat16>(a, m, s)
                           : launch_prologue_io<float>(a, m, s);
    if (e != cudaSuccess) return e;
  }
  if (a.state_out && a.W > 1) {
    const dim3 grid(64, (unsigned)a.N);
    prologue_state_kernel<<<grid, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
