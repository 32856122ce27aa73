// gdn_backward.cu -- gradients of the gated delta rule (reverse mode of the forward).
//
// The loss gradient with respect to out and h_final comes in (dout, dh_final); the gradients
// of q, k, v, g, beta and h0 go out.  The page "Add context parallelism to the Gated Delta
// Net", sections "Tests" and "Measured results", holds the sharded layer's backward to the
// single-device one; it prints no backward formulas, so these follow from the forward chunk
// map of its section "Why".  Per chunk of L tokens with S the state entering it, D the
// gradient of the state leaving it (from the tokens after the chunk), G the inclusive running
// sum of g, Gamma[t][s] = exp(G_t - G_s):
//   forward pieces:  A = strictly lower (diag(beta) (K K^T o Gamma)),  attn = lower (Q K^T o Gamma)
//                    R = V - diag(e^G) K S,  delta = (I + A)^-1 diag(beta) R,
//                    o = diag(e^G) Q S + attn delta,  h_out = e^{G_L} S + Kt^T delta,
//                    Kt = diag(e^{G_L - G}) K
//   gradients:       d_delta = attn^T dO + Kt D,   dB = (I + A)^-T d_delta,
//                    dA = -(dB delta^T) o strictly lower,  dattn = (dO delta^T) o lower,
//                    dv = diag(beta) dB,
//                    dbeta_t = dB_t . R_t + sum_s dA_ts Gamma_ts (k_t . k_s),
//                    dq = diag(e^G) dO S^T + (dattn o Gamma) K,
//                    dk = -diag(beta e^G) dB S^T + diag(beta) (dA o Gamma) K
//                         + (dA o Gamma)^T diag(beta) K + (dattn o Gamma)^T Q + diag(e^{G_L-G}) delta D^T,
//                    dG_t = -beta_t e^{G_t} dB_t . (K S)_t + (row t - column t of dA o A)
//                           + e^{G_t} dO_t . (Q S)_t + (row t - column t of dattn o attn)
//                           - Kt_t . (delta D^T)_t,
//                    dG_L += sum(Kt o delta D^T) + e^{G_L} <D, S>,   dg_t = sum_{u >= t} dG_u.
// S and D at every chunk boundary come from two column-parallel token recurrences (a state
// column only meets its own value column): the forward one stores each chunk's entering state,
// the reverse one (dh_prev = alpha (F - beta k (k^T F)), F = dh + q dout^T) each chunk's
// leaving gradient and, at the sequence start, dh0; both run in one launch, on fp32 CUDA cores.
// The per-chunk work runs as one CTA per (chunk, value head) that walks through the products
// above on the tensor cores (warp-level TF32 products with fp32 accumulation), with T = (I + A)^-1
// formed once in shared memory and its intermediates in a per-CTA slice of the workspace.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int C = kChunk;  // 64
constexpr int kGradThreads = 512;

__device__ __forceinline__ void st_io(void* p, int64_t i, float x, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else
    static_cast<float*>(p)[i] = x;
}

// eight consecutive I/O elements (16-byte aligned in bf16, 32-byte in fp32) as fp32 into dst
__device__ __forceinline__ void ld8(const void* p, int64_t i, bool bf16, float* dst) {
  if (bf16) {
    const uint4 x = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p) + i);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&x);
    const float2 f0 = __bfloat1622float2(h2[0]), f1 = __bfloat1622float2(h2[1]);
    const float2 f2 = __bfloat1622float2(h2[2]), f3 = __bfloat1622float2(h2[3]);
    *reinterpret_cast<float4*>(dst) = make_float4(f0.x, f0.y, f1.x, f1.y);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(f2.x, f2.y, f3.x, f3.y);
  } else {
    const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    *reinterpret_cast<float4*>(dst) = f[0];
    *reinterpret_cast<float4*>(dst + 4) = f[1];
  }
}

// first chunk slot of sequence n (slots enumerate (sequence, chunk) pairs; see slot_to_chunk)
__device__ __forceinline__ int64_t slot_base(const int32_t* cu, int n) {
  return cu ? (int64_t)cu[n] / C + n : 0;
}

// ------------------------------------------------------------------ column recurrences

constexpr int kPhases = 16;  // threads per state column; each holds K / kPhases contiguous rows
constexpr int kColBlock = 8;  // state columns per CTA
constexpr int kColThreads = kColBlock * kPhases;
constexpr int kStage = 16;   // tokens staged in shared memory at a time (a quarter chunk)
constexpr int kColMinBlocks = 7;  // CTAs per SM the registers must allow (1024 CTAs: ~6.7 per SM)
static_assert(kStage <= 32 && kColThreads >= 32 && kColBlock % 8 == 0, "one warp scans a block");

// A staged key (or query) row: the K values in kPhases segments of K / kPhases, each followed
// by 4 floats of padding, so that the phases' 16-byte reads of one row spread over the banks
// (at most two reads to a group of four banks).
template <int K>
__host__ __device__ constexpr int row_stride() { return K + 4 * kPhases; }

// Shared memory of one column CTA: kStage rows of k (and, reversed, q), the CTA's columns of v
// (or dout), exp(g), beta, the scale factors of the scaled state and two block scalars.
template <int K>
__host__ __device__ constexpr size_t column_smem() {
  return sizeof(float) * ((size_t)2 * kStage * row_stride<K>() + (size_t)kStage * kColBlock + 4 * kStage + 4);
}

// The scaled state.  Within a staged block the recurrences carry h~ with h = A h~, A the product
// of the decays exp(g) met so far in the block, so that a token's update is one multiply-add per
// element:
//   forward, token t (A' = A exp(g_t)):  delta = beta (v - A' k.h~),  h~ += k delta / A'
//   reverse, token t (B the decays of the block's later tokens):  F~ = h~ + q dout / B,
//            h~ = F~ - beta k (k.F~)
// and h = A h~ again at the block's end.  A comes from a warp prefix sum P of g: A'_t = e^{P_t},
// B_t = e^{P_end - P_t}.  A block whose partial sums leave [-27, 27] (factors beyond ~5e11) takes
// the unscaled recurrence instead.
struct ColStage {
  float *ks, *qs, *vs, *gs, *bs, *sc, *iv, *blk;  // blk[0]: 1 = scaled; blk[1]: e^{P_end}
};

// kStage tokens [t0, t0 + n) of chunk inputs into shared memory (fp32, padded rows); warp 0
// also forms the block's scale factors
template <int K, bool REVERSE>
__device__ __forceinline__ void stage_tokens(const BwdArgs& a, int64_t t0, int n, int j, int kh,
                                             int v0, ColStage st) {
  constexpr int RPL = K / kPhases, RS = row_stride<K>();
  const void* vin = REVERSE ? a.dout : a.v;
  if (threadIdx.x < 32) {
    const int t = threadIdx.x;
    const float g = t < n ? a.g[(t0 + t) * a.hv + j] : 0.f;
    if (t < n) {
      st.gs[t] = __expf(g);
      st.bs[t] = a.beta[(t0 + t) * a.hv + j];
    }
    float P = g;  // inclusive prefix sum of g over the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, P, o);
      if (t >= o) P += y;
    }
    const float Pn = __shfl_sync(0xffffffffu, P, n - 1);
    const bool ok = __all_sync(0xffffffffu, fabsf(P) <= 27.f);
    if (t < n) {
      if (REVERSE) {
        st.iv[t] = __expf(P - Pn);  // 1 / B before token t
      } else {
        st.sc[t] = __expf(P);       // A'
        st.iv[t] = __expf(-P);      // 1 / A'
      }
    }
    if (t == 0) {
      st.blk[0] = ok ? 1.f : 0.f;
      st.blk[1] = __expf(Pn);
    }
  }
  static_assert(RPL % 4 == 0, "whole 16-byte pieces per segment");
  for (int e = threadIdx.x; e < n * (K / 8); e += kColThreads) {
    const int t = e / (K / 8), i = 8 * (e % (K / 8));
    // the eight values land in one segment (RPL >= 8) or in two consecutive ones (RPL = 4)
    const int o0 = t * RS + (i / RPL) * (RPL + 4) + i % RPL;
    const int o1 = t * RS + ((i + 4) / RPL) * (RPL + 4) + (i + 4) % RPL;
    float x[8];
    ld8(a.k, ((t0 + t) * a.hk + kh) * K + i, a.bf16, x);
    *reinterpret_cast<float4*>(st.ks + o0) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(st.ks + o1) = make_float4(x[4], x[5], x[6], x[7]);
    if (REVERSE) {
      ld8(a.q, ((t0 + t) * a.hk + kh) * K + i, a.bf16, x);
      *reinterpret_cast<float4*>(st.qs + o0) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(st.qs + o1) = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  for (int e = threadIdx.x; e < n * (kColBlock / 8); e += kColThreads) {
    const int t = e / (kColBlock / 8), cc = 8 * (e % (kColBlock / 8));
    ld8(vin, ((t0 + t) * a.hv + j) * a.V + v0 + cc, a.bf16, st.vs + t * kColBlock + cc);
  }
}

// the dot product of a staged row segment with the thread's rows, summed over the column's
// phases
template <int RPL>
__device__ __forceinline__ float col_dot(const float* kv, const float* h) {
  float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
  for (int i = 0; i < RPL; i += 4) {
    d0 = fmaf(kv[i], h[i], d0);
    d1 = fmaf(kv[i + 1], h[i + 1], d1);
    d2 = fmaf(kv[i + 2], h[i + 2], d2);
    d3 = fmaf(kv[i + 3], h[i + 3], d3);
  }
  float d = (d0 + d1) + (d2 + d3);
#pragma unroll
  for (int o = 1; o < kPhases; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  return d;
}
template <int RPL>
__device__ __forceinline__ void ld_seg(const float* src, float* dst) {
#pragma unroll
  for (int i = 0; i < RPL / 4; ++i) {
    const float4 f = reinterpret_cast<const float4*>(src)[i];
    dst[4 * i] = f.x; dst[4 * i + 1] = f.y; dst[4 * i + 2] = f.z; dst[4 * i + 3] = f.w;
  }
}

// One direction of one CTA: sequence n, value head j, kColBlock state columns; thread (column,
// phase p) holds rows [p RPL, (p + 1) RPL) of its column.  Forward: stores the state entering
// every chunk as states[slot][j][v][i] (a state column contiguous).  Reverse: stores the gradient
// of the state leaving every chunk in the same layout, and dh0.
template <int K, bool REVERSE>
__device__ __forceinline__ void column_run(const BwdArgs& a, float* csm) {
  constexpr int RPL = K / kPhases, RS = row_stride<K>();
  ColStage st;
  st.ks = csm;                         // [kStage][RS]
  st.qs = st.ks + kStage * RS;         // [kStage][RS] (reverse)
  st.vs = st.qs + kStage * RS;         // [kStage][kColBlock]
  st.gs = st.vs + kStage * kColBlock;  // [kStage] exp(g)
  st.bs = st.gs + kStage;              // [kStage] beta
  st.sc = st.bs + kStage;              // [kStage] A' (forward)
  st.iv = st.sc + kStage;              // [kStage] 1 / A' (forward), 1 / B (reverse)
  st.blk = st.iv + kStage;             // [2]
  const int nj = blockIdx.x, n = nj / a.hv, j = nj % a.hv, kh = j / (a.hv / a.hk);
  const int col = threadIdx.x / kPhases, p = threadIdx.x % kPhases;
  const int v0 = blockIdx.y * kColBlock, v = v0 + col;
  int64_t t0, t1;
  if (!seq_bounds(a.cu, n, a.T, a.status, t0, t1)) return;
  const int64_t KV = (int64_t)K * a.V;
  float h[RPL];
  const float* init = REVERSE ? a.dh_final : a.h0;
#pragma unroll
  for (int i = 0; i < RPL; ++i)
    h[i] = init ? init[((int64_t)n * a.hv + j) * KV + (int64_t)(p * RPL + i) * a.V + v] : 0.f;
  float* store = REVERSE ? a.dstates : a.states;
  const int64_t nc = (t1 - t0 + C - 1) / C, sb = slot_base(a.cu, n);
  const int ko = p * (RPL + 4);  // this phase's segment of a staged row
  for (int64_t ci = 0; ci < nc; ++ci) {
    const int64_t c = REVERSE ? nc - 1 - ci : ci;
    const int64_t c0 = t0 + c * C;
    const int L = (int)((t1 - c0) < C ? (t1 - c0) : C);
    float4* dst = reinterpret_cast<float4*>(store + (((sb + c) * a.hv + j) * a.V + v) * K + p * RPL);
#pragma unroll
    for (int i = 0; i < RPL / 4; ++i) dst[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    const int nb = (L + kStage - 1) / kStage;
    for (int bi = 0; bi < nb; ++bi) {
      const int b = REVERSE ? nb - 1 - bi : bi;
      const int bn = (L - b * kStage) < kStage ? (L - b * kStage) : kStage;
      __syncthreads();  // the previous block's inputs have been used
      stage_tokens<K, REVERSE>(a, c0 + b * kStage, bn, j, kh, v0, st);
      __syncthreads();
      if (st.blk[0] != 0.f) {  // the scaled state
#pragma unroll 2
        for (int s = 0; s < bn; ++s) {
          const int t = REVERSE ? bn - 1 - s : s;
          const float beta = st.bs[t], x = st.vs[t * kColBlock + col], ivt = st.iv[t];
          float kv[RPL];
          ld_seg<RPL>(st.ks + t * RS + ko, kv);
          if (REVERSE) {  // F~ = h~ + q dout / B;  h~ <- F~ - beta k (k . F~)
            float qv[RPL];
            ld_seg<RPL>(st.qs + t * RS + ko, qv);
            const float xs = x * ivt;
#pragma unroll
            for (int i = 0; i < RPL; ++i) h[i] = fmaf(qv[i], xs, h[i]);
            const float bd = beta * col_dot<RPL>(kv, h);
#pragma unroll
            for (int i = 0; i < RPL; ++i) h[i] = fmaf(-kv[i], bd, h[i]);
          } else {  // delta = beta (v - A' k . h~);  h~ += k delta / A'
            const float d = col_dot<RPL>(kv, h);
            const float f = beta * fmaf(-st.sc[t], d, x) * ivt;
#pragma unroll
            for (int i = 0; i < RPL; ++i) h[i] = fmaf(kv[i], f, h[i]);
          }
        }
        const float mult = st.blk[1];
#pragma unroll
        for (int i = 0; i < RPL; ++i) h[i] *= mult;
      } else {  // the plain recurrence
        for (int s = 0; s < bn; ++s) {
          const int t = REVERSE ? bn - 1 - s : s;
          const float alpha = st.gs[t], beta = st.bs[t], x = st.vs[t * kColBlock + col];
          float kv[RPL];
          ld_seg<RPL>(st.ks + t * RS + ko, kv);
          if (REVERSE) {  // F = dh + q dout^T;  dd = k . F;  dh <- alpha (F - beta k dd)
            float qv[RPL];
            ld_seg<RPL>(st.qs + t * RS + ko, qv);
#pragma unroll
            for (int i = 0; i < RPL; ++i) h[i] = fmaf(qv[i], x, h[i]);
            const float bd = beta * col_dot<RPL>(kv, h);
#pragma unroll
            for (int i = 0; i < RPL; ++i) h[i] = alpha * fmaf(-kv[i], bd, h[i]);
          } else {  // delta = beta (v - alpha k . h);  h <- alpha h + k delta
            const float dl = beta * (x - alpha * col_dot<RPL>(kv, h));
#pragma unroll
            for (int i = 0; i < RPL; ++i) h[i] = fmaf(kv[i], dl, alpha * h[i]);
          }
        }
      }
    }
  }
  if (REVERSE && a.dh0) {
#pragma unroll
    for (int i = 0; i < RPL; ++i)
      a.dh0[((int64_t)n * a.hv + j) * KV + (int64_t)(p * RPL + i) * a.V + v] = h[i];
  }
}

// grid (N hv, V / kColBlock, 2): z = 0 the forward recurrence, z = 1 the reverse one; the two
// directions are independent and share the SMs.
template <int K>
__global__ void __launch_bounds__(kColThreads, kColMinBlocks) column_kernel(BwdArgs a) {
  extern __shared__ __align__(16) float csm[];
  if (blockIdx.z == 0)
    column_run<K, false>(a, csm);
  else
    column_run<K, true>(a, csm);
}

// ------------------------------------------------------------------ per-chunk gradients

struct GradSmem {
  float GKK[C][C + 1];  // Gamma o K K^T, strictly lower (A = diag(beta) GKK)
  float At[C][C + 1];   // attn = Gamma o Q K^T, lower
  float dA[C][C + 1], dat[C][C + 1];
  float G[C], eG[C], ekt[C], b[C], dG[C];
  float scal[4];
  float As[2 * C][36];  // product tiles (row strides of 4 and 8 banks mod 32: the tensor-core
  float Bs[32][136];    // fragments read them without bank conflicts); As holds 128 rows when
                        // two products that share B run as one
  float X[C][129];      // d_delta (the back solve's right-hand side)
  float Tm[C][C + 1];   // T = (I + A)^-1, unit lower triangular
  float red[16];        // per-warp partial sums
  float KF[C][129], QF[C][129];  // k, q of the chunk (fp32; rows past the chunk are zero)
};

// floats of one CTA's workspace slice: K S, Q S, R, delta, d_delta (then dB), dout as [C][V];
// delta D^T as [C][K]
template <int K, int V>
__host__ __device__ constexpr int64_t grad_slice() { return 6 * (int64_t)C * V + (int64_t)C * K; }

// TF32 operand (round to nearest, ties away) and one warp-level tensor-core product
// D(16 x 8) += A(16 x 8) B(8 x 8) with fp32 accumulation
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// out(i, c, x) for i < M, c < N with x = sum_{y < Y} A(i, y) B(y, c) (Y a multiple of 32), on
// the tensor cores: 32-wide slices of y are staged in shared memory (each thread fetches its
// share of the next slice into registers, from before the barrier that precedes the current
// slice's multiply until after it).  M = 64, or 128
// for two 64-row products that share B (rows 64.. the second).  Warp w owns 16 rows from
// 16 (w mod M/16) and N M / 256 columns, as 16 x 8 tiles.
// TF3: each operand is split into a TF32 head and a TF32 remainder and three products are
// summed (head x remainder, remainder x head, head x head), which keeps fp32 accuracy; without
// it the operands are rounded to TF32 once.  AI / BY: the operand's contiguous index is i (for
// A) / y (for B), so that the fetches walk memory in order.
template <int M, int N, bool AI, bool BY, bool TF3, typename FA, typename FB, typename FO>
__device__ __forceinline__ void mm(GradSmem& sm, int Y, FA A, FB B, FO out) {
  constexpr int MB = M / 16;                // row blocks
  constexpr int NC = N * M / 256;           // columns of a warp
  constexpr int NT = NC / 8;                // its 16 x 8 tiles
  constexpr int NA = M * 32 / kGradThreads, NB = 32 * N / kGradThreads;
  static_assert(kGradThreads == 512 && (M == 64 || M == 128) && NT >= 1, "16 warps over M rows");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 2, tig = lane & 3;
  const int r0 = 16 * (warp % MB) + grp, c0 = (warp / MB) * NC + grp;
  float acc[NT][4];
#pragma unroll
  for (int m = 0; m < NT; ++m)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
  float pa[NA], pb[NB];
  auto fetch = [&](int y0) {
#pragma unroll
    for (int k = 0; k < NA; ++k) {
      const int e = tid + k * kGradThreads;
      pa[k] = A(AI ? e % M : e / 32, y0 + (AI ? e / M : e % 32));
    }
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int e = tid + k * kGradThreads;
      pb[k] = B(y0 + (BY ? e % 32 : e / N), BY ? e / 32 : e % N);
    }
  };
  fetch(0);
  for (int y0 = 0; y0 < Y; y0 += 32) {
    __syncthreads();  // the previous slice (or product) is done with the tiles
#pragma unroll
    for (int k = 0; k < NA; ++k) {
      const int e = tid + k * kGradThreads;
      sm.As[AI ? e % M : e / 32][AI ? e / M : e % 32] = pa[k];
    }
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int e = tid + k * kGradThreads;
      sm.Bs[BY ? e % 32 : e / N][BY ? e / 32 : e % N] = pb[k];
    }
    if (y0 + 32 < Y) fetch(y0 + 32);  // (reads the operands' sources, not the tiles)
    __syncthreads();
#pragma unroll
    for (int k8 = 0; k8 < 32; k8 += 8) {
      const float af[4] = {sm.As[r0][k8 + tig], sm.As[r0 + 8][k8 + tig], sm.As[r0][k8 + tig + 4],
                           sm.As[r0 + 8][k8 + tig + 4]};
      uint32_t ah[4], al[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ah[q] = to_tf32(af[q]);
        if (TF3) al[q] = to_tf32(af[q] - __uint_as_float(ah[q]));
      }
#pragma unroll
      for (int m = 0; m < NT; ++m) {
        const float bf[2] = {sm.Bs[k8 + tig][c0 + 8 * m], sm.Bs[k8 + tig + 4][c0 + 8 * m]};
        uint32_t bh[2], bl[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          bh[q] = to_tf32(bf[q]);
          if (TF3) bl[q] = to_tf32(bf[q] - __uint_as_float(bh[q]));
        }
        if (TF3) {
          mma_tf32(acc[m], al, bh);
          mma_tf32(acc[m], ah, bl);
        }
        mma_tf32(acc[m], ah, bh);
      }
    }
  }
  const int cc = (warp / MB) * NC + 2 * tig;
#pragma unroll
  for (int m = 0; m < NT; ++m) {
    out(r0, cc + 8 * m, acc[m][0]);
    out(r0, cc + 8 * m + 1, acc[m][1]);
    out(r0 + 8, cc + 8 * m, acc[m][2]);
    out(r0 + 8, cc + 8 * m + 1, acc[m][3]);
  }
}

// One CTA per (chunk slot, value head); grid-stride over the units.
template <int K, int V, bool TF3>
__global__ void __launch_bounds__(kGradThreads) chunk_grad_kernel(BwdArgs a) {
  extern __shared__ __align__(16) uint8_t smraw[];
  GradSmem& sm = *reinterpret_cast<GradSmem*>(smraw);
  const int tid = threadIdx.x;
  const int64_t nslots = a.nslots, units = nslots * a.hv;
  float* ws = a.scratch + (int64_t)blockIdx.x * grad_slice<K, V>();
  float* KS = ws;            // [C][V]  K S
  float* QS = KS + C * V;    // [C][V]  Q S
  float* R = QS + C * V;     // [C][V]  V - e^G K S
  float* DL = R + C * V;     // [C][V]  delta
  float* DD = DL + C * V;    // [C][V]  d_delta, then dB
  float* DO = DD + C * V;    // [C][V]  dout (fp32)
  float* XD = DO + C * V;    // [C][K]  delta D^T
  auto KF = [&](int t, int i) -> float& { return sm.KF[t][i]; };
  auto QF = [&](int t, int i) -> float& { return sm.QF[t][i]; };
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t slot = u / a.hv;
    const int j = (int)(u % a.hv), kh = j / (a.hv / a.hk);
    int n;
    int64_t cidx;
    if (!slot_to_chunk(a.cu, a.N, a.T, slot, n, cidx)) continue;
    int64_t sb, se;
    if (!seq_bounds(a.cu, n, a.T, a.status, sb, se)) continue;
    const int64_t t0 = sb + cidx * C;
    const int L = (int)((se - t0) < C ? (se - t0) : C);
    const float* Sx = a.states + ((slot * a.hv + j) * (int64_t)V) * K;   // S[i][v] = Sx[v K + i]
    const float* Dx = a.dstates + ((slot * a.hv + j) * (int64_t)V) * K;
    __syncthreads();  // the previous unit is done with the shared and workspace buffers
    // ---- decays (running sum by one warp); q, k, dout as fp32
    if (tid < 32) {
      const float g0 = tid < L ? a.g[(t0 + tid) * a.hv + j] : 0.f;
      const float g1 = tid + 32 < L ? a.g[(t0 + tid + 32) * a.hv + j] : 0.f;
      float x0 = g0, x1 = g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (tid >= o) { x0 += y0; x1 += y1; }
      }
      x1 += __shfl_sync(0xffffffffu, x0, 31);
      const float GL = (L - 1) < 32 ? __shfl_sync(0xffffffffu, x0, (L - 1) & 31)
                                    : __shfl_sync(0xffffffffu, x1, (L - 1) & 31);
      sm.G[tid] = x0;
      sm.G[tid + 32] = x1;
      sm.eG[tid] = __expf(x0);
      sm.eG[tid + 32] = __expf(x1);
      sm.ekt[tid] = __expf(GL - x0);
      sm.ekt[tid + 32] = __expf(GL - x1);
      sm.b[tid] = tid < L ? a.beta[(t0 + tid) * a.hv + j] : 0.f;
      sm.b[tid + 32] = tid + 32 < L ? a.beta[(t0 + tid + 32) * a.hv + j] : 0.f;
      if (tid == 0) sm.scal[0] = __expf(GL);
    }
    for (int e8 = tid; e8 < C * K / 8; e8 += kGradThreads) {  // eight elements a load
      const int t = 8 * e8 / K, i = 8 * e8 % K;
      float k8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, q8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (t < L) {
        ld8(a.k, ((t0 + t) * a.hk + kh) * K + i, a.bf16, k8);
        ld8(a.q, ((t0 + t) * a.hk + kh) * K + i, a.bf16, q8);
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        KF(t, i + m) = k8[m];
        QF(t, i + m) = q8[m];
      }
    }
    for (int e8 = tid; e8 < C * V / 8; e8 += kGradThreads) {
      const int e = 8 * e8, t = e / V, c = e % V;
      if (t < L) {
        ld8(a.dout, ((t0 + t) * a.hv + j) * V + c, a.bf16, DO + e);
      } else {
        reinterpret_cast<float4*>(DO + e)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4*>(DO + e)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncthreads();
    auto gam = [&](int t, int s) { return __expf(sm.G[t] - sm.G[s]); };  // for s <= t
    // ---- Gamma o K K^T (strictly lower), attn; K S, Q S
    mm<2 * C, C, false, true, TF3>(  // rows 0-63: K K^T, rows 64-127: Q K^T (they share K^T)
        sm, K, [&](int t, int y) { return t < C ? KF(t, y) : QF(t - C, y); },
        [&](int y, int s) { return KF(s, y); },
        [&](int t, int s, float x) {
          if (t < C) sm.GKK[t][s] = (s < t && t < L) ? gam(t, s) * x : 0.f;
          else sm.At[t - C][s] = (s <= t - C && t - C < L) ? gam(t - C, s) * x : 0.f;
        });
    mm<C, V, false, true, TF3>(sm, K, [&](int t, int y) { return KF(t, y); },
                       [&](int y, int c) { return Sx[c * K + y]; },
                       [&](int t, int c, float x) { KS[t * V + c] = x; });
    mm<C, V, false, true, TF3>(sm, K, [&](int t, int y) { return QF(t, y); },
                       [&](int y, int c) { return Sx[c * K + y]; },
                       [&](int t, int c, float x) { QS[t * V + c] = x; });
    __syncthreads();
    // ---- R = V - e^G K S;  T = (I + A)^-1 in shared memory (blockwise: the diagonal blocks by
    // substitution, the rest from them); delta = T diag(beta) R
    for (int e8 = tid; e8 < C * V / 8; e8 += kGradThreads) {
      const int e = 8 * e8, t = e / V, c = e % V;
      float v8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (t < L) ld8(a.v, ((t0 + t) * a.hv + j) * V + c, a.bf16, v8);
#pragma unroll
      for (int m = 0; m < 8; ++m) R[e + m] = t < L ? v8[m] - sm.eG[t] * KS[e + m] : 0.f;
    }
    {  // the four 16 x 16 diagonal blocks of T by substitution, eight threads per column
      const int c = tid >> 3, p = tid & 7, c0 = c & ~15;  // (a warp's four columns share a block)
      for (int t = p; t < C; t += 8) sm.Tm[t][c] = t == c ? 1.f : 0.f;
      __syncwarp();
      for (int t = c0 + 1; t < c0 + 16; ++t) {  // T[t][c] = -beta_t sum_{c <= s < t} GKK[t][s] T[s][c]
        float x = 0.f;
        for (int s = c + p; s < t; s += 8) x = fmaf(sm.GKK[t][s], sm.Tm[s][c], x);
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        if (p == 0 && t > c) sm.Tm[t][c] = -sm.b[t] * x;
        __syncwarp();
      }
    }
    // the blocks below the diagonal, one band at a time (block (i, j) needs the bands nearer the
    // diagonal): T_ij = -T_ii sum_{j <= k < i} A_ik T_kj with A = diag(beta) GKK; the sums go
    // through sm.X (free until d_delta)
    float* Pb = &sm.X[0][0];  // [3][16][16]
    for (int d = 1; d < 4; ++d) {
      __syncthreads();
      for (int e = tid; e < (4 - d) * 256; e += kGradThreads) {
        const int j = e >> 8, i = j + d, r = (e >> 4) & 15, cc = e & 15;
        const int row = 16 * i + r;
        float x = 0.f;
        for (int s = 16 * j; s < 16 * i; ++s) x = fmaf(sm.GKK[row][s], sm.Tm[s][16 * j + cc], x);
        Pb[e] = sm.b[row] * x;
      }
      __syncthreads();
      for (int e = tid; e < (4 - d) * 256; e += kGradThreads) {
        const int j = e >> 8, i = j + d, r = (e >> 4) & 15, cc = e & 15;
        float x = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) x = fmaf(sm.Tm[16 * i + r][16 * i + m], Pb[(j << 8) + (m << 4) + cc], x);
        sm.Tm[16 * i + r][16 * j + cc] = -x;
      }
    }
    __syncthreads();
    mm<C, V, false, false, TF3>(sm, C, [&](int t, int s) { return sm.Tm[t][s]; },
                             [&](int s, int c) { return sm.b[s] * R[s * V + c]; },
                             [&](int t, int c, float x) { DL[t * V + c] = x; });
    __syncthreads();
    // ---- d_delta = attn^T dO + Kt D
    mm<C, V, true, false, TF3>(sm, C, [&](int t, int s) { return sm.At[s][t]; },
                       [&](int s, int c) { return DO[s * V + c]; },
                       [&](int t, int c, float x) { DD[t * V + c] = x; });
    mm<C, V, false, true, TF3>(sm, K, [&](int t, int y) { return sm.ekt[t] * KF(t, y); },
                       [&](int y, int c) { return Dx[c * K + y]; },
                       [&](int t, int c, float x) { sm.X[t][c] = t < L ? DD[t * V + c] + x : 0.f; });
    __syncthreads();
    // ---- dB = T^T d_delta
    mm<C, V, true, false, TF3>(sm, C, [&](int t, int s) { return sm.Tm[s][t]; },
                            [&](int s, int c) { return sm.X[s][c]; },
                            [&](int t, int c, float x) {
                              DD[t * V + c] = x;
                              if (t < L) st_io(a.dv, ((t0 + t) * a.hv + j) * V + c, sm.b[t] * x, a.bf16);
                            });
    __syncthreads();
    // ---- dA = -(dB delta^T) o strictly lower, dattn = (dO delta^T) o lower
    mm<2 * C, C, false, true, TF3>(  // rows 0-63: dB delta^T, rows 64-127: dO delta^T
        sm, V, [&](int t, int c) { return t < C ? DD[t * V + c] : DO[(t - C) * V + c]; },
        [&](int c, int s) { return DL[s * V + c]; },
        [&](int t, int s, float x) {
          if (t < C) sm.dA[t][s] = (s < t && t < L) ? -x : 0.f;
          else sm.dat[t - C][s] = (s <= t - C && t - C < L) ? x : 0.f;
        });
    // ---- delta D^T
    mm<C, K, false, false, TF3>(sm, V, [&](int t, int c) { return DL[t * V + c]; },
                        [&](int c, int i) { return Dx[c * K + i]; },
                        [&](int t, int i, float x) { XD[t * K + i] = x; });
    __syncthreads();
    // ---- per row: dbeta and dG (eight threads a row)
    {
      const int t = tid >> 3, p = tid & 7;
      float db = 0.f, dg = 0.f, kd = 0.f;
      if (t < L) {
        for (int c = p; c < V; c += 8) {
          db = fmaf(DD[t * V + c], R[t * V + c], db);
          dg = fmaf(-sm.b[t] * sm.eG[t] * DD[t * V + c], KS[t * V + c], dg);
          dg = fmaf(sm.eG[t] * DO[t * V + c], QS[t * V + c], dg);
        }
        for (int s = p; s < L; s += 8) {
          if (s < t) db = fmaf(sm.dA[t][s], sm.GKK[t][s], db);
          dg += sm.dA[t][s] * sm.b[t] * sm.GKK[t][s] - sm.dA[s][t] * sm.b[s] * sm.GKK[s][t];
          dg += sm.dat[t][s] * sm.At[t][s] - sm.dat[s][t] * sm.At[s][t];
        }
        for (int i = p; i < K; i += 8) kd = fmaf(KF(t, i), XD[t * K + i], kd);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        db += __shfl_xor_sync(0xffffffffu, db, o);
        dg += __shfl_xor_sync(0xffffffffu, dg, o);
        kd += __shfl_xor_sync(0xffffffffu, kd, o);
      }
      kd *= sm.ekt[t];
      if (p == 0) {
        if (t < L) a.dbeta[(t0 + t) * a.hv + j] = db;
        sm.dG[t] = t < L ? dg - kd : 0.f;
        sm.X[t][0] = t < L ? kd : 0.f;  // (summed below)
      }
    }
    __syncthreads();
    {  // <S, D> over the whole CTA
      float ds = 0.f;
      for (int e = 4 * tid; e < K * V; e += 4 * kGradThreads) {
        const float4 x = *reinterpret_cast<const float4*>(Sx + e);
        const float4 y = *reinterpret_cast<const float4*>(Dx + e);
        ds = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, ds))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, o);
      if ((tid & 31) == 0) sm.red[tid >> 5] = ds;
    }
    __syncthreads();
    if (tid < 32) {  // dG_L += sum_t Kt_t . (delta D^T)_t + e^{G_L} <D, S>
      float tot = sm.X[tid][0] + sm.X[tid + 32][0], ds = tid < kGradThreads / 32 ? sm.red[tid] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        ds += __shfl_xor_sync(0xffffffffu, ds, o);
      }
      if (tid == 0) sm.dG[L - 1] += tot + sm.scal[0] * ds;
      __syncwarp();
      // dg_t = sum_{u >= t} dG_u (reverse running sum over the chunk)
      float x0 = sm.dG[63 - tid], x1 = sm.dG[31 - tid];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (tid >= o) { x0 += y0; x1 += y1; }
      }
      x1 += __shfl_sync(0xffffffffu, x0, 31);
      const int r0 = 63 - tid, r1 = 31 - tid;
      if (r0 < L) a.dg[(t0 + r0) * a.hv + j] = x0;
      if (r1 < L) a.dg[(t0 + r1) * a.hv + j] = x1;
    }
    // ---- dA o Gamma and dattn o Gamma in place
    for (int e = tid; e < C * C; e += kGradThreads) {
      const int t = e / C, s = e % C;
      const float gm = s <= t ? gam(t, s) : 0.f;
      sm.dA[t][s] *= gm;
      sm.dat[t][s] *= gm;
    }
    // ---- dq = diag(e^G) dO S^T + (dattn o Gamma) K  (per value head; the group sum follows)
    float* dqv = a.dqv + (t0 * a.hv + j) * (int64_t)K;
    float* dkv = a.dkv + (t0 * a.hv + j) * (int64_t)K;
    const int64_t rs = (int64_t)a.hv * K;  // row stride of dqv, dkv
    mm<C, K, false, false, TF3>(sm, V, [&](int t, int c) { return DO[t * V + c]; },
                        [&](int c, int i) { return Sx[c * K + i]; },
                        [&](int t, int i, float x) { if (t < L) dqv[t * rs + i] = sm.eG[t] * x; });
    mm<C, K, false, false, TF3>(sm, C, [&](int t, int s) { return sm.dat[t][s]; },
                        [&](int s, int i) { return KF(s, i); },
                        [&](int t, int i, float x) { if (t < L) dqv[t * rs + i] += x; });
    // ---- dk = -diag(beta e^G) dB S^T + diag(e^{G_L - G}) delta D^T + diag(beta) (dA o Gamma) K
    //          + (dA o Gamma)^T diag(beta) K + (dattn o Gamma)^T Q
    mm<C, K, false, false, TF3>(sm, V, [&](int t, int c) { return DD[t * V + c]; },
                        [&](int c, int i) { return Sx[c * K + i]; },
                        [&](int t, int i, float x) {
                          if (t < L) dkv[t * rs + i] = sm.ekt[t] * XD[t * K + i] - sm.b[t] * sm.eG[t] * x;
                        });
    mm<C, K, false, false, TF3>(sm, C, [&](int t, int s) { return sm.dA[t][s]; },
                        [&](int s, int i) { return KF(s, i); },
                        [&](int t, int i, float x) { if (t < L) dkv[t * rs + i] += sm.b[t] * x; });
    mm<C, K, true, false, TF3>(sm, C, [&](int t, int s) { return sm.dA[s][t] * sm.b[s]; },
                       [&](int s, int i) { return KF(s, i); },
                       [&](int t, int i, float x) { if (t < L) dkv[t * rs + i] += x; });
    mm<C, K, true, false, TF3>(sm, C, [&](int t, int s) { return sm.dat[s][t]; },
                       [&](int s, int i) { return QF(s, i); },
                       [&](int t, int i, float x) { if (t < L) dkv[t * rs + i] += x; });
  }
}

// dq, dk of each key head: the sum over the value heads that read it, in the I/O dtype.
__global__ void group_sum_kernel(BwdArgs a) {
  const int64_t n = a.T * a.hk * (int64_t)a.K;
  const int grp = a.hv / a.hk;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = e / ((int64_t)a.hk * a.K);
    const int kh = (int)((e / a.K) % a.hk), i = (int)(e % a.K);
    float sq = 0.f, sk = 0.f;
    for (int m = 0; m < grp; ++m) {
      const int64_t o = (t * a.hv + kh * grp + m) * (int64_t)a.K + i;
      sq += a.dqv[o];
      sk += a.dkv[o];
    }
    st_io(a.dq, e, sq, a.bf16);
    st_io(a.dk, e, sk, a.bf16);
  }
}

template <int K, int V>
cudaError_t launch_all(const BwdArgs& a, cudaStream_t s) {
  const dim3 cg((unsigned)(a.N * a.hv), (unsigned)(V / kColBlock), 2);
  cudaError_t e = cudaFuncSetAttribute(column_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)column_smem<K>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_grad_kernel<K, V, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(GradSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_grad_kernel<K, V, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(GradSmem));
  if (e != cudaSuccess) return e;
  column_kernel<K><<<cg, kColThreads, column_smem<K>(), s>>>(a);
  if (a.bf16)  // TF32 products (their error is far below the bf16 rounding of the results)
    chunk_grad_kernel<K, V, false><<<a.grad_ctas, kGradThreads, sizeof(GradSmem), s>>>(a);
  else  // split-TF32 products: fp32 accuracy
    chunk_grad_kernel<K, V, true><<<a.grad_ctas, kGradThreads, sizeof(GradSmem), s>>>(a);
  group_sum_kernel<<<1024, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int64_t bwd_slots(int64_t T, int N) { return T / kChunk + N; }

size_t bwd_scratch_floats(int K, int V, int ctas) {
  return (size_t)ctas * (6 * (size_t)kChunk * V + (size_t)kChunk * K);
}

cudaError_t backward(const BwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.K == 128 && a.V == 128) return launch_all<128, 128>(a, s);
  if (a.K == 128 && a.V == 64) return launch_all<128, 64>(a, s);
  if (a.K == 64 && a.V == 128) return launch_all<64, 128>(a, s);
  return launch_all<64, 64>(a, s);
}

}  // namespace gdn
