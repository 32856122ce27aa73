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
// leaving gradient and, at the sequence start, dh0.  Everything is fp32 arithmetic on CUDA
// cores; the per-chunk work runs as one CTA per (chunk, value head) that walks through the
// products above with its intermediates in a per-CTA slice of the workspace.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int C = kChunk;  // 64
constexpr int kColThreads = 128;   // 32 state columns per CTA, 4 lanes per column
constexpr int kGradThreads = 256;

__device__ __forceinline__ float ld_io(const void* p, int64_t i, bool bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
              : static_cast<const float*>(p)[i];
}
__device__ __forceinline__ void st_io(void* p, int64_t i, float x, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else
    static_cast<float*>(p)[i] = x;
}

// first chunk slot of sequence n (slots enumerate (sequence, chunk) pairs; see slot_to_chunk)
__device__ __forceinline__ int64_t slot_base(const int32_t* cu, int n) {
  return cu ? (int64_t)cu[n] / C + n : 0;
}

// ------------------------------------------------------------------ column recurrences

// One CTA: sequence n, value head j, 32 state columns; thread = (column, quarter of the rows).
// Forward: stores the state entering every chunk, as states[slot][j][v][i] (a column of the
// state contiguous).  Reverse: stores the gradient of the state leaving every chunk in the same
// layout, and dh0.
template <int K, bool REVERSE>
__global__ void __launch_bounds__(kColThreads) column_kernel(BwdArgs a) {
  constexpr int RPL = K / 4;
  const int nj = blockIdx.x, n = nj / a.hv, j = nj % a.hv, kh = j / (a.hv / a.hk);
  const int v = blockIdx.y * 32 + (threadIdx.x >> 2), part = threadIdx.x & 3;
  const int r0 = part * RPL;
  int64_t t0, t1;
  if (!seq_bounds(a.cu, n, a.T, a.status, t0, t1)) return;
  const int64_t KV = (int64_t)K * a.V;
  float h[RPL];
  const float* init = REVERSE ? a.dh_final : a.h0;
#pragma unroll
  for (int i = 0; i < RPL; ++i)
    h[i] = init ? init[((int64_t)n * a.hv + j) * KV + (int64_t)(r0 + i) * a.V + v] : 0.f;
  float* store = REVERSE ? a.dstates : a.states;
  const int64_t nc = (t1 - t0 + C - 1) / C, sb = slot_base(a.cu, n);
  for (int64_t ci = 0; ci < nc; ++ci) {
    const int64_t c = REVERSE ? nc - 1 - ci : ci;
    const int64_t c0 = t0 + c * C, c1 = (c0 + C < t1) ? c0 + C : t1;
    float* dst = store + (((sb + c) * a.hv + j) * a.V + v) * K + r0;
#pragma unroll
    for (int i = 0; i < RPL; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(h[i], h[i + 1], h[i + 2], h[i + 3]);
    for (int64_t s = 0; s < c1 - c0; ++s) {
      const int64_t t = REVERSE ? c1 - 1 - s : c0 + s;
      const float alpha = __expf(a.g[t * a.hv + j]), beta = a.beta[t * a.hv + j];
      float kk[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i) kk[i] = ld_io(a.k, (t * a.hk + kh) * K + r0 + i, a.bf16);
      if (REVERSE) {  // F = dh + q dout^T;  dd = k . F;  dh <- alpha (F - beta k dd)
        const float dov = ld_io(a.dout, (t * a.hv + j) * a.V + v, a.bf16);
#pragma unroll
        for (int i = 0; i < RPL; ++i) h[i] = fmaf(ld_io(a.q, (t * a.hk + kh) * K + r0 + i, a.bf16), dov, h[i]);
      }
      float p = 0.f;
#pragma unroll
      for (int i = 0; i < RPL; ++i) p = fmaf(kk[i], h[i], p);
      p += __shfl_xor_sync(0xffffffffu, p, 1);
      p += __shfl_xor_sync(0xffffffffu, p, 2);
      if (REVERSE) {
        const float bd = beta * p;
#pragma unroll
        for (int i = 0; i < RPL; ++i) h[i] = alpha * fmaf(-kk[i], bd, h[i]);
      } else {  // delta = beta (v - alpha p);  h <- alpha h + k delta
        const float d = beta * (ld_io(a.v, (t * a.hv + j) * a.V + v, a.bf16) - alpha * p);
#pragma unroll
        for (int i = 0; i < RPL; ++i) h[i] = fmaf(kk[i], d, alpha * h[i]);
      }
    }
  }
  if (REVERSE && a.dh0) {
#pragma unroll
    for (int i = 0; i < RPL; ++i) a.dh0[((int64_t)n * a.hv + j) * KV + (int64_t)(r0 + i) * a.V + v] = h[i];
  }
}

// ------------------------------------------------------------------ per-chunk gradients

// out[i][c] (+)= sum_y A(i, y) B(y, c) for i < M, c < N: every thread takes output elements in
// turn; operands are read through accessor functors (smem or the CTA's workspace slice).
template <typename FA, typename FB, typename FO>
__device__ __forceinline__ void mm(int M, int N, int Y, FA A, FB B, FO out) {
  for (int e = threadIdx.x; e < M * N; e += blockDim.x) {
    const int i = e / N, c = e % N;
    float s0 = 0.f, s1 = 0.f;
    int y = 0;
    for (; y + 1 < Y; y += 2) {
      s0 = fmaf(A(i, y), B(y, c), s0);
      s1 = fmaf(A(i, y + 1), B(y + 1, c), s1);
    }
    if (y < Y) s0 = fmaf(A(i, y), B(y, c), s0);
    out(i, c, s0 + s1);
  }
}

struct GradSmem {
  float KK[C][C + 1], QK[C][C + 1], Am[C][C + 1], At[C][C + 1];  // A, attn; then dA o Gamma etc.
  float dA[C][C + 1], dat[C][C + 1];
  float G[C], eG[C], ekt[C], b[C], dG[C], red[C];
  float scal[4];
};

// floats of one CTA's workspace slice: K S, Q S, R, delta, d_delta (then dB), dout as [C][V];
// k, q, delta D^T as [C][K]
template <int K, int V>
__host__ __device__ constexpr int64_t grad_slice() { return 6 * (int64_t)C * V + 3 * (int64_t)C * K; }

// One CTA per (chunk slot, value head); grid-stride over the units.
template <int K, int V>
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
  float* DD = DL + C * V;    // [C][V]  d_delta, then dB in place
  float* DO = DD + C * V;    // [C][V]  dout (fp32)
  float* KF = DO + C * V;    // [C][K]  k (fp32)
  float* QF = KF + C * K;    // [C][K]  q (fp32)
  float* X = QF + C * K;     // [C][K]  delta D^T
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
    // ---- inputs: decays (running sum by one warp), q, k, dout as fp32
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
    for (int e = tid; e < C * K; e += kGradThreads) {
      const int t = e / K, i = e % K;
      const bool ok = t < L;
      KF[e] = ok ? ld_io(a.k, ((t0 + t) * a.hk + kh) * K + i, a.bf16) : 0.f;
      QF[e] = ok ? ld_io(a.q, ((t0 + t) * a.hk + kh) * K + i, a.bf16) : 0.f;
    }
    for (int e = tid; e < C * V; e += kGradThreads) {
      const int t = e / V, c = e % V;
      DO[e] = t < L ? ld_io(a.dout, ((t0 + t) * a.hv + j) * V + c, a.bf16) : 0.f;
    }
    __syncthreads();
    // ---- K K^T, Q K^T; K S, Q S
    mm(C, C, K, [&](int t, int y) { return KF[t * K + y]; }, [&](int y, int s) { return KF[s * K + y]; },
       [&](int t, int s, float x) { sm.KK[t][s] = x; });
    mm(C, C, K, [&](int t, int y) { return QF[t * K + y]; }, [&](int y, int s) { return KF[s * K + y]; },
       [&](int t, int s, float x) { sm.QK[t][s] = x; });
    mm(C, V, K, [&](int t, int y) { return KF[t * K + y]; }, [&](int y, int c) { return Sx[c * K + y]; },
       [&](int t, int c, float x) { KS[t * V + c] = x; });
    mm(C, V, K, [&](int t, int y) { return QF[t * K + y]; }, [&](int y, int c) { return Sx[c * K + y]; },
       [&](int t, int c, float x) { QS[t * V + c] = x; });
    __syncthreads();
    // ---- A, attn (rows >= L are zero); R = V - e^G K S
    for (int e = tid; e < C * C; e += kGradThreads) {
      const int t = e / C, s = e % C;
      const bool in = t < L && s < L;
      const float gam = __expf(sm.G[t] - sm.G[s < t ? s : t]);  // Gamma for s <= t
      sm.Am[t][s] = (in && s < t) ? sm.b[t] * gam * sm.KK[t][s] : 0.f;
      sm.At[t][s] = (in && s <= t) ? gam * sm.QK[t][s] : 0.f;
    }
    for (int e = tid; e < C * V; e += kGradThreads) {
      const int t = e / V, c = e % V;
      R[e] = t < L ? ld_io(a.v, ((t0 + t) * a.hv + j) * V + c, a.bf16) - sm.eG[t] * KS[e] : 0.f;
    }
    __syncthreads();
    // ---- delta = (I + A)^-1 diag(beta) R: forward substitution, one column per thread
    for (int c = tid; c < V; c += kGradThreads) {
      for (int t = 0; t < L; ++t) {
        float x = sm.b[t] * R[t * V + c];
        for (int s = 0; s < t; ++s) x = fmaf(-sm.Am[t][s], DL[s * V + c], x);
        DL[t * V + c] = x;
      }
      for (int t = L; t < C; ++t) DL[t * V + c] = 0.f;
    }
    __syncthreads();
    // ---- d_delta = attn^T dO + Kt D
    mm(C, V, C, [&](int t, int s) { return sm.At[s][t]; }, [&](int s, int c) { return DO[s * V + c]; },
       [&](int t, int c, float x) { DD[t * V + c] = x; });
    __syncthreads();
    mm(C, V, K, [&](int t, int y) { return sm.ekt[t] * KF[t * K + y]; }, [&](int y, int c) { return Dx[c * K + y]; },
       [&](int t, int c, float x) { DD[t * V + c] += t < L ? x : 0.f; });
    __syncthreads();
    // ---- dB = (I + A)^-T d_delta: back substitution in place
    for (int c = tid; c < V; c += kGradThreads) {
      for (int t = L - 1; t >= 0; --t) {
        float x = DD[t * V + c];
        for (int s = t + 1; s < L; ++s) x = fmaf(-sm.Am[s][t], DD[s * V + c], x);
        DD[t * V + c] = x;
      }
    }
    __syncthreads();
    // ---- dA = -(dB delta^T) o strictly lower, dattn = (dO delta^T) o lower;  dv = beta dB
    mm(C, C, V, [&](int t, int c) { return DD[t * V + c]; }, [&](int c, int s) { return DL[s * V + c]; },
       [&](int t, int s, float x) { sm.dA[t][s] = (s < t && t < L) ? -x : 0.f; });
    mm(C, C, V, [&](int t, int c) { return DO[t * V + c]; }, [&](int c, int s) { return DL[s * V + c]; },
       [&](int t, int s, float x) { sm.dat[t][s] = (s <= t && t < L) ? x : 0.f; });
    for (int e = tid; e < L * V; e += kGradThreads) {
      const int t = e / V, c = e % V;
      st_io(a.dv, ((t0 + t) * a.hv + j) * V + c, sm.b[t] * DD[e], a.bf16);
    }
    __syncthreads();
    // ---- per-row sums: dbeta and the decay gradient dG
    for (int t = tid; t < C; t += kGradThreads) {
      float db = 0.f, dg = 0.f;
      if (t < L) {
        for (int c = 0; c < V; ++c) {
          db = fmaf(DD[t * V + c], R[t * V + c], db);
          dg = fmaf(-sm.b[t] * sm.eG[t] * DD[t * V + c], KS[t * V + c], dg);
          dg = fmaf(sm.eG[t] * DO[t * V + c], QS[t * V + c], dg);
        }
        for (int s = 0; s < L; ++s) {
          const float gam = __expf(sm.G[t] - sm.G[s < t ? s : t]);
          if (s < t) db = fmaf(sm.dA[t][s] * gam, sm.KK[t][s], db);
          dg += sm.dA[t][s] * sm.Am[t][s] - sm.dA[s][t] * sm.Am[s][t];
          dg += sm.dat[t][s] * sm.At[t][s] - sm.dat[s][t] * sm.At[s][t];
        }
        a.dbeta[(t0 + t) * a.hv + j] = db;
      }
      sm.dG[t] = dg;
    }
    __syncthreads();
    // ---- dA o Gamma and dattn o Gamma in place
    for (int e = tid; e < C * C; e += kGradThreads) {
      const int t = e / C, s = e % C;
      const float gam = s <= t ? __expf(sm.G[t] - sm.G[s]) : 0.f;
      sm.dA[t][s] *= gam;
      sm.dat[t][s] *= gam;
    }
    __syncthreads();
    // ---- delta D^T into X ([C][K] rows): its row sums against Kt go to dG, dk takes it
    mm(C, K, V, [&](int t, int c) { return DL[t * V + c]; }, [&](int c, int i) { return Dx[c * K + i]; },
       [&](int t, int i, float x) { X[t * K + i] = x; });
    __syncthreads();
    if (tid < 32) {  // dG_t -= Kt_t . (delta D^T)_t;  dG_L += sum of it + e^{G_L} <D, S>
      float tot = 0.f;
      for (int t = tid; t < L; t += 32) {
        float s = 0.f;
        for (int i = 0; i < K; ++i) s = fmaf(KF[t * K + i], X[t * K + i], s);
        s *= sm.ekt[t];
        sm.dG[t] -= s;
        tot += s;
      }
      float ds = 0.f;
      for (int e = tid; e < K * V; e += 32) ds = fmaf(Sx[e], Dx[e], ds);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        ds += __shfl_xor_sync(0xffffffffu, ds, o);
      }
      __syncwarp();
      if (tid == 0) sm.dG[L - 1] += tot + sm.scal[0] * ds;
    }
    __syncthreads();
    if (tid < 32) {  // dg_t = sum_{u >= t} dG_u (reverse running sum over the chunk)
      float x0 = sm.dG[63 - tid], x1 = sm.dG[31 - tid];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (tid >= o) { x0 += y0; x1 += y1; }
      }
      x1 += __shfl_sync(0xffffffffu, x0, 31);
      const int r0 = 63 - tid, r1 = 31 - tid;  // rows of x0, x1
      if (r0 < L) a.dg[(t0 + r0) * a.hv + j] = x0;
      if (r1 < L) a.dg[(t0 + r1) * a.hv + j] = x1;
    }
    // ---- dq = diag(e^G) dO S^T + (dattn o Gamma) K;  per value head, summed over the group later
    float* dqv = a.dqv + (t0 * a.hv + j) * (int64_t)K;
    float* dkv = a.dkv + (t0 * a.hv + j) * (int64_t)K;
    const int64_t rs = (int64_t)a.hv * K;  // row stride of dqv, dkv
    mm(L, K, V, [&](int t, int c) { return DO[t * V + c]; }, [&](int c, int i) { return Sx[c * K + i]; },
       [&](int t, int i, float x) { dqv[t * rs + i] = sm.eG[t] * x; });
    __syncthreads();
    mm(L, K, L, [&](int t, int s) { return sm.dat[t][s]; }, [&](int s, int i) { return KF[s * K + i]; },
       [&](int t, int i, float x) { dqv[t * rs + i] += x; });
    // ---- dk = -diag(beta e^G) dB S^T + diag(beta) (dA o Gamma) K + (dA o Gamma)^T diag(beta) K
    //          + (dattn o Gamma)^T Q + diag(e^{G_L - G}) delta D^T
    mm(L, K, V, [&](int t, int c) { return DD[t * V + c]; }, [&](int c, int i) { return Sx[c * K + i]; },
       [&](int t, int i, float x) { dkv[t * rs + i] = sm.ekt[t] * X[t * K + i] - sm.b[t] * sm.eG[t] * x; });
    __syncthreads();
    mm(L, K, L, [&](int t, int s) { return sm.dA[t][s]; }, [&](int s, int i) { return KF[s * K + i]; },
       [&](int t, int i, float x) { dkv[t * rs + i] += sm.b[t] * x; });
    __syncthreads();
    mm(L, K, L, [&](int t, int s) { return sm.dA[s][t] * sm.b[s]; }, [&](int s, int i) { return KF[s * K + i]; },
       [&](int t, int i, float x) { dkv[t * rs + i] += x; });
    __syncthreads();
    mm(L, K, L, [&](int t, int s) { return sm.dat[s][t]; }, [&](int s, int i) { return QF[s * K + i]; },
       [&](int t, int i, float x) { dkv[t * rs + i] += x; });
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
  const dim3 cg((unsigned)(a.N * a.hv), (unsigned)(V / 32));
  column_kernel<K, false><<<cg, kColThreads, 0, s>>>(a);
  column_kernel<K, true><<<cg, kColThreads, 0, s>>>(a);
  cudaError_t e = cudaFuncSetAttribute(chunk_grad_kernel<K, V>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(GradSmem));
  if (e != cudaSuccess) return e;
  chunk_grad_kernel<K, V><<<a.grad_ctas, kGradThreads, sizeof(GradSmem), s>>>(a);
  group_sum_kernel<<<1024, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int64_t bwd_slots(int64_t T, int N) { return T / kChunk + N; }

size_t bwd_scratch_floats(int K, int V, int ctas) {
  return (size_t)ctas * (6 * (size_t)kChunk * V + 3 * (size_t)kChunk * K);
}

cudaError_t backward(const BwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.K == 128 && a.V == 128) return launch_all<128, 128>(a, s);
  if (a.K == 128 && a.V == 64) return launch_all<128, 64>(a, s);
  if (a.K == 64 && a.V == 128) return launch_all<64, 128>(a, s);
  return launch_all<64, 64>(a, s);
}

}  // namespace gdn
