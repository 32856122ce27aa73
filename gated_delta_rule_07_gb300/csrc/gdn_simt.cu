// gdn_simt.cu -- SIMT (CUDA-core, fp32 arithmetic) kernels for every step of the chunked
// gated delta rule forward.  They serve the fp32 I/O path (whose tolerance needs fp32
// operands) and any shape the tensor-core kernels do not cover.
//
// Chunk factors follow "Add context parallelism to the Gated Delta Net (Qwen3-Next /
// Qwen3.5)", section "Why" (the affine chunk map) with the definitions of gdn.h; the
// segment phases follow its section "Implementation".
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int C = kChunk;
constexpr int kColBlock = 32;  // state columns per CTA (columns of h, M, U are independent)
constexpr int kScanCols = 16;  // the scan: narrower blocks, twice the CTAs (two per SM), for its latency

// ------------------------------------------------------------------ validation

__global__ void validate_cu_kernel(const int32_t* cu, int N, int64_t T, int32_t* st) {
  bool bad = false;
  if (threadIdx.x == 0 && (cu[0] != 0 || (int64_t)cu[N] != T)) bad = true;
  for (int n = threadIdx.x; n < N; n += blockDim.x)
    if (cu[n + 1] < cu[n]) bad = true;
  if (bad) set_status(st, GDN_ERR_DEVICE_INPUT);
}

// ------------------------------------------------------------------ prepare

// One CTA per (chunk slot, value head): loads the chunk's k, v, g, beta, forms the masked
// gram A, inverts the unit lower-triangular (I + A) by forward substitution and writes
// w = T diag(beta e^G) K, u = T diag(beta) V and the within-chunk cumulative decay.
template <typename TIO, int KD, int VD>
__global__ void __launch_bounds__(kThreads) simt_prepare_kernel(Args a) {
  constexpr int KP = KD + 1, VP = VD + 1, CP = C + 1;
  extern __shared__ float sm[];
  float* ks = sm;            // [C][KP]
  float* vs = ks + C * KP;   // [C][VP]
  float* A = vs + C * VP;    // [C][CP]
  float* Tm = A + C * CP;    // [C][CP]
  float* G = Tm + C * CP;    // [C]
  float* bs = G + C;         // [C]  beta
  float* bw = bs + C;        // [C]  beta e^G

  const int j = blockIdx.y;
  int n;
  int64_t chunk;
  if (!slot_to_chunk(a.cu, a.N, a.T, blockIdx.x, n, chunk)) return;
  int64_t sb, se;
  if (!seq_bounds(a.cu, n, a.T, a.status, sb, se)) return;
  const int64_t t0 = sb + chunk * C;
  const int L = (int)((se - t0) < C ? (se - t0) : C);
  const int kh = j / (a.hv / a.hk);
  const TIO* k = static_cast<const TIO*>(a.k);
  const TIO* v = static_cast<const TIO*>(a.v);
  const int tid = threadIdx.x;

  for (int e = tid; e < C * KD; e += kThreads) {
    const int t = e / KD, i = e % KD;
    ks[t * KP + i] = t < L ? to_f32(k[((t0 + t) * a.hk + kh) * KD + i]) : 0.f;
  }
  for (int e = tid; e < C * VD; e += kThreads) {
    const int t = e / VD, c = e % VD;
    vs[t * VP + c] = t < L ? to_f32(v[((t0 + t) * a.hv + j) * VD + c]) : 0.f;
  }
  if (tid < C) bs[tid] = tid < L ? a.beta[(t0 + tid) * a.hv + j] : 0.f;
  if (tid == 0) {
    float acc = 0.f;
    for (int t = 0; t < C; ++t) {
      acc += t < L ? a.g[(t0 + t) * a.hv + j] : 0.f;
      G[t] = acc;
    }
  }
  __syncthreads();
  if (tid < C) bw[tid] = bs[tid] * __expf(G[tid]);
  // A[t][i] = beta_t e^{G_t - G_i} (k_t . k_i) for i < t
  for (int e = tid; e < C * C; e += kThreads) {
    const int t = e / C, i = e % C;
    float x = 0.f;
    if (i < t) {
      for (int d = 0; d < KD; ++d) x += ks[t * KP + d] * ks[i * KP + d];
      x *= bs[t] * __expf(G[t] - G[i]);
    }
    A[t * CP + i] = x;
    Tm[t * CP + i] = (t == i) ? 1.f : 0.f;
  }
  __syncthreads();
  // Forward substitution, column-parallel: column c of T depends only on column c, so four
  // lanes per column split the inner sum and combine with shuffles.
  {
    const int c = tid >> 2, sub = tid & 3;
    for (int t = 1; t < C; ++t) {
      float x = 0.f;
      for (int i = sub; i < t; i += 4) x += A[t * CP + i] * Tm[i * CP + c];
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      if (sub == 0 && t > c) Tm[t * CP + c] = -x;
      __syncwarp();
    }
  }
  __syncthreads();
  float* w = static_cast<float*>(a.w_out);
  float* u = static_cast<float*>(a.u_out);
  for (int e = tid; e < C * KD; e += kThreads) {
    const int t = e / KD, i = e % KD;
    if (t >= L) continue;
    float x = 0.f;
    for (int s = 0; s <= t; ++s) x += Tm[t * CP + s] * bw[s] * ks[s * KP + i];
    w[((t0 + t) * a.hv + j) * KD + i] = x;
  }
  for (int e = tid; e < C * VD; e += kThreads) {
    const int t = e / VD, c = e % VD;
    if (t >= L) continue;
    float x = 0.f;
    for (int s = 0; s <= t; ++s) x += Tm[t * CP + s] * bs[s] * vs[s * VP + c];
    u[((t0 + t) * a.hv + j) * VD + c] = x;
  }
  if (tid < L) a.gcum_out[(t0 + tid) * a.hv + j] = G[tid];
}

// ------------------------------------------------------------------ phase 1

// One CTA per (segment, value head, block of 32 columns of X = [M | U]).  From X = [I | 0],
// per chunk: D = [0 | u] - w X, X <- gamma X + k_tilde^T D (the low-rank composition of M
// and the chunk map of the zero-start state U share this form).
template <typename TIO, int KD, int VD>
__global__ void __launch_bounds__(kThreads) simt_summary_kernel(Args a) {
  constexpr int KP = KD + 1, XP = kColBlock + 1;
  extern __shared__ float sm[];
  float* ws = sm;              // [C][KP]
  float* kt = ws + C * KP;     // [C][KP]   k_tilde
  float* Xs = kt + C * KP;     // [KD][XP]
  float* D = Xs + KD * XP;     // [C][XP]
  float* us = D + C * XP;      // [C][XP]
  float* G = us + C * XP;      // [C]

  const int seg = blockIdx.x, j = blockIdx.y, cb = blockIdx.z;
  const int n = seg / a.P, r = seg % a.P;
  const int col0 = cb * kColBlock;             // column of X
  const bool is_u = col0 >= KD;
  const int ucol0 = col0 - KD;
  const int kh = j / (a.hv / a.hk);
  const int tid = threadIdx.x;
  int64_t sb, se;
  if (!seq_bounds(a.cu, n, a.T, a.status, sb, se)) return;
  int64_t c0, c1;
  segment_chunks(se - sb, a.P, r, c0, c1);
  const TIO* k = static_cast<const TIO*>(a.k);
  const float* w = static_cast<const float*>(a.w);
  const float* u = static_cast<const float*>(a.u);

  for (int e = tid; e < KD * kColBlock; e += kThreads) {
    const int i = e / kColBlock, c = e % kColBlock;
    Xs[i * XP + c] = (!is_u && i == col0 + c) ? 1.f : 0.f;
  }
  for (int64_t ch = c0; ch < c1; ++ch) {
    const int64_t t0 = sb + ch * C;
    const int L = (int)((se - t0) < C ? (se - t0) : C);
    __syncthreads();
    if (tid < C) G[tid] = tid < L ? a.gcum[(t0 + tid) * a.hv + j] : 0.f;
    __syncthreads();
    const float GL = G[L - 1];
    for (int e = tid; e < C * KD; e += kThreads) {
      const int t = e / KD, i = e % KD;
      float wv = 0.f, kv = 0.f;
      if (t < L) {
        wv = w[((t0 + t) * a.hv + j) * KD + i];
        kv = to_f32(k[((t0 + t) * a.hk + kh) * KD + i]) * __expf(GL - G[t]);
      }
      ws[t * KP + i] = wv;
      kt[t * KP + i] = kv;
    }
    if (is_u)
      for (int e = tid; e < C * kColBlock; e += kThreads) {
        const int t = e / kColBlock, c = e % kColBlock;
        us[t * XP + c] = t < L ? u[((t0 + t) * a.hv + j) * VD + ucol0 + c] : 0.f;
      }
    __syncthreads();
    for (int e = tid; e < C * kColBlock; e += kThreads) {
      const int t = e / kColBlock, c = e % kColBlock;
      float x = is_u ? us[t * XP + c] : 0.f;
      for (int i = 0; i < KD; ++i) x -= ws[t * KP + i] * Xs[i * XP + c];
      D[t * XP + c] = x;
    }
    __syncthreads();
    const float gamma = __expf(GL);
    for (int e = tid; e < KD * kColBlock; e += kThreads) {
      const int i = e / kColBlock, c = e % kColBlock;
      float x = 0.f;
      for (int t = 0; t < C; ++t) x += kt[t * KP + i] * D[t * XP + c];
      Xs[i * XP + c] = gamma * Xs[i * XP + c] + x;
    }
  }
  __syncthreads();
  for (int e = tid; e < KD * kColBlock; e += kThreads) {
    const int i = e / kColBlock, c = e % kColBlock;
    if (is_u)
      a.U_out[(((int64_t)seg * a.hv + j) * KD + i) * VD + ucol0 + c] = Xs[i * XP + c];
    else
      a.M_out[(((int64_t)seg * a.hv + j) * KD + i) * KD + col0 + c] = Xs[i * XP + c];
  }
}

// ------------------------------------------------------------------ phase 2

// One CTA per (sequence, value head, block of kScanCols state columns); serial over segments:
// h_in[r] = h, h <- M_r h + U_r.  Each M_r (KD x KD fp32) is read as a batch of 16-byte loads
// into registers one segment ahead, so that its latency overlaps the previous step; a thread
// owns one column and NO rows of the product, whose sums run side by side.
template <int KD, int VD>
__global__ void __launch_bounds__(kThreads) simt_scan_kernel(Args a) {
  constexpr int KP = KD + 4, XP = kScanCols + 1;  // 16-byte rows for M; conflict-free reads
  constexpr int NV = KD * KD / 4 / kThreads;      // float4 of M per thread
  constexpr int RS = kThreads / kScanCols, NO = KD / RS;  // row stride, rows per thread
  static_assert(NV * 4 * kThreads == KD * KD && RS * NO == KD, "the CTA tiles M and h");
  extern __shared__ float sm[];
  float* Ms = sm;              // [KD][KP]
  float* hs = Ms + KD * KP;    // [KD][XP]
  const int n = blockIdx.x, j = blockIdx.y, col0 = blockIdx.z * kScanCols;
  const int tid = threadIdx.x, c = tid % kScanCols, i0 = tid / kScanCols;
  // the segments whose M is read: all but the last, unless the last step feeds h_final
  const int steps = a.h_final ? a.P : a.P - 1;
  float4 mv[NV];
  auto load_m = [&](int r) {
    const float4* src = reinterpret_cast<const float4*>(
        a.M + ((((int64_t)n * a.P + r) * a.hv + j) * KD) * KD);
#pragma unroll
    for (int k = 0; k < NV; ++k) mv[k] = src[tid + kThreads * k];
  };
  if (steps > 0) load_m(0);
  float h[NO];  // h[i0 + RS m][c]
#pragma unroll
  for (int m = 0; m < NO; ++m)
    h[m] = a.h0 ? a.h0[(((int64_t)n * a.hv + j) * KD + i0 + RS * m) * VD + col0 + c] : 0.f;
  for (int r = 0; r < a.P; ++r) {
    const int64_t base = (((int64_t)n * a.P + r) * a.hv + j) * KD;  // row 0 of segment r
    if (a.h_in_out) {
#pragma unroll
      for (int m = 0; m < NO; ++m) a.h_in_out[(base + i0 + RS * m) * VD + col0 + c] = h[m];
    }
    if (r == steps) return;  // the last summary only feeds h_final
    float u[NO];
#pragma unroll
    for (int m = 0; m < NO; ++m) u[m] = a.U[(base + i0 + RS * m) * VD + col0 + c];
    __syncthreads();  // the previous step has read Ms and hs
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int e = 4 * (tid + kThreads * k), i = e / KD, b = e % KD;
      *reinterpret_cast<float4*>(&Ms[i * KP + b]) = mv[k];
    }
#pragma unroll
    for (int m = 0; m < NO; ++m) hs[(i0 + RS * m) * XP + c] = h[m];
    __syncthreads();
    if (r + 1 < steps) load_m(r + 1);  // lands while this step computes
#pragma unroll 4
    for (int b = 0; b < KD; ++b) {
      const float hb = hs[b * XP + c];
#pragma unroll
      for (int m = 0; m < NO; ++m) u[m] += Ms[(i0 + RS * m) * KP + b] * hb;
    }
#pragma unroll
    for (int m = 0; m < NO; ++m) h[m] = u[m];
  }
  if (a.h_final) {
#pragma unroll
    for (int m = 0; m < NO; ++m)
      a.h_final[(((int64_t)n * a.hv + j) * KD + i0 + RS * m) * VD + col0 + c] = h[m];
  }
}

// ------------------------------------------------------------------ phase 3

// One CTA per (segment, value head, block of 32 state columns).  From h = h_in, per chunk:
// delta = u - w h;  o = q_g h + attn_i delta;  h <- gamma h + k_tilde^T delta.
template <typename TIO, int KD, int VD>
__global__ void __launch_bounds__(kThreads) simt_emit_kernel(Args a) {
  constexpr int KP = KD + 1, XP = kColBlock + 1, CP = C + 1;
  extern __shared__ float sm[];
  float* qs = sm;              // [C][KP]  q, then q_g
  float* ks = qs + C * KP;     // [C][KP]  k, then k_tilde
  float* ws = ks + C * KP;     // [C][KP]
  float* att = ws + C * KP;    // [C][CP]
  float* hs = att + C * CP;    // [KD][XP]
  float* D = hs + KD * XP;     // [C][XP]
  float* us = D + C * XP;      // [C][XP]
  float* G = us + C * XP;      // [C]

  const int seg = blockIdx.x, j = blockIdx.y, col0 = blockIdx.z * kColBlock;
  const int n = seg / a.P, r = seg % a.P;
  const int kh = j / (a.hv / a.hk);
  const int tid = threadIdx.x;
  int64_t sb, se;
  if (!seq_bounds(a.cu, n, a.T, a.status, sb, se)) return;
  int64_t c0, c1;
  segment_chunks(se - sb, a.P, r, c0, c1);
  const TIO* q = static_cast<const TIO*>(a.q);
  const TIO* k = static_cast<const TIO*>(a.k);
  const float* w = static_cast<const float*>(a.w);
  const float* u = static_cast<const float*>(a.u);
  TIO* out = static_cast<TIO*>(a.out);

  for (int e = tid; e < KD * kColBlock; e += kThreads) {
    const int i = e / kColBlock, c = e % kColBlock;
    hs[i * XP + c] = a.h_in ? a.h_in[(((int64_t)seg * a.hv + j) * KD + i) * VD + col0 + c] : 0.f;
  }
  for (int64_t ch = c0; ch < c1; ++ch) {
    const int64_t t0 = sb + ch * C;
    const int L = (int)((se - t0) < C ? (se - t0) : C);
    __syncthreads();
    if (tid < C) G[tid] = tid < L ? a.gcum[(t0 + tid) * a.hv + j] : 0.f;
    for (int e = tid; e < C * KD; e += kThreads) {
      const int t = e / KD, i = e % KD;
      const bool ok = t < L;
      qs[t * KP + i] = ok ? to_f32(q[((t0 + t) * a.hk + kh) * KD + i]) : 0.f;
      ks[t * KP + i] = ok ? to_f32(k[((t0 + t) * a.hk + kh) * KD + i]) : 0.f;
      ws[t * KP + i] = ok ? w[((t0 + t) * a.hv + j) * KD + i] : 0.f;
    }
    for (int e = tid; e < C * kColBlock; e += kThreads) {
      const int t = e / kColBlock, c = e % kColBlock;
      us[t * XP + c] = t < L ? u[((t0 + t) * a.hv + j) * VD + col0 + c] : 0.f;
    }
    __syncthreads();
    const float GL = G[L - 1];
    for (int e = tid; e < C * C; e += kThreads) {
      const int t = e / C, s = e % C;
      float x = 0.f;
      if (s <= t) {
        for (int i = 0; i < KD; ++i) x += qs[t * KP + i] * ks[s * KP + i];
        x *= __expf(G[t] - G[s]);
      }
      att[t * CP + s] = x;
    }
    for (int e = tid; e < C * kColBlock; e += kThreads) {
      const int t = e / kColBlock, c = e % kColBlock;
      float x = us[t * XP + c];
      for (int i = 0; i < KD; ++i) x -= ws[t * KP + i] * hs[i * XP + c];
      D[t * XP + c] = x;
    }
    __syncthreads();
    for (int e = tid; e < C * KD; e += kThreads) {
      const int t = e / KD, i = e % KD;
      qs[t * KP + i] *= __expf(G[t]);
      ks[t * KP + i] *= __expf(GL - G[t]);
    }
    __syncthreads();
    for (int e = tid; e < C * kColBlock; e += kThreads) {
      const int t = e / kColBlock, c = e % kColBlock;
      if (t >= L) continue;
      float x = 0.f;
      for (int i = 0; i < KD; ++i) x += qs[t * KP + i] * hs[i * XP + c];
      for (int s = 0; s <= t; ++s) x += att[t * CP + s] * D[s * XP + c];
      out[((t0 + t) * a.hv + j) * VD + col0 + c] = from_f32<TIO>(x);
    }
    __syncthreads();
    const float gamma = __expf(GL);
    for (int e = tid; e < KD * kColBlock; e += kThreads) {
      const int i = e / kColBlock, c = e % kColBlock;
      float x = 0.f;
      for (int t = 0; t < C; ++t) x += ks[t * KP + i] * D[t * XP + c];
      hs[i * XP + c] = gamma * hs[i * XP + c] + x;
    }
  }
  __syncthreads();
  if (a.h_final && r == a.P - 1)
    for (int e = tid; e < KD * kColBlock; e += kThreads) {
      const int i = e / kColBlock, c = e % kColBlock;
      a.h_final[(((int64_t)n * a.hv + j) * KD + i) * VD + col0 + c] = hs[i * XP + c];
    }
}

// ------------------------------------------------------------------ dispatch

template <typename Kern>
cudaError_t launch(Kern kern, dim3 grid, size_t smem, cudaStream_t s, const Args& a) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename TIO, int KD, int VD>
struct Simt {
  static cudaError_t prepare(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * (C * (KD + 1) + C * (VD + 1) + 2 * C * (C + 1) + 3 * C);
    const int64_t slots = a.T / C + a.N;
    return launch(simt_prepare_kernel<TIO, KD, VD>, dim3((unsigned)slots, a.hv, 1), smem, s, a);
  }
  static cudaError_t summary(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(float) *
        (2 * C * (KD + 1) + KD * (kColBlock + 1) + 2 * C * (kColBlock + 1) + C);
    return launch(simt_summary_kernel<TIO, KD, VD>,
                  dim3((unsigned)(a.N * a.P), a.hv, (KD + VD) / kColBlock), smem, s, a);
  }
  static cudaError_t scan(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * (KD * (KD + 4) + KD * (kScanCols + 1));
    return launch(simt_scan_kernel<KD, VD>, dim3((unsigned)a.N, a.hv, VD / kScanCols), smem, s,
                  a);
  }
  static cudaError_t emit(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * (3 * C * (KD + 1) + C * (C + 1) + KD * (kColBlock + 1) +
                                         2 * C * (kColBlock + 1) + C);
    return launch(simt_emit_kernel<TIO, KD, VD>,
                  dim3((unsigned)(a.N * a.P), a.hv, VD / kColBlock), smem, s, a);
  }
};

template <template <typename, int, int> class Op, typename... R>
cudaError_t dispatch(const Args& a, cudaStream_t s) {
  const int key = (a.K == 128 ? 2 : 0) + (a.V == 128 ? 1 : 0);
  if (a.bf16) {
    switch (key) {
      case 0: return Op<__nv_bfloat16, 64, 64>::run(a, s);
      case 1: return Op<__nv_bfloat16, 64, 128>::run(a, s);
      case 2: return Op<__nv_bfloat16, 128, 64>::run(a, s);
      default: return Op<__nv_bfloat16, 128, 128>::run(a, s);
    }
  }
  switch (key) {
    case 0: return Op<float, 64, 64>::run(a, s);
    case 1: return Op<float, 64, 128>::run(a, s);
    case 2: return Op<float, 128, 64>::run(a, s);
    default: return Op<float, 128, 128>::run(a, s);
  }
}

template <typename TIO, int KD, int VD> struct PrepOp {
  static cudaError_t run(const Args& a, cudaStream_t s) { return Simt<TIO, KD, VD>::prepare(a, s); }
};
template <typename TIO, int KD, int VD> struct SumOp {
  static cudaError_t run(const Args& a, cudaStream_t s) { return Simt<TIO, KD, VD>::summary(a, s); }
};
template <typename TIO, int KD, int VD> struct ScanOp {
  static cudaError_t run(const Args& a, cudaStream_t s) { return Simt<TIO, KD, VD>::scan(a, s); }
};
template <typename TIO, int KD, int VD> struct EmitOp {
  static cudaError_t run(const Args& a, cudaStream_t s) { return Simt<TIO, KD, VD>::emit(a, s); }
};

}  // namespace

cudaError_t launch_validate_cu(const Args& a, cudaStream_t s) {
  if (a.cu == nullptr) return cudaSuccess;
  validate_cu_kernel<<<1, 256, 0, s>>>(a.cu, a.N, a.T, a.status);
  return cudaGetLastError();
}

cudaError_t simt_prepare(const Args& a, cudaStream_t s) { return dispatch<PrepOp>(a, s); }
cudaError_t simt_summary(const Args& a, cudaStream_t s) { return dispatch<SumOp>(a, s); }
cudaError_t simt_scan(const Args& a, cudaStream_t s) { return dispatch<ScanOp>(a, s); }
cudaError_t simt_emit(const Args& a, cudaStream_t s) { return dispatch<EmitOp>(a, s); }

}  // namespace gdn
