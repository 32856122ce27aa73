// gdn_decode.cu -- one decode step of the gated delta rule over a pool of per-slot states.
//
// Page "RFC(qwen35): TP Phase2", sections "Execution Contract" (decode kernels run against the
// head and state shapes and update only request-local recurrent state) and "Partition
// Contract" (the recurrent state is [Hv, K, V] f32 per request); section "Request-State
// Lifecycle" keeps states in slots that are reused.  Each row b of the batch is one request's
// next token; its state is state[slot[b]].  Per value head j (key head j / (hv / hk)):
//     h <- exp(g) (I - beta k k^T) h + beta k v^T,     o = h^T q
// which is computed from one read of the old state as
//     P = alpha h^T k,  R = alpha h^T q  (alpha = exp(g)),   delta = beta (v - P),
//     h' = alpha h + k delta^T,   o = R + (k . q) delta.
//
// The step is bound by HBM: it reads and writes the K x V fp32 state (128 KiB per row and
// value head at K = V = 128) and little else.  One CTA of 256 threads per (row, value head)
// holds the state in registers: thread (row group rg, column group cg) owns rows
// [rg * RPT, rg * RPT + RPT) and columns [4 cg, 4 cg + 4), so that each warp reads whole
// 512-byte (or two 256-byte) state rows with 16-byte accesses.  The two mat-vecs are reduced
// across row groups in shared memory; then every thread writes its rows of h'.
//
// Slots are checked on the device: a negative slot marks a padding row (its output row is
// zeroed; no state is touched); a slot outside the pool, or one that another row also names,
// skips the row (state and output untouched) and records GDN_ERR_DEVICE_INPUT.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kDecThreads = 256;

template <typename IO>
__device__ __forceinline__ void load_vec(const IO* src, float* dst, int n) {
#pragma unroll
  for (int i = 0; i < n; ++i) dst[i] = to_f32(src[i]);
}

template <int K, int V, typename IO>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(DecodeArgs a) {
  constexpr int CG = V / 4;                // column groups of 4
  constexpr int RG = kDecThreads / CG;     // row groups
  constexpr int RPT = K / RG;              // state rows per thread
  static_assert(CG * RG == kDecThreads && RPT * RG == K && RPT >= 1, "thread layout");
  __shared__ float red_p[RG][V], red_r[RG][V];
  __shared__ float red_kq[RG];
  __shared__ float delta_s[V];

  const int b = blockIdx.x, j = blockIdx.y;
  const int tid = threadIdx.x, cg = tid % CG, rg = tid / CG;
  const int kh = j / (a.hv / a.hk);
  const int s = a.slot[b];
  IO* out = static_cast<IO*>(a.out) + ((int64_t)b * a.hv + j) * V;
  if (s < 0) {  // padding row
    for (int c = tid; c < V; c += kDecThreads) out[c] = from_f32<IO>(0.f);
    return;
  }
  if (s >= a.slots) {
    if (tid == 0) set_status(a.status, GDN_ERR_DEVICE_INPUT);
    return;
  }
  float* st = a.state + ((int64_t)s * a.hv + j) * K * V;
  float4 h[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    h[i] = *reinterpret_cast<const float4*>(st + (int64_t)(rg * RPT + i) * V + 4 * cg);
  // another row naming the same slot: the two updates would race, so neither is made
  bool dup = false;
  for (int e = tid; e < a.batch; e += kDecThreads) dup |= (e != b && a.slot[e] == s);
  if (__syncthreads_or(dup)) {
    if (tid == 0) set_status(a.status, GDN_ERR_DEVICE_INPUT);
    return;
  }
  const IO* qp = static_cast<const IO*>(a.q) + ((int64_t)b * a.hk + kh) * K + rg * RPT;
  const IO* kp = static_cast<const IO*>(a.k) + ((int64_t)b * a.hk + kh) * K + rg * RPT;
  float qv[RPT], kv[RPT];
  load_vec(qp, qv, RPT);
  load_vec(kp, kv, RPT);
  const float g = a.g[(int64_t)b * a.hv + j], beta = a.beta[(int64_t)b * a.hv + j];
  const float alpha = __expf(g);

  // partial h^T k and h^T q over this thread's rows, and k . q over the row group's rows
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
  float kq = 0.f;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    pk.x = fmaf(h[i].x, kv[i], pk.x);
    pk.y = fmaf(h[i].y, kv[i], pk.y);
    pk.z = fmaf(h[i].z, kv[i], pk.z);
    pk.w = fmaf(h[i].w, kv[i], pk.w);
    pq.x = fmaf(h[i].x, qv[i], pq.x);
    pq.y = fmaf(h[i].y, qv[i], pq.y);
    pq.z = fmaf(h[i].z, qv[i], pq.z);
    pq.w = fmaf(h[i].w, qv[i], pq.w);
    kq = fmaf(kv[i], qv[i], kq);
  }
  *reinterpret_cast<float4*>(&red_p[rg][4 * cg]) = pk;
  *reinterpret_cast<float4*>(&red_r[rg][4 * cg]) = pq;
  if (cg == 0) red_kq[rg] = kq;
  __syncthreads();
  for (int c = tid; c < V; c += kDecThreads) {
    float P = 0.f, R = 0.f, KQ = 0.f;
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      P += red_p[r][c];
      R += red_r[r][c];
      KQ += red_kq[r];
    }
    const float vv = to_f32(static_cast<const IO*>(a.v)[((int64_t)b * a.hv + j) * V + c]);
    const float d = beta * (vv - alpha * P);
    delta_s[c] = d;
    out[c] = from_f32<IO>(fmaf(KQ, d, alpha * R));
  }
  __syncthreads();
  const float4 d4 = *reinterpret_cast<const float4*>(&delta_s[4 * cg]);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    float4 x;
    x.x = fmaf(kv[i], d4.x, alpha * h[i].x);
    x.y = fmaf(kv[i], d4.y, alpha * h[i].y);
    x.z = fmaf(kv[i], d4.z, alpha * h[i].z);
    x.w = fmaf(kv[i], d4.w, alpha * h[i].w);
    *reinterpret_cast<float4*>(st + (int64_t)(rg * RPT + i) * V + 4 * cg) = x;
  }
}

template <int K, int V>
cudaError_t launch_kv(const DecodeArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)a.batch, (unsigned)a.hv);
  if (a.bf16)
    decode_kernel<K, V, __nv_bfloat16><<<grid, kDecThreads, 0, s>>>(a);
  else
    decode_kernel<K, V, float><<<grid, kDecThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode_step(const DecodeArgs& a, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  if (a.K == 128 && a.V == 128) return launch_kv<128, 128>(a, s);
  if (a.K == 128 && a.V == 64) return launch_kv<128, 64>(a, s);
  if (a.K == 64 && a.V == 128) return launch_kv<64, 128>(a, s);
  return launch_kv<64, 64>(a, s);
}

}  // namespace gdn
