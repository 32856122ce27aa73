// gdn_api.cu -- the C ABI of libgdn: host-side validation, workspace carving and the
// order of kernel launches for each entry point declared in include/gdn.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

using gdn::Args;

constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernel family a problem runs on (the problem decides; there is no caller-side choice):
// the tcgen05 tensor-core kernels cover bf16 I/O with K = V = 128.
bool use_tensor_path(const gdn_problem* p) {
  return p->io_dtype == GDN_BF16 && p->k_dim == 128 && p->v_dim == 128;
}

// Phase 1 and phase 3 with the factors recomputed on chip (tensor-core kernels).
cudaError_t fused_summary(const gdn_problem*, const Args& a, cudaStream_t s,
                          cudaEvent_t mid = nullptr) {
  return gdn::tc5_summary(a, s, mid);
}
cudaError_t fused_emit(const gdn_problem*, const Args& a, cudaStream_t s) {
  return gdn::tc5_emit(a, s);
}

gdn_status check_problem(const gdn_problem* p) {
  if (!p) return GDN_ERR_INVALID_ARGUMENT;
  if (p->total_tokens < 0 || p->total_tokens > (int64_t)INT32_MAX || p->num_seqs < 1 ||
      p->hk < 1 || p->hv < 1 || p->k_dim < 1 || p->v_dim < 1 || p->chunk < 1 ||
      p->segments_per_seq < 1)
    return GDN_ERR_INVALID_ARGUMENT;
  if (p->hv % p->hk != 0) return GDN_ERR_INVALID_ARGUMENT;
  if (p->io_dtype != GDN_BF16 && p->io_dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
  if (p->chunk != 64) return GDN_ERR_UNSUPPORTED;
  if ((p->k_dim != 64 && p->k_dim != 128) || (p->v_dim != 64 && p->v_dim != 128))
    return GDN_ERR_UNSUPPORTED;
  if (p->hv > 65535) return GDN_ERR_UNSUPPORTED;  // grid.y
  // grid.x of the per-segment kernels and element offsets in 64 bits
  if ((int64_t)p->num_seqs * p->segments_per_seq > (int64_t)INT32_MAX)
    return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

Args base_args(const gdn_problem* p) {
  Args a;
  memset(&a, 0, sizeof(a));
  a.T = p->total_tokens;
  a.N = p->num_seqs;
  a.hk = p->hk;
  a.hv = p->hv;
  a.K = p->k_dim;
  a.V = p->v_dim;
  a.P = p->segments_per_seq;
  a.bf16 = p->io_dtype == GDN_BF16;
  return a;
}

// cu_seqlens may be null only for a single sequence.
bool cu_ok(const gdn_problem* p, const int32_t* cu) { return cu != nullptr || p->num_seqs == 1; }

// The last CUDA error an entry point met on this host thread (reported by
// gdn_last_error_string).
thread_local cudaError_t t_last_error = cudaSuccess;

gdn_status to_status(cudaError_t e) {
  if (e == cudaSuccess) return GDN_OK;
  t_last_error = e;
  return GDN_ERR_CUDA;
}

#define GDN_TRY(expr)                              \
  do {                                             \
    cudaError_t _e = (expr);                       \
    if (_e != cudaSuccess) return to_status(_e);   \
  } while (0)

struct Layout {
  size_t status, M, U, h_in, w, u, gcum, wy, total;
};

// Workspace: [status word | M | U | h_in | w | u | gcum | records], each piece 256-byte
// aligned.  The summaries and incoming states exist only for P > 1; the materialised chunk
// factors only on the SIMT path (the tensor-core kernels recompute them on chip); the records
// (-w^T, fp16 K, u^T and the decay of each chunk, 49,664 bytes per chunk and value head) only
// on the tcgen05 path with P > 1, where the U summary writes them and the M summary and the
// emit kernel read them.
Layout layout(const gdn_problem* p, bool records = true) {
  Layout L;
  const size_t S = (size_t)p->num_seqs * p->segments_per_seq * p->hv;
  const size_t K = p->k_dim, V = p->v_dim, T = (size_t)p->total_tokens;
  const bool seg = p->segments_per_seq > 1;
  const bool mat = !use_tensor_path(p);
  size_t off = 0;
  L.status = off;
  off += kStatusBytes;
  L.M = off;
  off += seg ? align_up(S * K * K * 4) : 0;
  L.U = off;
  off += seg ? align_up(S * K * V * 4) : 0;
  L.h_in = off;
  off += seg ? align_up(S * K * V * 4) : 0;
  L.w = off;
  off += mat ? align_up(T * p->hv * K * 4) : 0;
  L.u = off;
  off += mat ? align_up(T * p->hv * V * 4) : 0;
  L.gcum = off;
  off += mat ? align_up(T * p->hv * 4) : 0;
  L.wy = off;  // tcgen05 path: the U summary's per-chunk records for the M summary
  off += (records && seg && !mat)
             ? align_up(gdn::tc5_records_bytes(p->total_tokens, p->num_seqs, p->hv))
             : 0;
  L.total = off;
  return L;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARGUMENT: return "GDN_ERR_INVALID_ARGUMENT: bad pointer, size or alignment";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: dtype/K/V/chunk outside the built set";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA launch or runtime call failed";
    case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT: a bounded device wait expired";
    case GDN_ERR_DEVICE_INPUT: return "GDN_ERR_DEVICE_INPUT: cu_seqlens inconsistent on the device";
    case GDN_ERR_DEVICE_RANGE: return "GDN_ERR_DEVICE_RANGE: a tensor-core operand exceeded the fp16 range";
  }
  return "GDN_UNKNOWN_STATUS";
}

int gdn_version(void) { return 100; }

const char* gdn_last_error_string(void) {
  return t_last_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(t_last_error);
}

gdn_status gdn_check_problem(const gdn_problem* p) { return check_problem(p); }

size_t gdn_workspace_size(const gdn_problem* p) {
  if (check_problem(p) != GDN_OK) return 0;
  return layout(p).total;
}

}  // extern "C"

size_t gdn::workspace_min_bytes(const gdn_problem* p) {
  return check_problem(p) != GDN_OK ? 0 : layout(p, false).total;
}

extern "C" {

gdn_status gdn_chunk_prepare(const gdn_problem* p, const void* k, const void* v, const float* g,
                             const float* beta, const int32_t* cu_seqlens, void* w, void* u,
                             float* gcum, int32_t* dev_status, cudaStream_t stream) {
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (p->total_tokens > 0 && (!k || !v || !g || !beta || !w || !u || !gcum))
    return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_ok(p, cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(k) || !aligned16(v) || !aligned16(w) || !aligned16(u))
    return GDN_ERR_INVALID_ARGUMENT;
  Args a = base_args(p);
  a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu = cu_seqlens;
  a.w_out = w; a.u_out = u; a.gcum_out = gcum; a.status = dev_status;
  if (a.T == 0) return GDN_OK;
  GDN_TRY(gdn::launch_validate_cu(a, stream));
  return to_status(gdn::simt_prepare(a, stream));
}

gdn_status gdn_segment_summary(const gdn_problem* p, const void* k, const void* w, const void* u,
                               const float* gcum, const int32_t* cu_seqlens, float* M, float* U,
                               int32_t* dev_status, cudaStream_t stream) {
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (!M || !U) return GDN_ERR_INVALID_ARGUMENT;
  if (p->total_tokens > 0 && (!k || !w || !u || !gcum)) return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_ok(p, cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(k) || !aligned16(w) || !aligned16(u) || !aligned16(M) || !aligned16(U))
    return GDN_ERR_INVALID_ARGUMENT;
  Args a = base_args(p);
  a.k = k; a.w = w; a.u = u; a.gcum = gcum; a.cu = cu_seqlens;
  a.M_out = M; a.U_out = U; a.status = dev_status;
  GDN_TRY(gdn::launch_validate_cu(a, stream));
  return to_status(gdn::simt_summary(a, stream));
}

gdn_status gdn_state_prefix_scan(const gdn_problem* p, const float* M, const float* U,
                                 const float* h0, float* h_in, float* h_final,
                                 cudaStream_t stream) {
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (!M || !U || !h_in) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(M) || !aligned16(U) || !aligned16(h_in) || !aligned16(h0) || !aligned16(h_final))
    return GDN_ERR_INVALID_ARGUMENT;
  Args a = base_args(p);
  a.M = M; a.U = U; a.h0 = h0; a.h_in_out = h_in; a.h_final = h_final;
  return to_status(gdn::simt_scan(a, stream));
}

gdn_status gdn_chunk_emit(const gdn_problem* p, const void* q, const void* k, const void* w,
                          const void* u, const float* gcum, const float* h_in,
                          const int32_t* cu_seqlens, void* out, float* h_final,
                          int32_t* dev_status, cudaStream_t stream) {
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (p->total_tokens > 0 && (!q || !k || !w || !u || !gcum || !out))
    return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_ok(p, cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(w) || !aligned16(u) || !aligned16(out) ||
      !aligned16(h_in) || !aligned16(h_final))
    return GDN_ERR_INVALID_ARGUMENT;
  Args a = base_args(p);
  a.q = q; a.k = k; a.w = w; a.u = u; a.gcum = gcum; a.h_in = h_in; a.cu = cu_seqlens;
  a.out = out; a.h_final = h_final; a.status = dev_status;
  GDN_TRY(gdn::launch_validate_cu(a, stream));
  return to_status(gdn::simt_emit(a, stream));
}

}  // extern "C"

namespace {
// gdn_forward, recording ev[0..4] (when given) before phase 1, after phase 1, after the scan,
// after phase 3, and between the two kernels of phase 1 (after phase 1's only launch on the
// paths with one).
gdn_status forward_impl(const gdn_problem* p, const void* q, const void* k, const void* v,
                        const float* g, const float* beta, const float* h0,
                        const int32_t* cu_seqlens, void* out, float* h_final, void* workspace,
                        size_t ws_bytes, cudaStream_t stream, cudaEvent_t* ev,
                        long long wait_cycles = 0, int fault = 0) {
  auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], stream) : cudaSuccess; };
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (p->total_tokens > 0 && (!q || !k || !v || !g || !beta || !out))
    return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_ok(p, cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(h0) ||
      !aligned16(h_final))
    return GDN_ERR_INVALID_ARGUMENT;
  // The records are optional: without room for them both summaries compute their factors.
  const Layout Lr = layout(p, true), L = ws_bytes >= Lr.total ? Lr : layout(p, false);
  if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return GDN_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
  GDN_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), stream));

  Args a = base_args(p);
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.cu = cu_seqlens;
  a.out = out; a.h_final = h_final; a.status = status;
  a.wait_cycles = wait_cycles;
  a.fault = fault;
  const bool seg = p->segments_per_seq > 1;
  if (seg) {
    a.M_out = reinterpret_cast<float*>(ws + L.M);
    a.U_out = reinterpret_cast<float*>(ws + L.U);
    a.M = a.M_out;
    a.U = a.U_out;
    a.h_in_out = reinterpret_cast<float*>(ws + L.h_in);
    if (use_tensor_path(p) && L.total == Lr.total && Lr.total > Lr.wy)
      a.wy = ws + L.wy;
  }
  // With P = 1 the incoming state of the only segment is h0 itself.
  a.h_in = seg ? a.h_in_out : h0;
  GDN_TRY(gdn::launch_validate_cu(a, stream));

  GDN_TRY(mark(0));
  if (use_tensor_path(p)) {
    if (seg) {
      Args ma = a;
      ma.skip_last_summary = true;
      GDN_TRY(fused_summary(p, ma, stream, ev ? ev[4] : nullptr));
      GDN_TRY(mark(1));
      Args sa = a;
      sa.h_final = nullptr;  // the last segment's emit writes the final state
      GDN_TRY(gdn::simt_scan(sa, stream));
    } else {
      GDN_TRY(mark(1));
      GDN_TRY(mark(4));
    }
    GDN_TRY(mark(2));
    GDN_TRY(fused_emit(p, a, stream));
    return to_status(mark(3));
  }
  a.w_out = ws + L.w;
  a.u_out = ws + L.u;
  a.gcum_out = reinterpret_cast<float*>(ws + L.gcum);
  a.w = a.w_out;
  a.u = a.u_out;
  a.gcum = a.gcum_out;
  if (a.T > 0) GDN_TRY(gdn::simt_prepare(a, stream));
  if (seg) {
    GDN_TRY(gdn::simt_summary(a, stream));  // (the SIMT summary computes every segment)
    GDN_TRY(mark(4));
    GDN_TRY(mark(1));
    Args sa = a;
    sa.h_final = nullptr;
    GDN_TRY(gdn::simt_scan(sa, stream));
  } else {
    GDN_TRY(mark(1));
    GDN_TRY(mark(4));
  }
  GDN_TRY(mark(2));
  GDN_TRY(gdn::simt_emit(a, stream));
  return to_status(mark(3));
}
}  // namespace

extern "C" {

gdn_status gdn_forward(const gdn_problem* p, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* h0,
                       const int32_t* cu_seqlens, void* out, float* h_final, void* workspace,
                       size_t ws_bytes, cudaStream_t stream) {
  return forward_impl(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, workspace, ws_bytes,
                      stream, nullptr);
}

gdn_status gdn_forward_with_limits(const gdn_problem* p, const void* q, const void* k,
                                   const void* v, const float* g, const float* beta,
                                   const float* h0, const int32_t* cu_seqlens, void* out,
                                   float* h_final, void* workspace, size_t ws_bytes,
                                   cudaStream_t stream, long long wait_cycles, int fault) {
  if (wait_cycles < 0 || fault < 0 || fault > 1) return GDN_ERR_INVALID_ARGUMENT;
  return forward_impl(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, workspace, ws_bytes,
                      stream, nullptr, wait_cycles, fault);
}

gdn_status gdn_forward_timed(const gdn_problem* p, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* h0,
                             const int32_t* cu_seqlens, void* out, float* h_final,
                             void* workspace, size_t ws_bytes, cudaStream_t stream,
                             float* phase_ms) {
  if (!phase_ms) return GDN_ERR_INVALID_ARGUMENT;
  cudaEvent_t ev[5] = {};
  for (int i = 0; i < 5; ++i)
    if (cudaEventCreate(&ev[i]) != cudaSuccess) {
      for (int k2 = 0; k2 < i; ++k2) cudaEventDestroy(ev[k2]);
      return to_status(cudaGetLastError());
    }
  gdn_status st = forward_impl(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, workspace,
                               ws_bytes, stream, ev);
  if (st == GDN_OK) {
    cudaError_t e = cudaEventSynchronize(ev[3]);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventElapsedTime(&phase_ms[i], ev[i], ev[i + 1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&phase_ms[3], ev[0], ev[4]);
    if (e != cudaSuccess) st = to_status(e);
  }
  for (int i = 0; i < 5; ++i) cudaEventDestroy(ev[i]);
  return st;
}

gdn_status gdn_segment_summary_fused(const gdn_problem* p, const void* k, const void* v,
                                     const float* g, const float* beta,
                                     const int32_t* cu_seqlens, float* M, float* U,
                                     int skip_last, int32_t* dev_status, cudaStream_t stream) {
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (!use_tensor_path(p)) return GDN_ERR_UNSUPPORTED;
  if (!M || !U) return GDN_ERR_INVALID_ARGUMENT;
  if (p->total_tokens > 0 && (!k || !v || !g || !beta)) return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_ok(p, cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(k) || !aligned16(v) || !aligned16(M) || !aligned16(U))
    return GDN_ERR_INVALID_ARGUMENT;
  Args a = base_args(p);
  a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu = cu_seqlens;
  a.M_out = M; a.U_out = U; a.status = dev_status; a.skip_last_summary = skip_last != 0;
  GDN_TRY(gdn::launch_validate_cu(a, stream));
  return to_status(fused_summary(p, a, stream));
}

gdn_status gdn_chunk_emit_fused(const gdn_problem* p, const void* q, const void* k,
                                const void* v, const float* g, const float* beta,
                                const float* h_in, const int32_t* cu_seqlens, void* out,
                                float* h_final, int32_t* dev_status, cudaStream_t stream) {
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (!use_tensor_path(p)) return GDN_ERR_UNSUPPORTED;
  if (p->total_tokens > 0 && (!q || !k || !v || !g || !beta || !out))
    return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_ok(p, cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(h_in) ||
      !aligned16(h_final))
    return GDN_ERR_INVALID_ARGUMENT;
  Args a = base_args(p);
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h_in = h_in; a.cu = cu_seqlens;
  a.out = out; a.h_final = h_final; a.status = dev_status;
  GDN_TRY(gdn::launch_validate_cu(a, stream));
  return to_status(fused_emit(p, a, stream));
}

// ------------------------------------------------------------------ backward

// CTAs of the per-chunk gradient kernel (two per SM of a 152-SM GB300); the workspace holds one
// slice of intermediates for each.  The kernel walks all units with a grid stride, so any SM
// count computes the same result.
constexpr int kGradCtas = 304;

struct BwdLayout {
  size_t status, states, dstates, dqv, dkv, scratch, total;
};
BwdLayout bwd_layout(const gdn_problem* p) {
  BwdLayout L;
  const size_t K = p->k_dim, V = p->v_dim, T = (size_t)p->total_tokens;
  const size_t slots = (size_t)gdn::bwd_slots(p->total_tokens, p->num_seqs);
  size_t off = 0;
  L.status = off;
  off += kStatusBytes;
  L.states = off;
  off += align_up(slots * p->hv * K * V * 4);
  L.dstates = off;
  off += align_up(slots * p->hv * K * V * 4);
  L.dqv = off;
  off += align_up(T * p->hv * K * 4);
  L.dkv = off;
  off += align_up(T * p->hv * K * 4);
  L.scratch = off;
  off += align_up(gdn::bwd_scratch_floats(p->k_dim, p->v_dim, kGradCtas) * 4);
  L.total = off;
  return L;
}

gdn_status gdn_prologue(const gdn_prologue_problem* p, const void* x, const float* conv_w,
                        const void* conv_state_in, const void* a, const void* b,
                        const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                        void* q, void* k, void* v, float* g, float* beta, void* conv_state_out,
                        int32_t* dev_status, cudaStream_t stream) {
  if (!p) return GDN_ERR_INVALID_ARGUMENT;
  if (p->total_tokens < 0 || p->total_tokens > (int64_t)INT32_MAX || p->num_seqs < 1 ||
      p->hk < 1 || p->hv < 1 || p->k_dim < 1 || p->v_dim < 1 || p->hv % p->hk != 0)
    return GDN_ERR_INVALID_ARGUMENT;
  if (p->io_dtype != GDN_BF16 && p->io_dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
  if (p->k_dim > 128 || p->v_dim > 128 || p->k_dim % 8 || p->v_dim % 8 || p->conv_width < 1 ||
      p->conv_width > 4 ||
      (p->activation != 0 && p->activation != 1) || 2 * p->hk + p->hv > 65535)
    return GDN_ERR_UNSUPPORTED;
  if (!conv_w || !A_log || !dt_bias || (p->total_tokens > 0 &&
      (!x || !a || !b || !q || !k || !v || !g || !beta)))
    return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_seqlens && p->num_seqs != 1) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return GDN_ERR_INVALID_ARGUMENT;
  gdn::PrologueArgs pa;
  memset(&pa, 0, sizeof(pa));
  pa.T = p->total_tokens;
  pa.N = p->num_seqs;
  pa.hk = p->hk;
  pa.hv = p->hv;
  pa.K = p->k_dim;
  pa.V = p->v_dim;
  pa.W = p->conv_width;
  pa.bf16 = p->io_dtype == GDN_BF16;
  pa.silu = p->activation == 1;
  pa.x = x; pa.state_in = conv_state_in; pa.a = a; pa.b = b;
  pa.conv_w = conv_w; pa.A_log = A_log; pa.dt_bias = dt_bias; pa.cu = cu_seqlens;
  pa.q = q; pa.k = k; pa.v = v; pa.state_out = conv_state_out; pa.g = g; pa.beta = beta;
  pa.status = dev_status;
  if (cu_seqlens) {
    Args va;
    memset(&va, 0, sizeof(va));
    va.T = p->total_tokens;
    va.N = p->num_seqs;
    va.cu = cu_seqlens;
    va.status = dev_status;
    GDN_TRY(gdn::launch_validate_cu(va, stream));
  }
  return to_status(gdn::prologue(pa, stream));
}

gdn_status gdn_check_decode_problem(const gdn_decode_problem* p) {
  if (!p) return GDN_ERR_INVALID_ARGUMENT;
  if (p->batch < 0 || p->slots < 1 || p->hk < 1 || p->hv < 1 || p->k_dim < 1 || p->v_dim < 1)
    return GDN_ERR_INVALID_ARGUMENT;
  if (p->hv % p->hk != 0) return GDN_ERR_INVALID_ARGUMENT;
  if (p->io_dtype != GDN_BF16 && p->io_dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
  if ((p->k_dim != 64 && p->k_dim != 128) || (p->v_dim != 64 && p->v_dim != 128))
    return GDN_ERR_UNSUPPORTED;
  if (p->hv > 65535) return GDN_ERR_UNSUPPORTED;  // grid.y
  return GDN_OK;
}

gdn_status gdn_decode_step(const gdn_decode_problem* p, const void* q, const void* k,
                           const void* v, const float* g, const float* beta,
                           const int32_t* slot, float* state, void* out, int32_t* dev_status,
                           cudaStream_t stream) {
  gdn_status st = gdn_check_decode_problem(p);
  if (st != GDN_OK) return st;
  if (p->batch == 0) return GDN_OK;
  if (!q || !k || !v || !g || !beta || !slot || !state || !out) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
      !aligned16(slot) || !aligned16(state) || !aligned16(out))
    return GDN_ERR_INVALID_ARGUMENT;
  gdn::DecodeArgs a;
  memset(&a, 0, sizeof(a));
  a.batch = p->batch;
  a.slots = p->slots;
  a.hk = p->hk;
  a.hv = p->hv;
  a.K = p->k_dim;
  a.V = p->v_dim;
  a.bf16 = p->io_dtype == GDN_BF16;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.slot = slot;
  a.state = state;
  a.out = out;
  a.status = dev_status;
  return to_status(gdn::decode_step(a, stream));
}

size_t gdn_backward_workspace_size(const gdn_problem* p) {
  return check_problem(p) != GDN_OK ? 0 : bwd_layout(p).total;
}

gdn_status gdn_backward(const gdn_problem* p, const void* q, const void* k, const void* v,
                        const float* g, const float* beta, const float* h0,
                        const int32_t* cu_seqlens, const void* dout, const float* dh_final,
                        void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0,
                        void* workspace, size_t ws_bytes, cudaStream_t stream) {
  gdn_status st = check_problem(p);
  if (st != GDN_OK) return st;
  if (p->total_tokens > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv ||
                              !dg || !dbeta))
    return GDN_ERR_INVALID_ARGUMENT;
  if (!cu_ok(p, cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(h0) || !aligned16(dh_final) ||
      !aligned16(dh0))
    return GDN_ERR_INVALID_ARGUMENT;
  const BwdLayout L = bwd_layout(p);
  if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return GDN_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
  GDN_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), stream));
  Args va = base_args(p);
  va.cu = cu_seqlens;
  va.status = status;
  GDN_TRY(gdn::launch_validate_cu(va, stream));
  gdn::BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.T = p->total_tokens;
  a.nslots = gdn::bwd_slots(p->total_tokens, p->num_seqs);
  a.N = p->num_seqs;
  a.hk = p->hk;
  a.hv = p->hv;
  a.K = p->k_dim;
  a.V = p->v_dim;
  a.bf16 = p->io_dtype == GDN_BF16;
  a.q = q; a.k = k; a.v = v; a.dout = dout;
  a.g = g; a.beta = beta; a.h0 = h0; a.dh_final = dh_final; a.cu = cu_seqlens;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
  a.states = reinterpret_cast<float*>(ws + L.states);
  a.dstates = reinterpret_cast<float*>(ws + L.dstates);
  a.dqv = reinterpret_cast<float*>(ws + L.dqv);
  a.dkv = reinterpret_cast<float*>(ws + L.dkv);
  a.scratch = reinterpret_cast<float*>(ws + L.scratch);
  a.grad_ctas = kGradCtas;
  a.status = status;
  if (a.T == 0) {  // no tokens: the state passes through, dh0 = dh_final
    if (dh0) {
      const size_t bytes = (size_t)p->num_seqs * p->hv * p->k_dim * p->v_dim * 4;
      if (dh_final)
        GDN_TRY(cudaMemcpyAsync(dh0, dh_final, bytes, cudaMemcpyDeviceToDevice, stream));
      else
        GDN_TRY(cudaMemsetAsync(dh0, 0, bytes, stream));
    }
    return GDN_OK;
  }
  return to_status(gdn::backward(a, stream));
}

gdn_status gdn_device_status(const void* status_word, int reset, cudaStream_t stream) {
  if (!status_word) return GDN_ERR_INVALID_ARGUMENT;
  int32_t host = 0;
  int32_t* dev = const_cast<int32_t*>(static_cast<const int32_t*>(status_word));
  GDN_TRY(cudaMemcpyAsync(&host, dev, sizeof(int32_t), cudaMemcpyDeviceToHost, stream));
  if (reset) GDN_TRY(cudaMemsetAsync(dev, 0, sizeof(int32_t), stream));
  GDN_TRY(cudaStreamSynchronize(stream));
  return static_cast<gdn_status>(host);
}

}  // extern "C"
