// gdn_internal.h -- launcher interface between the C ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Everything a kernel needs to know about one call.  Pointers are device pointers; the
// ones a given stage does not use are null.
struct Args {
  int64_t T;
  int N, hk, hv, K, V, P;
  bool bf16;
  const void *q, *k, *v;
  const float *g, *beta;
  const void *w, *u;
  const float* gcum;
  const float *h0, *h_in;
  const float *M, *U;
  const int32_t* cu;
  void* out;
  void *w_out, *u_out;
  void* wy;  // tcgen05 summaries: per-chunk factor records written by the U half (nullable)
  float* gcum_out;
  float *M_out, *U_out, *h_in_out, *h_final;
  int32_t* status;
  bool skip_last_summary;  // the fused forward never reads the last segment's summary
  // Limit of a bounded device wait in SM cycles (0: the default, about a second), and a fault
  // to inject for tests of those waits (0: none; 1: the chunk kernels' chain never signals its
  // first hand-off, so a wait for it expires).
  long long wait_cycles;
  int fault;
};

// Device-side check of cu_seqlens (cu[0] = 0, non-decreasing, cu[N] = T); records
// GDN_ERR_DEVICE_INPUT in the status word on failure.
cudaError_t launch_validate_cu(const Args& a, cudaStream_t s);

// SIMT kernels (fp32 arithmetic; any supported dtype/K/V).
cudaError_t simt_prepare(const Args& a, cudaStream_t s);
cudaError_t simt_summary(const Args& a, cudaStream_t s);
cudaError_t simt_scan(const Args& a, cudaStream_t s);
cudaError_t simt_emit(const Args& a, cudaStream_t s);

// Tensor-core kernels, tcgen05 generation (TMEM accumulators, fp16 operands, fp32 state;
// bf16 I/O, K = V = 128).  Factors are always recomputed on chip.
size_t tc5_smem_bytes();
// Workspace bytes gdn_forward needs without the optional factor records.
size_t workspace_min_bytes(const gdn_problem* p);
// Bytes of the per-chunk factor records the U summary stores for the M summary.
size_t tc5_records_bytes(int64_t T, int N, int hv);
// `mid`, when given, is recorded between the two launches of phase 1.
cudaError_t tc5_summary(const Args& a, cudaStream_t s, cudaEvent_t mid = nullptr);
cudaError_t tc5_emit(const Args& a, cudaStream_t s);

// One decode step over a pool of per-slot states (gdn_decode_step).
struct DecodeArgs {
  int batch, slots, hk, hv, K, V;
  bool bf16;
  const void *q, *k, *v;
  const float *g, *beta;
  const int32_t* slot;
  float* state;
  void* out;
  int32_t* status;
};
cudaError_t decode_step(const DecodeArgs& a, cudaStream_t s);

// Gradients of the forward (gdn_backward).  Workspace pieces: states / dstates
// [nslots, hv, V, K] fp32 (the state entering / the gradient of the state leaving every chunk,
// a state column contiguous), dqv / dkv [T, hv, K] fp32 (per value head, before the sum over
// the key head's group), scratch (grad_ctas slices of the per-chunk kernel's intermediates).
struct BwdArgs {
  int64_t T, nslots;
  int N, hk, hv, K, V;
  bool bf16;
  const void *q, *k, *v, *dout;
  const float *g, *beta, *h0, *dh_final;
  const int32_t* cu;
  void *dq, *dk, *dv;
  float *dg, *dbeta, *dh0;
  float *states, *dstates, *dqv, *dkv, *scratch;
  int grad_ctas;
  int32_t* status;
};
int64_t bwd_slots(int64_t T, int N);
size_t bwd_scratch_floats(int K, int V, int ctas);
cudaError_t backward(const BwdArgs& a, cudaStream_t s);

// The layer prologue (gdn_prologue).
struct PrologueArgs {
  int64_t T;
  int N, hk, hv, K, V, W;
  bool bf16, silu;
  const void *x, *state_in, *a, *b;
  const float *conv_w, *A_log, *dt_bias;
  const int32_t* cu;
  void *q, *k, *v, *state_out;
  float *g, *beta;
  int32_t* status;
};
cudaError_t prologue(const PrologueArgs& a, cudaStream_t s);

}  // namespace gdn
