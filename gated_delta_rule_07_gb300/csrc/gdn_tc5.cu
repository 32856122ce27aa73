// gdn_tc5.cu -- tcgen05 (5th-generation tensor core) kernels for the chunked gated delta
// rule forward, bf16 I/O, K = V = 128, C = 64, fp32 state.
//
// One CTA per (segment, value head) walks the segment's chunks ("Add context parallelism to
// the Gated Delta Net", section "Implementation": phase 3 re-emit, or phase 1 summary on one
// half of X = [M | U]).  Every contraction is a tcgen05.mma with fp32 accumulation in Tensor
// Memory; products are taken in transposed form so that M = 128 (a state or feature index)
// fills the 128 TMEM lanes:
//   [S ; QK]  = [K ; Q] K^T                       (128 x 64, K = 128)
//   w^T       = K^T (T diag(beta e^G))^T          (128 x 64, K = 64)
//   u^T       = V^T (T diag(beta))^T              (128 x 64, K = 64)
//   delta^T   = u^T + h^T (-w)^T                  (128 x 64, K = 128; h^T read from TMEM)
//   O1^T      = h^T Q^T                           (128 x 64, K = 128)
//   O2^T      = delta^T attn_i^T                  (128 x 64, K = 64; delta^T from TMEM)
//   Dh^T      = (diag(e^{G_last - G}) delta)^T K  (128 x 128, K = 64)
// and o = e^{G_t} O1 + O2, h <- gamma h + Dh.  The state h^T lives in registers (fp32) of
// the chain warps; its fp16 copy, delta and delta' are written back into TMEM as the A
// operands of the next products.  T = (I + A)^-1 is a blocked fp32 forward substitution.
//
// Warp roles (416 threads):
//   warps 0-7  chain:   TMEM lane = state row c; warps w and w + 4 split the columns
//   warps 8-11 prepare: chunk loads (cp.async, bf16 -> fp16), decay tables, masked gram and
//                       attn_i, the triangular solve, -w
//   warp 12    MMA:     one thread issues every tcgen05.mma and commit in program order
// Hand-offs use mbarriers; every wait is bounded and a wait that gives up records
// GDN_ERR_DEVICE_TIMEOUT, and all roles leave their loops (group decisions are made uniform
// with barrier reductions) so the CTA always reaches its TMEM release.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int C = kChunk;  // 64
constexpr int KD = 128, VD = 128;
constexpr int kChainThreads = 256, kPrepThreads = 128;
constexpr int kThreads = kChainThreads + kPrepThreads + 32;
constexpr int FP = C + 1;
constexpr uint32_t kWaitLimit = 1u << 21;
constexpr float kHalfMax = 65504.f;

enum Mode { kEmit = 0, kSumM = 1, kSumU = 2 };

// TMEM columns (512 allocated)
constexpr uint32_t TM_SQ = 0;    // [S ; QK]          64 fp32
constexpr uint32_t TM_W = 64;    // w^T               64 fp32
constexpr uint32_t TM_U = 128;   // u^T -> delta^T    64 fp32, then fp16 delta / delta'
constexpr uint32_t TM_O1 = 192;  // O1^T              64 fp32
constexpr uint32_t TM_O2 = 256;  // O2^T              64 fp32
constexpr uint32_t TM_H = 384;   // Dh^T              128 fp32, then fp16 h^T

// mbarriers
enum Bar { B_X0 = 0, B_X1, B_SQ, B_T, B_WU, B_WR, B_HR, B_D, B_DR, B_H, kNumBars };

struct Smem {
  uint8_t kq[2][2 * 128 * 128];  // per stage: [kblk][128 rows: K 0-63, Q 64-127][128 B]
  uint8_t v[2][2 * 64 * 128];    // per stage: [kblk][64 rows][128 B]
  uint8_t att[2][64 * 128];      // attn_i [t][s], K-major B
  uint8_t tw[64 * 128];          // T diag(beta e^G) [t][s], K-major B
  uint8_t tu[64 * 128];          // T diag(beta) [t][s], K-major B
  uint8_t nw[128 * 128];         // -w [i][t], MN-major B
  float A[C * FP];               // masked gram (fp32)
  float Ti[C * FP];              // (I + A)^-1 (fp32)
  float X[C * FP];               // solve scratch
  float G[3][C], alpha[3][C], eG[3][C], eGLG[3][C], beta[3][C], gamma[3];
  uint64_t bars[kNumBars];
  uint32_t tmem_base;
  int abort_flag;
  int range_bad;
};

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
// Barrier over `n` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// Group-uniform bounded wait: every thread polls, then the group agrees.
__device__ __forceinline__ bool aborted(Smem& S) {
  return *reinterpret_cast<volatile int*>(&S.abort_flag) != 0;
}
__device__ __forceinline__ void set_abort(Smem& S) {
  *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
}
__device__ __forceinline__ bool group_wait(Smem& S, int bar, uint32_t parity, int id, int n) {
  bool ok = !aborted(S) && mbar_wait(saddr(&S.bars[bar]), parity, kWaitLimit);
  ok = named_bar_and(id, n, ok);
  if (!ok) set_abort(S);
  return ok;
}
__device__ __forceinline__ bool single_wait(Smem& S, int bar, uint32_t parity) {
  if (aborted(S)) return false;
  if (mbar_wait(saddr(&S.bars[bar]), parity, kWaitLimit)) return true;
  set_abort(S);
  return false;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ bool fits_half(float x) { return fabsf(x) <= kHalfMax; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}

// In-place bf16 -> fp16 of one 16-byte chunk; false when a value leaves the fp16 range.
__device__ __forceinline__ bool to_half_chunk(uint8_t* p) {
  uint4 x = *reinterpret_cast<uint4*>(p);
  uint32_t* w = reinterpret_cast<uint32_t*>(&x);
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
    ok = ok && fits_half(f.x) && fits_half(f.y);
    w[i] = pack_h2(f.x, f.y);
  }
  *reinterpret_cast<uint4*>(p) = x;
  return ok;
}

// ------------------------------------------------------------------ the kernel

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) tc5_chunk_kernel(Args a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x, j = blockIdx.y;
  const int n_seq = seg / a.P, r = seg % a.P;
  if (MODE != kEmit && r == a.P - 1 && a.skip_last_summary) return;
  const int kh = j / (a.hv / a.hk);
  int64_t sb, se;
  if (!seq_bounds(a.cu, n_seq, a.T, a.status, sb, se)) return;
  int64_t c0, c1;
  segment_chunks(se - sb, a.P, r, c0, c1);
  const int nch = (int)(c1 - c0);

  // ---- setup: mbarriers, TMEM
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) mbar_init(saddr(&S.bars[b]), 1);
    S.abort_flag = 0;
    S.range_bad = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 12) {
    tmem_alloc(saddr(&S.tmem_base), 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = S.tmem_base;

  if (warp < 8) {
    // =============================================================== chain (256 threads)
    const int hf = warp >> 2;                 // column half of the state row
    const int c = (warp & 3) * 32 + lane;     // state row = TMEM lane
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    bool range_ok = true;
    float h[64];                              // h^T[c][64 hf .. 64 hf + 63]
    {
      const float* src = nullptr;
      if (MODE == kEmit && a.h_in) src = a.h_in + ((int64_t)seg * a.hv + j) * KD * VD;
#pragma unroll
      for (int q = 0; q < 64; ++q) {
        const int i = 64 * hf + q;
        float x = 0.f;
        if (MODE == kEmit) x = src ? src[i * VD + c] : 0.f;
        if (MODE == kSumM) x = (i == c) ? 1.f : 0.f;
        h[q] = x;
      }
    }
    auto publish_h = [&]() {  // fp16 h^T into TMEM (the A operand of delta and O1)
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        uint32_t p[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float x0 = h[16 * piece + 2 * q], x1 = h[16 * piece + 2 * q + 1];
          range_ok = range_ok && fits_half(x0) && fits_half(x1);
          p[q] = pack_h2(x0, x1);
        }
        tmem_st8(tm + lane_bits + TM_H + 64 * hf + 8 * piece, p);
      }
    };
    if (nch > 0) {
      publish_h();
      fence_before_sync();
      named_bar(2, kChainThreads);
      if (tid == 0) mbar_arrive(saddr(&S.bars[B_HR]));
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    for (int ci = 0; ci < nch; ++ci) {
      const int gb = ci % 3;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      // ---- delta: fp32 delta^T -> fp16 delta and delta' (= e^{G_last - G_t} delta)
      if (!group_wait(S, B_D, ci & 1, 2, kChainThreads)) break;
      fence_after_sync();
      {
        // read both 16-column pieces before writing: the packed results overwrite them
        float d0[16], d1[16];
        tmem_ld16(tm + lane_bits + TM_U + 32 * hf, d0);
        tmem_ld16(tm + lane_bits + TM_U + 32 * hf + 16, d1);
        {
          uint32_t pd[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            range_ok = range_ok && fits_half(d0[2 * q]) && fits_half(d0[2 * q + 1]) &&
                       fits_half(d1[2 * q]) && fits_half(d1[2 * q + 1]);
            pd[q] = pack_h2(d0[2 * q], d0[2 * q + 1]);
            pd[q + 8] = pack_h2(d1[2 * q], d1[2 * q + 1]);
          }
          tmem_st16(tm + lane_bits + TM_U + 32 * hf, pd);
        }
        {
          uint32_t pp[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int t = 32 * hf + 2 * q;
            pp[q] = pack_h2(d0[2 * q] * S.eGLG[gb][t], d0[2 * q + 1] * S.eGLG[gb][t + 1]);
            pp[q + 8] =
                pack_h2(d1[2 * q] * S.eGLG[gb][t + 16], d1[2 * q + 1] * S.eGLG[gb][t + 17]);
          }
          tmem_st16(tm + lane_bits + TM_U + 32 * hf + 16, pp);
        }
      }
      fence_before_sync();
      named_bar(2, kChainThreads);
      if (tid == 0) mbar_arrive(saddr(&S.bars[B_DR]));
      // ---- outputs and the state update
      if (!group_wait(S, B_H, ci & 1, 2, kChainThreads)) break;
      fence_after_sync();
      if (MODE == kEmit) {
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          float o1[16], o2[16];
          tmem_ld16(tm + lane_bits + TM_O1 + 32 * hf + 16 * piece, o1);
          tmem_ld16(tm + lane_bits + TM_O2 + 32 * hf + 16 * piece, o2);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int t = 32 * hf + 16 * piece + q;
            if (t < L)
              out[((t0 + t) * a.hv + j) * VD + c] =
                  __float2bfloat16_rn(S.eG[gb][t] * o1[q] + o2[q]);
          }
        }
      }
      {
        const float gam = S.gamma[gb];
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) {
          float dh[16];
          tmem_ld16(tm + lane_bits + TM_H + 64 * hf + 16 * piece, dh);
#pragma unroll
          for (int q = 0; q < 16; ++q) h[16 * piece + q] = gam * h[16 * piece + q] + dh[q];
        }
      }
      if (ci + 1 < nch) {
        publish_h();
        fence_before_sync();
        named_bar(2, kChainThreads);
        if (tid == 0) mbar_arrive(saddr(&S.bars[B_HR]));
      }
    }
    if (!range_ok) S.range_bad = 1;
    // ---- the final state: h^T[c][i] = h[i][c]
    float* dst = nullptr;
    if (MODE == kEmit) {
      if (a.h_final && r == a.P - 1) dst = a.h_final + ((int64_t)n_seq * a.hv + j) * KD * VD;
    } else if (MODE == kSumM) {
      dst = a.M_out + ((int64_t)seg * a.hv + j) * KD * KD;
    } else {
      dst = a.U_out + ((int64_t)seg * a.hv + j) * KD * VD;
    }
    if (dst && !aborted(S)) {
#pragma unroll
      for (int q = 0; q < 64; ++q) dst[(64 * hf + q) * VD + c] = h[q];
    }
  } else if (warp < 12) {
    // =============================================================== prepare (128 threads)
    const int pt = tid - kChainThreads;       // 0..127 = TMEM lane of this thread
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    bool range_ok = true;
    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(a.v);

    auto issue_loads = [&](int ci) {
      const int s = ci & 1;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      const uint32_t kq = saddr(S.kq[s]), vv = saddr(S.v[s]);
      for (int e = pt; e < C * 16; e += kPrepThreads) {
        const int t = e >> 4, col = (e & 15) << 3;
        const bool ok = t < L;
        const int64_t tt = ok ? t0 + t : sb;
        cp_async16(kq + sw128_offset(128, t, col), gk + (tt * a.hk + kh) * KD + col, ok);
        if (MODE == kEmit)
          cp_async16(kq + sw128_offset(128, 64 + t, col), gq + (tt * a.hk + kh) * KD + col, ok);
        if (MODE != kSumM)
          cp_async16(vv + sw128_offset(64, t, col), gv + (tt * a.hv + j) * VD + col, ok);
      }
      asm volatile("cp.async.commit_group;\n" ::: "memory");
    };
    auto finish_data = [&](int ci) {  // convert chunk ci to fp16, decay tables, arrive X
      const int s = ci & 1, gb = ci % 3;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
      for (int e = pt; e < C * 16; e += kPrepThreads) {
        const int t = e >> 4, col = (e & 15) << 3;
        range_ok &= to_half_chunk(S.kq[s] + sw128_offset(128, t, col));
        if (MODE == kEmit) range_ok &= to_half_chunk(S.kq[s] + sw128_offset(128, 64 + t, col));
        if (MODE != kSumM) range_ok &= to_half_chunk(S.v[s] + sw128_offset(64, t, col));
      }
      if (pt < 32) {  // within-chunk inclusive scan of g; rows >= L decay by nothing
        float g0 = pt < L ? a.g[(t0 + pt) * a.hv + j] : 0.f;
        float g1 = pt + 32 < L ? a.g[(t0 + pt + 32) * a.hv + j] : 0.f;
        float x0 = g0, x1 = g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
          const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
          if (pt >= o) { x0 += y0; x1 += y1; }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        const float GL = L - 1 < 32 ? __shfl_sync(0xffffffffu, x0, (L - 1) & 31)
                                    : __shfl_sync(0xffffffffu, x1, (L - 1) & 31);
        S.G[gb][pt] = x0;
        S.G[gb][pt + 32] = x1;
        S.alpha[gb][pt] = __expf(g0);
        S.alpha[gb][pt + 32] = __expf(g1);
        S.eG[gb][pt] = __expf(x0);
        S.eG[gb][pt + 32] = __expf(x1);
        S.eGLG[gb][pt] = __expf(GL - x0);
        S.eGLG[gb][pt + 32] = __expf(GL - x1);
        S.beta[gb][pt] = pt < L ? a.beta[(t0 + pt) * a.hv + j] : 0.f;
        S.beta[gb][pt + 32] = pt + 32 < L ? a.beta[(t0 + pt + 32) * a.hv + j] : 0.f;
        if (pt == 0) S.gamma[gb] = __expf(GL);
      }
      fence_async_smem();
      named_bar(1, kPrepThreads);
      if (pt == 0) mbar_arrive(saddr(&S.bars[B_X0 + s]));
    };

    if (nch > 0) {
      issue_loads(0);
      finish_data(0);
    }
    for (int ci = 0; ci < nch; ++ci) {
      const int gb = ci % 3;
      // ---- masked gram A (fp32) and attn_i (fp16) from [S ; QK]
      if (!group_wait(S, B_SQ, ci & 1, 1, kPrepThreads)) break;
      fence_after_sync();
      {
        const bool is_s = pt < 64;
        const int t = pt & 63;
        const float bt = S.beta[gb][t];
        float d = 1.f;  // e^{G_t - G_s} as s walks down from t (products of alpha <= 1)
#pragma unroll
        for (int hb = 1; hb >= 0; --hb) {  // columns [32 hb, 32 hb + 32), walked downwards
          float sv[32];
          tmem_ld32(tm + lane_bits + TM_SQ + 32 * hb, sv);
#pragma unroll
          for (int q = 31; q >= 0; --q) {
            const int s = 32 * hb + q;
            if (s < t) d *= S.alpha[gb][s + 1];
            sv[q] = is_s ? (s < t ? bt * d * sv[q] : 0.f) : (s <= t ? d * sv[q] : 0.f);
          }
          if (is_s) {
#pragma unroll
            for (int q = 0; q < 32; ++q) S.A[t * FP + 32 * hb + q] = sv[q];
          } else if (MODE == kEmit) {
            uint8_t* att = S.att[ci & 1];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              uint4 pk;
              pk.x = pack_h2(sv[8 * ch + 0], sv[8 * ch + 1]);
              pk.y = pack_h2(sv[8 * ch + 2], sv[8 * ch + 3]);
              pk.z = pack_h2(sv[8 * ch + 4], sv[8 * ch + 5]);
              pk.w = pack_h2(sv[8 * ch + 6], sv[8 * ch + 7]);
              *reinterpret_cast<uint4*>(att + sw128_offset(64, t, 32 * hb + 8 * ch)) = pk;
            }
          }
        }
      }
      fence_before_sync();
      named_bar(1, kPrepThreads);
      // ---- next chunk's loads into the stage chunk ci - 1 used (its MMAs are done)
      if (ci + 1 < nch) {
        if (ci >= 1 && !group_wait(S, B_H, (ci - 1) & 1, 1, kPrepThreads)) break;
        issue_loads(ci + 1);
      }
      // ---- T = (I + A)^-1: diagonal 16 x 16 blocks, one warp each, two lanes per column
      {
        const int b = (warp - 8) * 16, cc = lane & 15, half = lane >> 4;
        for (int t = 0; t < 16; ++t) S.Ti[(b + t) * FP + b + cc] = (t == cc) ? 1.f : 0.f;
        __syncwarp();
        for (int t = 1; t < 16; ++t) {
          float x = 0.f;
          for (int s = half; s < t; s += 2) x += S.A[(b + t) * FP + b + s] * S.Ti[(b + s) * FP + b + cc];
          x += __shfl_xor_sync(0xffffffffu, x, 16);
          if (half == 0 && t > cc) S.Ti[(b + t) * FP + b + cc] = -x;
          __syncwarp();
        }
      }
      named_bar(1, kPrepThreads);
      // off-diagonal blocks by sub-diagonal: T_ab = -T_aa sum_{m=b}^{a-1} A_am T_mb
      for (int dist = 1; dist < 4; ++dist) {
        const int nblk = 4 - dist;
        for (int e = pt; e < nblk * 256; e += kPrepThreads) {
          const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
          const int bb = blk, aa = blk + dist;
          float x = 0.f;
          for (int m = bb; m < aa; ++m)
#pragma unroll
            for (int s = 0; s < 16; ++s)
              x += S.A[(aa * 16 + rr) * FP + m * 16 + s] * S.Ti[(m * 16 + s) * FP + bb * 16 + cc];
          S.X[(aa * 16 + rr) * FP + bb * 16 + cc] = x;
        }
        named_bar(1, kPrepThreads);
        for (int e = pt; e < nblk * 256; e += kPrepThreads) {
          const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
          const int bb = blk, aa = blk + dist;
          float x = 0.f;
          for (int s = 0; s <= rr; ++s)
            x += S.Ti[(aa * 16 + rr) * FP + aa * 16 + s] * S.X[(aa * 16 + s) * FP + bb * 16 + cc];
          S.Ti[(aa * 16 + rr) * FP + bb * 16 + cc] = -x;
        }
        named_bar(1, kPrepThreads);
      }
      // T diag(beta e^G) and T diag(beta) as fp16 K-major tiles [t][s]
      for (int e = pt; e < C * 8; e += kPrepThreads) {
        const int t = e >> 3, ch = e & 7;
        uint32_t pw[4], pu[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int s = 8 * ch + 2 * q;
          const float v0 = s <= t ? S.Ti[t * FP + s] : 0.f;
          const float v1 = s + 1 <= t ? S.Ti[t * FP + s + 1] : 0.f;
          const float b0 = S.beta[gb][s], b1 = S.beta[gb][s + 1];
          const float w0 = v0 * b0 * S.eG[gb][s], w1 = v1 * b1 * S.eG[gb][s + 1];
          range_ok = range_ok && fits_half(w0) && fits_half(w1) && fits_half(v0 * b0) &&
                     fits_half(v1 * b1);
          pw[q] = pack_h2(w0, w1);
          pu[q] = pack_h2(v0 * b0, v1 * b1);
        }
        *reinterpret_cast<uint4*>(S.tw + sw128_offset(64, t, 8 * ch)) =
            make_uint4(pw[0], pw[1], pw[2], pw[3]);
        *reinterpret_cast<uint4*>(S.tu + sw128_offset(64, t, 8 * ch)) =
            make_uint4(pu[0], pu[1], pu[2], pu[3]);
      }
      fence_async_smem();
      named_bar(1, kPrepThreads);
      if (pt == 0) mbar_arrive(saddr(&S.bars[B_T]));
      // ---- -w: lane i holds w[t][i] for every t; written as the MN-major tile [i][t]
      if (!group_wait(S, B_WU, ci & 1, 1, kPrepThreads)) break;
      fence_after_sync();
      {
        const int i = pt;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float wv[32];
          tmem_ld32(tm + lane_bits + TM_W + 32 * hb, wv);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 pk;
            pk.x = pack_h2(-wv[8 * ch + 0], -wv[8 * ch + 1]);
            pk.y = pack_h2(-wv[8 * ch + 2], -wv[8 * ch + 3]);
            pk.z = pack_h2(-wv[8 * ch + 4], -wv[8 * ch + 5]);
            pk.w = pack_h2(-wv[8 * ch + 6], -wv[8 * ch + 7]);
#pragma unroll
            for (int q = 0; q < 8; ++q) range_ok = range_ok && fits_half(wv[8 * ch + q]);
            *reinterpret_cast<uint4*>(S.nw + sw128_offset(128, i, 32 * hb + 8 * ch)) = pk;
          }
        }
      }
      fence_async_smem();
      fence_before_sync();
      named_bar(1, kPrepThreads);
      if (pt == 0) mbar_arrive(saddr(&S.bars[B_WR]));
      // ---- the next chunk's data
      if (ci + 1 < nch) finish_data(ci + 1);
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    if (!range_ok) S.range_bad = 1;
  } else if (lane == 0) {
    // =============================================================== MMA issue (1 thread)
    const uint32_t ID_SQ = idesc_f16(128, 64, 0, 0);
    const uint32_t ID_WU = idesc_f16(128, 64, 1, 0);
    const uint32_t ID_D = idesc_f16(128, 64, 0, 1);
    const uint32_t ID_O = idesc_f16(128, 64, 0, 0);
    const uint32_t ID_DH = idesc_f16(128, 128, 0, 1);
    auto sq = [&](int ci) {
      const uint32_t kq = saddr(S.kq[ci & 1]);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t d = sdesc(kq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
        mma_ss(tm + TM_SQ, d, d, ID_SQ, ks > 0);
      }
      mma_commit(saddr(&S.bars[B_SQ]));
    };
    auto wu = [&](int ci) {
      const uint32_t kq = saddr(S.kq[ci & 1]), vv = saddr(S.v[ci & 1]);
      const uint32_t tw = saddr(S.tw), tu = saddr(S.tu);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tm + TM_W, sdesc(kq + ks * 2048, 16384, 1024), sdesc(tw + ks * 32, 16, 1024),
               ID_WU, ks > 0);
      if (MODE != kSumM) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ss(tm + TM_U, sdesc(vv + ks * 2048, 8192, 1024), sdesc(tu + ks * 32, 16, 1024),
                 ID_WU, ks > 0);
      }
      mma_commit(saddr(&S.bars[B_WU]));
    };
    if (nch > 0) {
      bool ok = single_wait(S, B_X0, 0);
      if (ok) sq(0);
      ok = ok && single_wait(S, B_T, 0);
      if (ok) wu(0);
      for (int ci = 0; ok && ci < nch; ++ci) {
        const uint32_t kq = saddr(S.kq[ci & 1]);
        // delta^T (+)= h^T (-w)^T ;  O1^T = h^T Q^T
        ok = single_wait(S, B_WR, ci & 1) && single_wait(S, B_HR, ci & 1);
        if (!ok) break;
        fence_after_sync();
        const uint32_t nw = saddr(S.nw);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ah = tm + TM_H + 64 * (ks >> 2) + 8 * (ks & 3);
          mma_ts(tm + TM_U, ah, sdesc(nw + ks * 2048, 16384, 1024), ID_D,
                 (MODE != kSumM) || ks > 0);
          if (MODE == kEmit)
            mma_ts(tm + TM_O1, ah,
                   sdesc(kq + (ks >> 2) * 16384 + 64 * 128 + (ks & 3) * 32, 16, 1024), ID_O,
                   ks > 0);
        }
        mma_commit(saddr(&S.bars[B_D]));
        if (ci + 1 < nch) {
          ok = single_wait(S, B_X0 + ((ci + 1) & 1), ((ci + 1) >> 1) & 1);
          if (!ok) break;
          sq(ci + 1);
        }
        // O2^T = delta^T attn_i^T ;  Dh^T = delta'^T K
        ok = single_wait(S, B_DR, ci & 1);
        if (!ok) break;
        fence_after_sync();
        const uint32_t att = saddr(S.att[ci & 1]);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t col = TM_U + 32 * (ks >> 1) + 8 * (ks & 1);
          if (MODE == kEmit)
            mma_ts(tm + TM_O2, tm + col, sdesc(att + ks * 32, 16, 1024), ID_O, ks > 0);
          mma_ts(tm + TM_H, tm + col + 16, sdesc(kq + ks * 2048, 16384, 1024), ID_DH, ks > 0);
        }
        mma_commit(saddr(&S.bars[B_H]));
        if (ci + 1 < nch) {
          ok = single_wait(S, B_T, (ci + 1) & 1);
          if (!ok) break;
          wu(ci + 1);
        }
      }
    }
  }

  // ---- teardown: every role has left its loop
  fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    if (aborted(S)) set_status(a.status, GDN_ERR_DEVICE_TIMEOUT);
    if (S.range_bad) set_status(a.status, GDN_ERR_DEVICE_RANGE);
  }
  if (warp == 12) {
    fence_after_sync();
    tmem_dealloc(tm, 512);
  }
}

template <int MODE>
cudaError_t launch5(const Args& a, cudaStream_t s) {
  const dim3 grid((unsigned)(a.N * a.P), a.hv, 1);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(tc5_chunk_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc5_chunk_kernel<MODE><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t tc5_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t tc5_summary(const Args& a, cudaStream_t s) {
  cudaError_t e = launch5<kSumM>(a, s);
  if (e != cudaSuccess) return e;
  return launch5<kSumU>(a, s);
}

cudaError_t tc5_emit(const Args& a, cudaStream_t s) { return launch5<kEmit>(a, s); }

}  // namespace gdn
