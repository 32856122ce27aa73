// gdn_tc5.cu -- tcgen05 (5th-generation tensor core) kernels for the chunked gated delta
// rule forward, bf16 I/O, K = V = 128, C = 64, fp32 state.
//
// One CTA per (segment, value head) walks the segment's chunks ("Add context parallelism to
// the Gated Delta Net", section "Implementation": phase 3 re-emit, or phase 1 summary on one
// half of X = [M | U]).  Every contraction is a tcgen05.mma with fp32 accumulation in Tensor
// Memory; products are taken in transposed form so that M = 128 (a state or feature index)
// fills the 128 TMEM lanes:
//   [S ; QK]     = [K ; Q] K^T                          (128 x 64, K = 128; bf16 as loaded)
//   w^T          = K^T (T diag(beta e^G))^T              (128 x 64, K = 64)
//   u^T          = V^T (T diag(beta))^T                  (128 x 64, K = 64)
//   O^T          = h^T q_g^T                            (128 x 64, K = 128)
//   D^T          = h^T (-w)^T                           (128 x 64, K = 128)
//   O^T         += delta^T attn_i^T                      (128 x 64, K = 64)
//   Dh^T         = (diag(e^{G_last - G}) delta)^T K      (128 x 128, K = 64)
// with delta = u + D, q_g = diag(e^G) Q, o = q_g h + attn_i delta and h <- gamma h + Dh.  The
// u product writes u^T into the D accumulator, so that the D product yields delta itself.
// [S ; QK] reads K and Q as loaded (bf16); the converter warps then write K as fp16 (a
// separate, double-buffered tile), and V and q_g as fp16 in place (q_g keeps Q's K-major
// layout, so it needs no transpose), and every later product has fp16 operands.  The state h^T lives in registers
// (fp32) of the chain warps; its fp16 copy, delta and delta' are written back into TMEM as the
// A operands of the next products.  T = (I + A)^-1 is blocked by 16 x 16: the diagonal inverses
// by fp32 forward substitution in registers, the off-diagonal blocks
// T_ab = -T_aa sum_m A_am T_mb with warp-level mma.sync.
//
// Phase 3 from factor records (kEmitR) loads Q and the chunk's record (-w^T, fp16 K, u^T) and
// prepares nothing: two prepare warps write Q^T (fp16, MN-major) beside -w^T, so that one
// N = 128 product gives [D^T | (Q h)^T] = h^T [-w^T | Q^T]; Q K^T takes Q^T and the record's K;
// attn_i delta goes to its own columns, and the chain forms o = e^{G_t} (Q h)_t + (attn_i delta)_t.
//
// Warp roles (512 threads):
//   warps 0-7   chain:     TMEM lane = state row c; warps w and w + 4 split the columns
//   warps 8-11  prepare:   masked gram and attn_i, the triangular solve, -w; one chunk ahead
//                          (kEmitR: warps 8, 9 attn_i, warps 10, 11 the fp16 Q^T)
//   warp 12     MMA:       waits for each product's inputs in a fixed order; lane 0 issues
//   warp 13     loader:    TMA boxes of K, Q, V, cp.async of g, beta and bulk copies of the
//                          factor records into the free stage
//   warps 14-15 converter: decay tables, fp16 K, V and q_g (kEmitR: the tables only; kSumML:
//                          idle)
// Hand-offs use mbarriers: a producing group arrives with every thread (the barrier counts the
// group), a consumer waits with hardware-suspended try_wait (no issue slots spent).  Every wait
// is bounded; one that gives up records GDN_ERR_DEVICE_TIMEOUT and the thread carries on, and
// each role checks the record at one group-uniform point per chunk and leaves its loop, so the
// CTA always reaches its TMEM release.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"
#include "gdn_tc5_util.cuh"
#include "gdn_warp_mma.cuh"

namespace gdn {
namespace {

using namespace sm100;
using namespace warp_mma;
using namespace tc5u;

constexpr int C = kChunk;  // 64
constexpr int KD = 128, VD = 128;
constexpr int kChainThreads = 256, kPrepThreads = 128, kConvThreads = 64;
constexpr int kThreads = kChainThreads + kPrepThreads + 64 + kConvThreads;
constexpr long long kWaitCycles = 2000000000LL;  // default wait limit: about a second
constexpr long long kDrainCycles = 200000000LL;  // teardown waits for in-flight copies, products

// With per-chunk factor records in the workspace, the U half stores each chunk's -w^T, fp16 K,
// u^T and the state update's decay; kSumML (the M half) and kEmitR (phase 3) load them instead
// of computing them, and run only what depends on the state (kEmitR also forms attn_i and q_g).
enum Mode { kEmit = 0, kSumM = 1, kSumU = 2, kSumML = 3, kEmitR = 4 };

// Record layout: the fp16 tiles -w^T [i][t] (MN-major), K [t][i] (MN-major) and u^T [c][t]
// (128-byte swizzled rows) as they sit in shared memory, then e^{G_last - G_t} (64 floats) and
// gamma.
constexpr uint32_t kRecNw = 0, kRecKh = 16384, kRecU = 32768, kRecTbl = 49152;
constexpr uint32_t kRecTblBytes = 272;
constexpr size_t kRecBytes = 49664;

// TMEM columns (512 allocated)
constexpr uint32_t TM_SQ = 0;    // [S ; QK]               64 fp32
constexpr uint32_t TM_W = 64;    // w^T                    64 fp32
constexpr uint32_t TM_U = 128;   // fp16 delta' (columns 32 hf + 0..15)
constexpr uint32_t TM_DO = 192;  // u^T + D = delta^T, then fp16 delta, in 0-63; o^T in 64-127
constexpr uint32_t TM_H = 320;   // Dh^T                   128 fp32, then fp16 h^T

// mbarriers: who completes them
enum Bar {
  B_SQ = 0,    // [S ; QK] of a chunk is in TMEM                      MMA commit
  B_E2,        // the gram has read it and the decay tables           prepare (128)
  B_TB,        // decay tables of a chunk are in shared memory        converter (64)
  B_CV,        // fp16 K, V and q_g of a chunk are ready              converter (64)
               //   (kEmitR: fp16 Q^T is ready                         transposer (64))
  B_T,         // the T tiles are ready                               prepare (128)
  B_WU,        // w^T, u^T are in TMEM                                MMA commit
  B_WR,        // -w^T is in shared memory                            prepare (128)
  B_HR,        // fp16 h^T is in TMEM and the previous o^T was read   chain (256)
  B_D,         // delta^T = u^T + D^T is in TMEM                      MMA commit
  B_DR,        // fp16 delta, delta' are in TMEM                      chain (256)
  B_H,         // Dh^T and o^T are complete                           MMA commit
  B_L0, B_L1, B_L2,  // stage loaded: byte count (+ 32 cp.async arrivals)  loader
  B_F0, B_F1, B_F2,  // stage free (its chunk's w, u and q_g h products are done)  MMA commit
  B_KF0, B_KF1,  // fp16 K tile free (its chunk's Dh is done)         MMA commit
  B_QF0, B_QF1,  // kEmitR: the staged bf16 Q, g and beta have been read  transposer + converter
  B_RL0, B_RL1,  // kEmitR: a record is staged (byte count)              loader
  B_RF0, B_RF1,  // kEmitR: its record stage is free (D, O2, Dh done)    MMA commit
  B_END,       // every product issued has completed                  MMA commit
  kNumBars
};
template <int MODE>
__device__ __forceinline__ uint32_t bar_count(int b) {
  return (b == B_E2 && MODE == kEmitR)         ? 64u  // (kEmitR: the two gram warps)
         : (b == B_QF0 || b == B_QF1)          ? (uint32_t)(64 + kConvThreads)
         : (b == B_E2 || b == B_T || b == B_WR)  ? (uint32_t)kPrepThreads
         : (b == B_TB || b == B_CV) ? (uint32_t)kConvThreads
         : (b == B_HR || b == B_DR)            ? (uint32_t)kChainThreads
         : (b >= B_L0 && b <= B_L2)            ? (MODE == kSumML ? 1u : 33u)
         : (b == B_RL0 || b == B_RL1)          ? 1u
                                               : 1u;
}

struct Smem {
  uint8_t kq[2][2 * 128 * 128];  // per stage: [kblk][K rows 0-63 | Q rows 64-127][128 B], bf16;
                                 // Q becomes fp16 q_g in place
  uint8_t v[2][2 * 64 * 128];    // per stage: [kblk][64 rows][128 B]; V -> fp16 in place
  uint8_t kh[2][2 * 64 * 128];   // fp16 K: [kblk][64 rows][128 B] (chunk parity)
  uint8_t att[2][64 * 128];      // attn_i [t][s] fp16, K-major B (chunk parity)
  uint8_t tw[64 * 128];          // T diag(beta e^G) [t][s] fp16, K-major B
  uint8_t tu[64 * 128];          // T diag(beta) [t][s] fp16, K-major B
  uint8_t nw[128 * 128];         // -w^T [i][t] fp16, MN-major B of D
  uint8_t ah[64 * 128];          // masked gram A [t][s], fp16
  uint8_t th[64 * 128];          // blocks of (I + A)^-1 [t][s], fp16 operands
  uint8_t xs[4][16 * 48];        // 16 x 16 fp16 blocks for mma.sync, 48-byte rows
  alignas(16) float adiag[C][20];  // the diagonal 16 x 16 blocks of A, fp32 (padded rows)
  float wd[4][16 * 17];          // per-warp fp32 16 x 16 block of T (padded rows)
  float gst[2][2][C];            // g and beta of a staged chunk
  float G[3][C], eG[3][C], eGLG[3][C], beta[3][C], gamma[4];
  // decay e^{G_t - G_s} (s <= t) of the chunk the gram reads next: on the 16-block of t it is
  // dd*[t][s & 15]; for s in an earlier block b it is rf*[t][b] * cf[s], with
  // rf = e^{G_t - G_e}, cf = e^{G_e - G_s} and e the last row of block b (both <= 1 for g <= 0).
  // The A rows (ddA, rfA) carry beta_t and exclude s = t; attn_i's (ddO, rfO) keep s = t.
  alignas(16) float ddA[C][20];  // padded rows: conflict-free 16-byte accesses by row
  alignas(16) float ddO[C][20];
  alignas(16) float rfA[C][4];
  alignas(16) float rfO[C][4];
  alignas(16) float cf[C];
  alignas(16) float tbl[3][68];  // kSumML: e^{G_last - G_t} and gamma of a staged record
  uint64_t bars[kNumBars];
  uint32_t tmem_base;
  int abort_flag;
  int range_bad;
  long long wait_cycles;  // this call's limit on a bounded wait
};

// Members read or written with 16-byte vector accesses, ldmatrix / stmatrix or the tensor core
// must sit on 16-byte (swizzled tiles: 1024-byte) boundaries of the 1024-aligned base.
static_assert(offsetof(Smem, kq) % 1024 == 0 && offsetof(Smem, v) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, kh) % 1024 == 0 && offsetof(Smem, att) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, tw) % 1024 == 0 && offsetof(Smem, tu) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, nw) % 1024 == 0 && offsetof(Smem, ah) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, th) % 1024 == 0 && offsetof(Smem, xs) % 16 == 0, "tile alignment");
static_assert(offsetof(Smem, ddA) % 16 == 0 && offsetof(Smem, ddO) % 16 == 0, "vector alignment");
static_assert(offsetof(Smem, rfA) % 16 == 0 && offsetof(Smem, rfO) % 16 == 0, "vector alignment");
static_assert(offsetof(Smem, adiag) % 16 == 0, "vector alignment");
static_assert(offsetof(Smem, cf) % 16 == 0 && offsetof(Smem, bars) % 8 == 0, "alignment");
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory per block");

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ bool aborted(Smem& S) {
  return *reinterpret_cast<volatile int*>(&S.abort_flag) != 0;
}
__device__ __forceinline__ void set_abort(Smem& S) {
  *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
}
// Bounded wait for the phase with the given parity, suspended in hardware between tries.  On
// giving up (about a second, or at once when another thread already gave up) it records the
// abort flag; the caller carries on and leaves at its next group-uniform check.
__device__ __noinline__ void wait_bar_slow(Smem& S, uint32_t a, uint32_t parity) {
  const long long t_end = clock64() + S.wait_cycles;
  while (!mbar_try(a, parity)) {
    if (clock64() > t_end || aborted(S)) {
      set_abort(S);
      return;
    }
  }
}
__device__ __forceinline__ void wait_bar(Smem& S, int bar, uint32_t parity) {
  const uint32_t a = saddr(&S.bars[bar]);
  if (mbar_try(a, parity)) return;
  wait_bar_slow(S, a, parity);
}
__device__ __forceinline__ void arrive(Smem& S, int bar) { mbar_arrive(saddr(&S.bars[bar])); }
// Teardown wait for this CTA's own in-flight copies or products: bounded, and it does not give up
// when the abort flag is set (the TMEM and shared memory must not be released under them).
__device__ __noinline__ void wait_bar_drain(Smem& S, int bar, uint32_t parity) {
  const uint32_t a = saddr(&S.bars[bar]);
  const long long t_end = clock64() + kDrainCycles;
  while (!mbar_try(a, parity) && clock64() < t_end) {
  }
}

// The record of chunk cg (index within sequence n, which starts at token sb) of value head j:
// slots are the 64-token windows of the packed token axis, plus n so that a sequence's last,
// partial chunk and the next sequence's first chunk never share one.
__device__ __forceinline__ char* chunk_record(const Args& a, int n, int64_t sb, int64_t cg,
                                              int j) {
  const int64_t slot = ((sb + C * cg) >> 6) + n;
  return static_cast<char*>(a.wy) + (slot * a.hv + j) * (int64_t)kRecBytes;
}

// ------------------------------------------------------------------ the kernel

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc5_chunk_kernel(Args a, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x, j = blockIdx.y;
  const int n_seq = seg / a.P, r = seg % a.P;
  constexpr bool OUT = MODE == kEmit || MODE == kEmitR;  // phase 3: outputs o
  if (!OUT && r == a.P - 1 && a.skip_last_summary) return;
  const int kh = j / (a.hv / a.hk);
  int64_t sb, se;
  if (!seq_bounds(a.cu, n_seq, a.T, a.status, sb, se)) return;
  int64_t c0, c1;
  segment_chunks(se - sb, a.P, r, c0, c1);
  const int nch = (int)(c1 - c0);

  // ---- setup: mbarriers, TMEM
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) mbar_init(saddr(&S.bars[b]), bar_count<MODE>(b));
    S.abort_flag = 0;
    S.wait_cycles = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
    S.range_bad = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 12) {
    tmem_alloc(saddr(&S.tmem_base), 512);
    tmem_relinquish();
  }
  if (MODE != kSumML && tid == kChainThreads) {
    if (MODE != kEmitR)
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    if (OUT)
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    if (MODE != kSumM && MODE != kEmitR)
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = S.tmem_base;
  // -w^T of chunk ci; the U half keeps two, the second in the attn_i tiles it has no use for,
  // so that the copy of one into the chunk's record overlaps the next chunk
  auto nw_tile = [&](int ci) -> uint8_t* {
    return (MODE == kSumU && (ci & 1)) ? S.att[0] : S.nw;
  };
  // kSumML stages: the -w^T and K tiles of a record, 32 KB each, in the K | Q and V tiles
  auto rec_stage = [&](int st) -> uint8_t* { return st == 0 ? S.kq[0] : st == 1 ? S.kq[1] : S.v[0]; };
  // kEmitR: the bf16 Q boxes of a stage land in tiles the factors would use (16 KB each); the
  // stage's K | Q tile holds [-w^T rows 0-63 | Q^T box 0 | -w^T rows 64-127 | Q^T box 1], so
  // that one MN-major operand with its second 64 columns 8 KB on is [-w^T | Q^T]
  auto qstage = [&](int sg) -> uint8_t* { return sg ? S.nw : S.tw; };

  if (warp < 8) {
    // =============================================================== chain (256 threads)
    const int hf = warp >> 2;                 // column half of the state row
    const int c = (warp & 3) * 32 + lane;     // state row = TMEM lane
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    bool range_ok = true;
    float h[64];                              // h^T[c][64 hf .. 64 hf + 63]
    {
      const float* src = nullptr;
      if (OUT && a.h_in) src = a.h_in + ((int64_t)seg * a.hv + j) * KD * VD;
#pragma unroll
      for (int q = 0; q < 64; ++q) {
        const int i = 64 * hf + q;
        float x = 0.f;
        if (OUT) x = src ? src[i * VD + c] : 0.f;
        if (MODE == kSumM || MODE == kSumML) x = (i == c) ? 1.f : 0.f;
        h[q] = x;
      }
    }
    // fp16 h^T into TMEM (the A operand of D and of q_g h).  Not range-checked: an infinite h^T
    // makes delta infinite or NaN, and delta is checked.
    auto publish_h = [&]() {
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        uint32_t p[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) p[q] = pack_h2(h[16 * piece + 2 * q], h[16 * piece + 2 * q + 1]);
        tmem_st8_nw(tm + lane_bits + TM_H + 64 * hf + 8 * piece, p);
      }
    };
    if (nch > 0) {
      publish_h();
      tmem_wait_st();
      fence_before_sync();
      // (a.fault == 1, for tests of the bounded waits: the first hand-off is never signalled,
      // so the MMA warp's wait for it must expire)
      if (a.fault != 1) arrive(S, B_HR);
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    for (int ci = 0; ci < nch; ++ci) {
      const int gb = ci % 3;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      const float* eglg = MODE == kSumML ? S.tbl[gb] : S.eGLG[gb];
      // ---- delta = u + D -> fp16 delta (into D's columns) and delta' (into u's columns).  TMEM
      // is read two 16-column pieces at a time with one wait, and written without a wait per
      // store (one wait before the hand-off).
      wait_bar(S, B_D, ci & 1);
      if (MODE == kEmitR) wait_bar(S, B_RL0 + (ci & 1), (ci >> 1) & 1);  // u^T of the record
      fence_after_sync();
      {
        uint32_t dr[2][16];
        tmem_ld16_nw(tm + lane_bits + TM_DO + 32 * hf, dr[0]);
        tmem_ld16_nw(tm + lane_bits + TM_DO + 32 * hf + 16, dr[1]);
        tmem_wait_ld16x2(dr[0], dr[1]);
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          float d[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) d[q] = __uint_as_float(dr[piece][q]);
          if (MODE == kEmitR) {  // u^T[c][t], fp16, 128-byte swizzled rows
            const uint8_t* ur = S.v[ci & 1] + c * 128;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int ch = 4 * hf + 2 * piece + h2;
              const uint4 x = *reinterpret_cast<const uint4*>(ur + ((ch ^ (c & 7)) << 4));
              const uint32_t* xw = reinterpret_cast<const uint32_t*>(&x);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xw[i]));
                d[8 * h2 + 2 * i] += f.x;
                d[8 * h2 + 2 * i + 1] += f.y;
              }
            }
          }
          uint32_t pd[8], pp[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int t = 32 * hf + 16 * piece + 2 * q;
            range_ok = range_ok && fits_half(d[2 * q]) && fits_half(d[2 * q + 1]);
            pd[q] = pack_h2(d[2 * q], d[2 * q + 1]);
            pp[q] = pack_h2(d[2 * q] * eglg[t], d[2 * q + 1] * eglg[t + 1]);
          }
          if (OUT) tmem_st8_nw(tm + lane_bits + TM_DO + 32 * hf + 8 * piece, pd);
          tmem_st8_nw(tm + lane_bits + TM_U + 32 * hf + 8 * piece, pp);
        }
        tmem_wait_st();
      }
      fence_before_sync();
      arrive(S, B_DR);

      // ---- the state update; its fp16 copy and the read of o^T before the hand-off
      wait_bar(S, B_H, ci & 1);
      fence_after_sync();
      {
        const float gam = MODE == kSumML ? S.tbl[gb][64] : S.gamma[gb];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t hr[2][16];
          tmem_ld16_nw(tm + lane_bits + TM_H + 64 * hf + 32 * half, hr[0]);
          tmem_ld16_nw(tm + lane_bits + TM_H + 64 * hf + 32 * half + 16, hr[1]);
          tmem_wait_ld16x2(hr[0], hr[1]);
#pragma unroll
          for (int p2 = 0; p2 < 2; ++p2)
#pragma unroll
            for (int q = 0; q < 16; ++q)
              h[32 * half + 16 * p2 + q] =
                  gam * h[32 * half + 16 * p2 + q] + __uint_as_float(hr[p2][q]);
        }
      }
      if (ci + 1 < nch) publish_h();  // (its stores complete at the wait below)
      uint32_t ob[16];
      if (OUT) {
        if (MODE == kEmitR) {  // o = e^{G_t} (q h)_t + (attn_i delta)_t, a piece at a time
#pragma unroll
          for (int piece = 0; piece < 2; ++piece) {
            uint32_t orr[16], o2r[16];
            tmem_ld16_nw(tm + lane_bits + TM_DO + 64 + 32 * hf + 16 * piece, orr);
            tmem_ld16_nw(tm + lane_bits + TM_W + 32 * hf + 16 * piece, o2r);
            tmem_wait_ld16x2(orr, o2r);
            const float* eg = &S.eG[gb][32 * hf + 16 * piece];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              ob[8 * piece + q] =
                  pack_bf2(fmaf(eg[2 * q], __uint_as_float(orr[2 * q]), __uint_as_float(o2r[2 * q])),
                           fmaf(eg[2 * q + 1], __uint_as_float(orr[2 * q + 1]),
                                __uint_as_float(o2r[2 * q + 1])));
          }
        } else {
          uint32_t orr[2][16];
          tmem_ld16_nw(tm + lane_bits + TM_DO + 64 + 32 * hf, orr[0]);
          tmem_ld16_nw(tm + lane_bits + TM_DO + 64 + 32 * hf + 16, orr[1]);
          tmem_wait_ld16x2(orr[0], orr[1]);
#pragma unroll
          for (int piece = 0; piece < 2; ++piece)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              ob[8 * piece + q] = pack_bf2(__uint_as_float(orr[piece][2 * q]),
                                           __uint_as_float(orr[piece][2 * q + 1]));
        }
      }
      tmem_wait_st();
      fence_before_sync();
      if (ci + 1 < nch) arrive(S, B_HR);
      if (OUT) {  // o[t][j][c] for t = 32 hf .. 32 hf + 31
        const int64_t stride = (int64_t)a.hv * VD;
        __nv_bfloat16* po = out + ((t0 + 32 * hf) * a.hv + j) * VD + c;
        const int nt = L - 32 * hf;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&ob[q]);
          if (2 * q < nt) po[0] = p2.x;
          if (2 * q + 1 < nt) po[stride] = p2.y;
          po += 2 * stride;
        }
      }
      if (!named_bar_and(2, kChainThreads, !aborted(S))) break;
    }
    if (!range_ok) S.range_bad = 1;
    // ---- the final state: h^T[c][i] = h[i][c]
    float* dst = nullptr;
    if (OUT) {
      if (a.h_final && r == a.P - 1) dst = a.h_final + ((int64_t)n_seq * a.hv + j) * KD * VD;
    } else if (MODE == kSumM || MODE == kSumML) {
      dst = a.M_out + ((int64_t)seg * a.hv + j) * KD * KD;
    } else {
      dst = a.U_out + ((int64_t)seg * a.hv + j) * KD * VD;
    }
    if (dst && !aborted(S)) {
#pragma unroll
      for (int q = 0; q < 64; ++q) dst[(64 * hf + q) * VD + c] = h[q];
    }
  } else if (warp < 12) {
    if (MODE != kSumML) {  // (kSumML loads what the prepare warps compute)
    // =============================================================== prepare (128 threads)
    const int pt = tid - kChainThreads;       // 0..127 = TMEM lane of this thread
    const int wb = warp - 8;                  // 0..3: this warp's 16-row block of T
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    const int g8 = lane >> 2, q4 = lane & 3;
    const uint32_t ah_s = saddr(S.ah), th_s = saddr(S.th);
    const bool lo_warps = pt < 64;

    // the strictly upper blocks of T diag(.), rows 0-31 x columns 32-63 of A and attn_i, and the
    // upper right 8 x 8 of each warp's fp32 block of T are zero for every chunk
    for (int e = pt; e < 64 * 128 / 16; e += kPrepThreads) {
      if (MODE != kEmitR) {  // (kEmitR stages records there)
        reinterpret_cast<uint4*>(S.tw)[e] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(S.tu)[e] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (MODE != kEmitR) reinterpret_cast<uint4*>(S.ah)[e] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(S.att[0])[e] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(S.att[1])[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = pt; e < 4 * 16 * 17; e += kPrepThreads) (&S.wd[0][0])[e] = 0.f;
    named_bar(1, kPrepThreads);

    // 32 fp32 values as fp16 into row t, columns 32 hb .. 32 hb + 31, of a 64-column tile
    auto put_row32 = [&](uint8_t* dst, int t, int hb, const float (&sv)[32]) {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint4 pk;
        pk.x = pack_h2(sv[8 * ch + 0], sv[8 * ch + 1]);
        pk.y = pack_h2(sv[8 * ch + 2], sv[8 * ch + 3]);
        pk.z = pack_h2(sv[8 * ch + 4], sv[8 * ch + 5]);
        pk.w = pack_h2(sv[8 * ch + 6], sv[8 * ch + 7]);
        *reinterpret_cast<uint4*>(dst + sw128_offset(64, t, 32 * hb + 8 * ch)) = pk;
      }
    };

    // ---- masked gram A (fp16 tile + fp32 diagonal blocks) and attn_i from [S ; QK].  Row t
    // meets 16-blocks below its own (decay rf[t][b] cf[s]), its own block (dd[t][s & 15]) and
    // blocks above (zero).  Rows 32-63 see only lower blocks in columns 0-31 and rows 0-31 only
    // upper blocks in columns 32-63 (left zero from the start), so each row computes one plain
    // half at most and one half holding its own block.
    auto gram = [&](int ci) {
      wait_bar(S, B_SQ, ci & 1);
      wait_bar(S, B_TB, ci & 1);
      fence_after_sync();
      // warps 8, 9: rows of A (kEmitR: of attn_i, from Q K^T); warps 10, 11: rows of attn_i
      const bool lo = pt < 64, is_s = MODE != kEmitR && lo;
      if (MODE == kEmit || lo) {
        const int t = pt & 63, hi = t >> 5, ab = (t >> 4) & 1;  // hi is warp-uniform
        const float4 rf4 = *reinterpret_cast<const float4*>(is_s ? S.rfA[t] : S.rfO[t]);
        uint8_t* dst = is_s ? S.ah : S.att[ci & 1];
        float sv[32];
        if (hi) {
          tmem_ld32(tm + lane_bits + TM_SQ, sv);
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4) {
            const float4 cf4 = *reinterpret_cast<const float4*>(&S.cf[c4]);
            const float f = c4 < 16 ? rf4.x : rf4.y;
            sv[c4 + 0] *= f * cf4.x;
            sv[c4 + 1] *= f * cf4.y;
            sv[c4 + 2] *= f * cf4.z;
            sv[c4 + 3] *= f * cf4.w;
          }
          put_row32(dst, t, 0, sv);
        }
        tmem_ld32(tm + lane_bits + TM_SQ + 32 * hi, sv);
        const float* ddr = is_s ? S.ddA[t] : S.ddO[t];
        const float fb = hi ? rf4.z : rf4.x;  // to the last row of block 2 hi (when ab = 1)
#pragma unroll
        for (int c4 = 0; c4 < 16; c4 += 4) {  // block 2 hi: own block (ab = 0) or below it
          const float4 cf4 = *reinterpret_cast<const float4*>(&S.cf[32 * hi + c4]);
          const float4 d4 = *reinterpret_cast<const float4*>(ddr + c4);
          sv[c4 + 0] *= ab ? fb * cf4.x : d4.x;
          sv[c4 + 1] *= ab ? fb * cf4.y : d4.y;
          sv[c4 + 2] *= ab ? fb * cf4.z : d4.z;
          sv[c4 + 3] *= ab ? fb * cf4.w : d4.w;
        }
#pragma unroll
        for (int c4 = 16; c4 < 32; c4 += 4) {  // block 2 hi + 1: own block (ab = 1) or above
          const float4 d4 = *reinterpret_cast<const float4*>(ddr + c4 - 16);
          sv[c4 + 0] *= ab ? d4.x : 0.f;
          sv[c4 + 1] *= ab ? d4.y : 0.f;
          sv[c4 + 2] *= ab ? d4.z : 0.f;
          sv[c4 + 3] *= ab ? d4.w : 0.f;
        }
        if (is_s) {
#pragma unroll
          for (int k4 = 0; k4 < 16; k4 += 4)
            *reinterpret_cast<float4*>(&S.adiag[t][k4]) =
                ab ? make_float4(sv[16 + k4], sv[17 + k4], sv[18 + k4], sv[19 + k4])
                   : make_float4(sv[k4], sv[1 + k4], sv[2 + k4], sv[3 + k4]);
        }
        put_row32(dst, t, hi, sv);
      }
      if (OUT && !is_s) fence_async_smem();  // attn_i feeds the tensor core
      fence_before_sync();
      arrive(S, B_E2);
    };

    // ---- 16 x 16 blocks on mma.sync (m16n8k16, two n8 tiles per block)
    // x += A_blk(a_r, a_c) B_blk(b_r, b_c), A from a tile [m][k] and B from a tile [k][n]
    auto mma_blk = [&](float (&x)[2][4], uint32_t a_base, int a_r, int a_c, uint32_t b_base,
                       int b_r, int b_c) {
      uint32_t af[4], bf[4];
      load_a<64>(a_base, a_r, a_c, af);
      load_b_kn<64>(b_base, b_r, b_c, bf);
      mma16816(x[0], af, bf[0], bf[1]);
      mma16816(x[1], af, bf[2], bf[3]);
    };
    // accumulator fragment -> fp16 block xs[tile] ([k][n], 48-byte rows)
    auto frag_to_xs = [&](const float (&x)[2][4], int tile) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<uint32_t*>(S.xs[tile] + g8 * 48 + (8 * nt + 2 * q4) * 2) =
            pack_h2(x[nt][0], x[nt][1]);
        *reinterpret_cast<uint32_t*>(S.xs[tile] + (g8 + 8) * 48 + (8 * nt + 2 * q4) * 2) =
            pack_h2(x[nt][2], x[nt][3]);
      }
    };
    // y += T_blk(a_r, a_c) xs[tile]
    auto mma_xs = [&](float (&y)[2][4], int a_r, int a_c, int tile) {
      uint32_t af[4], bf[4];
      load_a<64>(th_s, a_r, a_c, af);
      const int mi = lane >> 3, rr = lane & 7;
      ldsm_x4_t(saddr(S.xs[tile]) + (rr + ((mi & 1) << 3)) * 48 + ((mi >> 1) << 3) * 2, bf);
      mma16816(y[0], af, bf[0], bf[1]);
      mma16816(y[1], af, bf[2], bf[3]);
    };
    // T_ab = -y into th and its scaled copies tw, tu
    auto store_t = [&](const float (&y)[2][4], int ab, int bb, int gb) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int row = 16 * ab + g8 + 8 * hr, col = 16 * bb + 8 * nt + 2 * q4;
          const float v0 = -y[nt][2 * hr], v1 = -y[nt][2 * hr + 1];
          const float u0 = S.beta[gb][col], u1 = S.beta[gb][col + 1];
          const float w0 = u0 * S.eG[gb][col], w1 = u1 * S.eG[gb][col + 1];
          const uint32_t off = sw128_offset(64, row, col);
          *reinterpret_cast<uint32_t*>(S.th + off) = pack_h2(v0, v1);
          *reinterpret_cast<uint32_t*>(S.tw + off) = pack_h2(v0 * w0, v1 * w1);
          *reinterpret_cast<uint32_t*>(S.tu + off) = pack_h2(v0 * u0, v1 * u1);
        }
    };

    // ---- T = (I + A)^-1 and the two scaled copies the w / u products read.  T, w and h^T are
    // not range-checked: an infinite fp16 value there makes delta infinite or NaN.
    auto solve = [&](int ci) {
      const int gb = ci % 3;
      {  // Diagonal block wb = [[P, 0], [R, Q]] (8 x 8 parts): P^-1 and Q^-1 by forward
         // substitution side by side (lane c < 8: column c of P^-1, 8 <= c < 16: column c - 8
         // of Q^-1), then the lower left block -Q^-1 (R P^-1) by all lanes, in fp32 in wd.
        float* W = S.wd[wb];
        const float* Ab = &S.adiag[16 * wb][0];
        {
          const int c = lane & 7, rb = lane & 8;
          const float* Ar = Ab + rb * 21;  // A[rb + r][rb + s] = Ar[20 r + s]
          float x[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
          for (int r = 1; r < 8; ++r) {
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < r; ++s2) {
              if (s2 & 1) x1 += Ar[20 * r + s2] * x[s2];
              else x0 += Ar[20 * r + s2] * x[s2];
            }
            if (r > c) x[r] = -(x0 + x1);
          }
          if (lane < 16) {
#pragma unroll
            for (int r = 0; r < 8; ++r) W[(rb + r) * 17 + rb + c] = x[r];
          }
        }
        __syncwarp();
        const int c = lane & 7, m0 = 2 * (lane >> 3);  // rows m0, m0 + 1 of the lower left block
        {  // Y = R P^-1 into the lower left block
          float y0 = 0.f, y1 = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float pk = W[k * 17 + c];
            y0 += Ab[(8 + m0) * 20 + k] * pk;
            y1 += Ab[(9 + m0) * 20 + k] * pk;
          }
          W[(8 + m0) * 17 + c] = y0;
          W[(9 + m0) * 17 + c] = y1;
        }
        __syncwarp();
        {  // X = -Q^-1 Y in its place
          float z0 = 0.f, z1 = 0.f;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float ym = W[(8 + m) * 17 + c];
            z0 += W[(8 + m0) * 17 + 8 + m] * ym;
            z1 += W[(9 + m0) * 17 + 8 + m] * ym;
          }
          __syncwarp();
          W[(8 + m0) * 17 + c] = -z0;
          W[(9 + m0) * 17 + c] = -z1;
        }
        __syncwarp();
        {  // row r = lane / 2, columns 8 (lane & 1) .. + 7 of the block into th, tw, tu
          const int r = lane >> 1, col0 = 16 * wb + 8 * (lane & 1);
          const float* wr = W + r * 17 + 8 * (lane & 1);
          uint32_t ph[4], pw[4], pu[4];
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            const float v0 = wr[j], v1 = wr[j + 1];
            const float u0 = S.beta[gb][col0 + j], u1 = S.beta[gb][col0 + j + 1];
            const float w0 = u0 * S.eG[gb][col0 + j], w1 = u1 * S.eG[gb][col0 + j + 1];
            ph[j >> 1] = pack_h2(v0, v1);
            pw[j >> 1] = pack_h2(v0 * w0, v1 * w1);
            pu[j >> 1] = pack_h2(v0 * u0, v1 * u1);
          }
          const uint32_t off = sw128_offset(64, 16 * wb + r, col0);
          *reinterpret_cast<uint4*>(S.th + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4*>(S.tw + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(S.tu + off) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
        }
      }
      named_bar(1, kPrepThreads);
      // The off-diagonal blocks by doubling: T_10 and T_32 join the 16-blocks into 32-blocks
      // (T_ab = -T_aa A_ab T_bb), then the lower left 32-block is -T_BB X with
      // X = A_BA T_AA (A = blocks 0-1, B = blocks 2-3), whose products with the diagonal
      // blocks of T_AA are started meanwhile.
      float x[2][4] = {}, x2[2][4] = {};
      const int rw = 2 + (wb >> 1);  // warps 0, 2: row block of X
      if (wb & 1) {
        mma_blk(x, ah_s, 16 * wb, 16 * (wb - 1), th_s, 16 * (wb - 1), 16 * (wb - 1));
        frag_to_xs(x, wb);
        __syncwarp();
        float y[2][4] = {};
        mma_xs(y, 16 * wb, 16 * wb, wb);
        store_t(y, wb, wb - 1, gb);
      } else {
        mma_blk(x, ah_s, 16 * rw, 0, th_s, 0, 0);      // A_r0 T_00
        mma_blk(x2, ah_s, 16 * rw, 16, th_s, 16, 16);  // X_r1 = A_r1 T_11
      }
      named_bar(1, kPrepThreads);
      if (!(wb & 1)) {
        mma_blk(x, ah_s, 16 * rw, 16, th_s, 16, 0);    // X_r0 = A_r0 T_00 + A_r1 T_10
        frag_to_xs(x, wb);                              // X_20, X_21, X_30, X_31 -> xs[0..3]
        frag_to_xs(x2, wb + 1);
      }
      named_bar(1, kPrepThreads);
      {  // warp wb: T_{r c}, r = 2 + wb / 2, c = wb % 2:  T_2c = -T_22 X_2c,
         // T_3c = -(T_32 X_2c + T_33 X_3c)
        float y[2][4] = {};
        if (rw == 3) mma_xs(y, 48, 32, wb & 1);
        mma_xs(y, 16 * rw, 16 * rw, wb);
        store_t(y, rw, wb & 1, gb);
      }
      fence_async_smem();
      arrive(S, B_T);
      named_bar(1, kPrepThreads);  // the next gram rewrites A
    };

    // ---- -w: lane i holds w[t][i] for every t; written as the MN-major tile [i][t]
    auto neg_w = [&](int ci) {
      wait_bar(S, B_WU, ci & 1);
      fence_after_sync();
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
          *reinterpret_cast<uint4*>(nw_tile(ci) + sw128_offset(128, i, 32 * hb + 8 * ch)) = pk;
        }
      }
      if (MODE == kSumU && a.wy) {  // u^T [c][t] fp16 for phase 3, in the Q rows it never loads
        uint8_t* ut = S.kq[ci & 1] + 8192 + (i >> 6) * 16384 + (i & 63) * 128;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float uv[32];
          tmem_ld32(tm + lane_bits + TM_DO + 32 * hb, uv);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 pk;
            pk.x = pack_h2(uv[8 * ch + 0], uv[8 * ch + 1]);
            pk.y = pack_h2(uv[8 * ch + 2], uv[8 * ch + 3]);
            pk.z = pack_h2(uv[8 * ch + 4], uv[8 * ch + 5]);
            pk.w = pack_h2(uv[8 * ch + 6], uv[8 * ch + 7]);
            *reinterpret_cast<uint4*>(ut + (((4 * hb + ch) ^ (i & 7)) << 4)) = pk;
          }
        }
      }
      fence_async_smem();
      fence_before_sync();
      arrive(S, B_WR);
    };

    if (MODE == kEmitR && lo_warps) {  // the factors come from the records: attn_i only
      for (int ci = 0; ci < nch; ++ci) {
        gram(ci);
        if (!named_bar_and(1, 64, !aborted(S))) break;
      }
    }
    if (MODE == kEmitR && !lo_warps) {
      // Q (bf16, rows t) -> Q^T (fp16, rows i), the MN-major operand of Q K^T and of q h.  Warp
      // 10 + b takes the features of box b, as 8 x 8 blocks (t-block tb, i-block ib): four per
      // step through ldmatrix.trans, and stmatrix to rows i, column chunk tb.
      const int box = warp - 10, m = lane >> 3, r = lane & 7;
      __nv_bfloat162 mx2 = __floats2bfloat162_rn(0.f, 0.f);
      for (int ci = 0; ci < nch; ++ci) {
        const int sg = ci & 1;
        wait_bar(S, B_L0 + sg, (ci >> 1) & 1);
        // Q K^T of the previous chunk is done, and with it [D | q h] of ci - 2, the last reader of
        // this stage's Q^T (this also keeps Q^T at most one chunk ahead of the MMA warp's wait)
        if (ci >= 1) wait_bar(S, B_SQ, (ci - 1) & 1);
        const uint32_t src = saddr(qstage(sg)) + box * 8192;
        const uint32_t dst = saddr(S.kq[sg]) + 8192 + box * 16384;
#pragma unroll 2
        for (int g = 0; g < 16; ++g) {
          const int tb = g >> 1, ib = 4 * (g & 1) + m;
          uint32_t x[4];
          ldsm_x4_t(src + (8 * tb + r) * 128 + ((ib ^ r) << 4), x);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&x[k]);
            mx2 = __hmax2(mx2, __habs2(b2));
            const float2 f = __bfloat1622float2(b2);
            x[k] = pack_h2(f.x, f.y);
          }
          stsm_x4(dst + (8 * ib + r) * 128 + ((tb ^ r) << 4), x);
        }
        fence_async_smem();  // Q^T feeds the tensor core
        fence_before_sync();
        arrive(S, B_CV);
        arrive(S, B_QF0 + sg);
        if (!named_bar_and(4, 64, !aborted(S))) break;
      }
      const float2 mx = __bfloat1622float2(mx2);
      if (!(fmaxf(mx.x, mx.y) <= kHalfMax)) S.range_bad = 1;
    }
    // one chunk ahead: the gram of chunk ci + 1 is built while w of chunk ci is computed
    bool go = MODE != kEmitR && nch > 0;
    if (go) {
      gram(0);
      go = named_bar_and(1, kPrepThreads, !aborted(S));
    }
    for (int ci = 0; go && ci < nch; ++ci) {
      solve(ci);
      if (ci + 1 < nch) gram(ci + 1);
      neg_w(ci);
      // the U half stores -w^T for the M half; the tile is rewritten two chunks later, and
      // this thread has seen its earlier copy read before the barrier of the chunk between
      if (MODE == kSumU && a.wy && pt == 0) bulk_wait_read();
      go = named_bar_and(1, kPrepThreads, !aborted(S));  // also: the gram's A is complete
      if (MODE == kSumU && a.wy && pt == 0 && go) {
        char* rec = chunk_record(a, n_seq, sb, c0 + ci, j);
        bulk_s2g(rec + kRecNw, saddr(nw_tile(ci)), 16384);
        bulk_s2g(rec + kRecU, saddr(S.kq[ci & 1]) + 8192, 8192);
        bulk_s2g(rec + kRecU + 8192, saddr(S.kq[ci & 1]) + 16384 + 8192, 8192);
      }
    }
    if (MODE == kSumU && a.wy && pt == 0) bulk_wait_all();
    }
  } else if (warp == 13) {
    // =============================================================== loader (1 warp)
    // copies issued per barrier, so that a loader that stops early still waits for them
    int nl0 = 0, nl1 = 0, nl2 = 0, nr0 = 0, nr1 = 0;
    if (MODE == kSumML) {  // the records of the U half, three stages
      for (int ci = 0; ci < nch; ++ci) {
        const int st = ci % 3;
        if (ci >= 3) wait_bar(S, B_F0 + st, ((ci / 3) + 1) & 1);
        if (__any_sync(0xffffffffu, aborted(S))) break;
        if (lane == 0) {
          const char* rec = chunk_record(a, n_seq, sb, c0 + ci, j);
          const uint32_t bar = saddr(&S.bars[B_L0 + st]);
          const uint32_t dst = saddr(rec_stage(st));
          mbar_expect_tx(bar, 32768u + kRecTblBytes);
          bulk_g2s(dst, rec + kRecNw, 16384u, bar);
          bulk_g2s(dst + 16384u, rec + kRecKh, 16384u, bar);
          bulk_g2s(saddr(S.tbl[st]), rec + kRecTbl, kRecTblBytes, bar);
        }
        nl0 += st == 0;
        nl1 += st == 1;
        nl2 += st == 2;
        __syncwarp();
      }
    }
    for (int ci = 0; MODE != kSumML && ci < nch; ++ci) {
      const int sg = ci & 1;
      // the stage was last used by chunk ci - 2: wait for its w, u (and q_g h) products, or
      // (kEmitR) for its Q, g and beta to have been read
      if (ci >= 2) wait_bar(S, (MODE == kEmitR ? B_QF0 : B_F0) + sg, ((ci >> 1) + 1) & 1);
      if (__any_sync(0xffffffffu, aborted(S))) break;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      const uint32_t bar = saddr(&S.bars[B_L0 + sg]);
      if (lane == 0) {  // rows past T read zeros; rows in [L, 64) only meet zero weights
        const uint32_t kq = saddr(S.kq[sg]), vv = saddr(S.v[sg]);
        const uint32_t bytes = MODE == kEmitR ? 2u * 8192u
                                              : (OUT ? 4u : 2u) * 8192u + (MODE != kSumM ? 2u : 0u) * 8192u;
        mbar_expect_tx(bar, bytes);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          if (MODE == kEmitR) {  // Q only: [S ; QK] takes fp16 K from the record
            tma_box(saddr(qstage(sg)) + kb * 8192, &tm_q, 64 * kb, kh, (int)t0, bar);
            continue;
          }
          tma_box(kq + kb * 16384, &tm_k, 64 * kb, kh, (int)t0, bar);
          if (OUT) tma_box(kq + kb * 16384 + 8192, &tm_q, 64 * kb, kh, (int)t0, bar);
          if (MODE != kSumM) tma_box(vv + kb * 8192, &tm_v, 64 * kb, j, (int)t0, bar);
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {  // g and beta, zero past the sequence's end
        const int t = lane + 32 * h2;
        const bool ok = t < L;
        const int64_t tt = ok ? t0 + t : sb;
        cp_async4(saddr(&S.gst[sg][0][t]), a.g + tt * a.hv + j, ok);
        cp_async4(saddr(&S.gst[sg][1][t]), a.beta + tt * a.hv + j, ok);
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar)
                   : "memory");
      nl0 += sg == 0;
      nl1 += sg == 1;
      if (MODE == kEmitR) {  // the chunk's record (-w^T, fp16 K, u^T), once Dh of ci - 2 is done
        if (ci >= 2) wait_bar(S, B_RF0 + sg, ((ci >> 1) + 1) & 1);
        if (lane == 0) {
          const char* rec = chunk_record(a, n_seq, sb, c0 + ci, j);
          const uint32_t rb = saddr(&S.bars[B_RL0 + sg]);
          mbar_expect_tx(rb, 3u * 16384u);
          bulk_g2s(saddr(S.kq[sg]), rec + kRecNw, 8192u, rb);
          bulk_g2s(saddr(S.kq[sg]) + 16384u, rec + kRecNw + 8192, 8192u, rb);
          bulk_g2s(saddr(S.kh[sg]), rec + kRecKh, 16384u, rb);
          bulk_g2s(saddr(S.v[sg]), rec + kRecU, 16384u, rb);
        }
        nr0 += sg == 0;
        nr1 += sg == 1;
        __syncwarp();
      }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    if (lane == 0) {  // every copy issued has landed before the shared memory is released
      if (nl0) wait_bar_drain(S, B_L0, (nl0 - 1) & 1);
      if (nl1) wait_bar_drain(S, B_L1, (nl1 - 1) & 1);
      if (nl2) wait_bar_drain(S, B_L2, (nl2 - 1) & 1);
      if (nr0) wait_bar_drain(S, B_RL0, (nr0 - 1) & 1);
      if (nr1) wait_bar_drain(S, B_RL1, (nr1 - 1) & 1);
    }
    __syncwarp();
  } else if (warp >= 14) {
    // =============================================================== converter (64 threads)
    const int p = tid - (kThreads - kConvThreads);  // 0..63
    float maxabs = 0.f;
    for (int ci = 0; MODE != kSumML && ci < nch; ++ci) {
      const int sg = ci & 1, gb = ci % 3;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      wait_bar(S, B_L0 + sg, (ci >> 1) & 1);
      // the decay tables are single: the previous chunk's gram must be done with them
      if (ci >= 1) wait_bar(S, B_E2, (ci - 1) & 1);
      if (p < 32) {  // within-chunk inclusive scan of g; rows >= L decay by nothing
        float x0 = S.gst[sg][0][p], x1 = S.gst[sg][0][p + 32];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
          const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
          if (p >= o) { x0 += y0; x1 += y1; }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        const float GL = L - 1 < 32 ? __shfl_sync(0xffffffffu, x0, (L - 1) & 31)
                                    : __shfl_sync(0xffffffffu, x1, (L - 1) & 31);
        // G at the last row of this lane's 16-block: rows p | 15 and (p | 15) + 32
        const float e0 = __shfl_sync(0xffffffffu, x0, p | 15);
        const float e1 = __shfl_sync(0xffffffffu, x1, p | 15);
        S.G[gb][p] = x0;
        S.G[gb][p + 32] = x1;
        S.eG[gb][p] = __expf(x0);
        S.eG[gb][p + 32] = __expf(x1);
        S.eGLG[gb][p] = __expf(GL - x0);
        S.eGLG[gb][p + 32] = __expf(GL - x1);
        S.beta[gb][p] = S.gst[sg][1][p];
        S.beta[gb][p + 32] = S.gst[sg][1][p + 32];
        S.cf[p] = __expf(e0 - x0);
        S.cf[p + 32] = __expf(e1 - x1);
        if (p == 0) S.gamma[gb] = __expf(GL);
        if (MODE == kSumU && a.wy) {  // the state update's decay, for the M half
          float* tb = reinterpret_cast<float*>(chunk_record(a, n_seq, sb, c0 + ci, j) + kRecTbl);
          tb[p] = S.eGLG[gb][p];
          tb[p + 32] = S.eGLG[gb][p + 32];
          if (p == 0) tb[64] = S.gamma[gb];
        }
      }
      // the K tile stored two chunks back has been read before it is rewritten
      if (MODE == kSumU && a.wy && p == 0) bulk_wait_read();
      if (!named_bar_and(3, kConvThreads, !aborted(S))) break;
      if (MODE == kEmitR) arrive(S, B_QF0 + sg);  // g and beta of the stage have been read
      {  // row t: its own 16-block directly, the factor to each earlier block's last row;
         // the A rows' copies carry beta_t and leave out s = t
        const int t = p, at = t >> 4, k0 = t & 15;
        const float Gt = S.G[gb][t], bt = S.beta[gb][t];
        // (the summaries read only A's tables, phase 3 from records only attn_i's)
        constexpr bool kA = MODE != kEmitR, kO = MODE == kEmit || MODE == kEmitR;
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
          float d[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) d[i] = __expf(Gt - S.G[gb][16 * at + k4 + i]);
          if (kO)
            *reinterpret_cast<float4*>(&S.ddO[t][k4]) =
                make_float4(k4 + 0 <= k0 ? d[0] : 0.f, k4 + 1 <= k0 ? d[1] : 0.f,
                            k4 + 2 <= k0 ? d[2] : 0.f, k4 + 3 <= k0 ? d[3] : 0.f);
          if (kA)
            *reinterpret_cast<float4*>(&S.ddA[t][k4]) =
                make_float4(k4 + 0 < k0 ? bt * d[0] : 0.f, k4 + 1 < k0 ? bt * d[1] : 0.f,
                            k4 + 2 < k0 ? bt * d[2] : 0.f, k4 + 3 < k0 ? bt * d[3] : 0.f);
        }
        float4 f;
        f.x = at > 0 ? __expf(Gt - S.G[gb][15]) : 0.f;
        f.y = at > 1 ? __expf(Gt - S.G[gb][31]) : 0.f;
        f.z = at > 2 ? __expf(Gt - S.G[gb][47]) : 0.f;
        f.w = 0.f;
        if (kO) *reinterpret_cast<float4*>(&S.rfO[t][0]) = f;
        if (kA)
          *reinterpret_cast<float4*>(&S.rfA[t][0]) = make_float4(bt * f.x, bt * f.y, bt * f.z, 0.f);
      }
      if (MODE == kEmit) wait_bar(S, B_SQ, ci & 1);  // [S ; QK] has read the bf16 Q
      arrive(S, B_TB);
      if (MODE != kSumM && MODE != kEmitR) {  // V -> fp16 in place (read only by the u product)
        uint8_t* vb = S.v[sg] + 16 * p;
#pragma unroll 1
        for (int k0 = 0; k0 < 16; k0 += 4)
          maxabs = to_half_chunks<4, false>(vb + 1024 * k0, vb + 1024 * k0, nullptr, maxabs);
      }
      // fp16 K into its tile, once the chunk that last used the tile has finished Dh
      if (MODE != kEmitR && ci >= 2) wait_bar(S, B_KF0 + sg, ((ci >> 1) + 1) & 1);
      if (MODE != kEmitR) {  // (kEmitR: fp16 K comes with the record)
        const uint8_t* kb = S.kq[sg] + 16 * p;
        uint8_t* kd = S.kh[sg] + 16 * p;
#pragma unroll 1
        for (int k0 = 0; k0 < 16; k0 += 4)
          maxabs = to_half_chunks<4, false>(kb + (k0 >> 3) * 16384 + 1024 * (k0 & 7),
                                            kd + (k0 >> 3) * 8192 + 1024 * (k0 & 7), nullptr, maxabs);
      }
      if (MODE == kSumU && a.wy) {  // fp16 K into the chunk's record, for the M half
        fence_async_smem();
        named_bar(3, kConvThreads);
        if (p == 0)
          bulk_s2g(chunk_record(a, n_seq, sb, c0 + ci, j) + kRecKh, saddr(S.kh[sg]), 16384);
      }
      if (MODE == kEmit) {  // q_g = diag(e^G) Q as fp16, in place: the K-major B of q_g h
        uint8_t* qb = S.kq[sg] + 8192 + 16 * p;
#pragma unroll 1
        for (int k0 = 0; k0 < 16; k0 += 4) {
          uint8_t* pq = qb + (k0 >> 3) * 16384 + 1024 * (k0 & 7);
          maxabs = to_half_chunks<4, true>(pq, pq, &S.eG[gb][(p >> 3) + 8 * (k0 & 7)], maxabs);
        }
      }
      if (MODE != kEmitR) {  // (kEmitR: the transposer hands over Q^T)
        // the MMA warp has waited for the previous chunk's hand-off
        if (ci >= 1) wait_bar(S, B_WU, (ci - 1) & 1);
        fence_async_smem();
        arrive(S, B_CV);
      }
    }
    if (!(maxabs <= kHalfMax)) S.range_bad = 1;
    if (MODE == kSumU && a.wy && p == 0) bulk_wait_all();
  } else {
    // =============================================================== MMA (warp 12)
    // Fixed order per chunk c: w, u (c); q_g h (c); D (c); O2, Dh (c); [S ; QK] (c + 2).  Every lane
    // waits, lane 0 issues and commits.
    const bool leader = lane == 0;
    const uint32_t ID_SQ = idesc_f16(128, 64, 0, 0, 1);           // bf16 [K ; Q] K^T
    const uint32_t ID_WU = idesc_f16(128, 64, 1, 0);              // K^T, V^T x T tiles
    const uint32_t ID_D = idesc_f16(128, 64, 0, 1);               // h^T (-w)^T
    const uint32_t ID_QH = idesc_f16(128, 64, 0, 0);              // h^T q_g^T
    const uint32_t ID_O2 = idesc_f16(128, 64, 0, 0);              // delta^T attn_i^T
    const uint32_t ID_DH = idesc_f16(128, 128, 0, 1);             // delta'^T K
    if (MODE == kSumML) {  // D and Dh of each loaded record
      for (int ci = 0; ci < nch; ++ci) {
        const int st = ci % 3;
        const uint32_t nw = saddr(rec_stage(st)), khs = nw + 16384u;
        wait_bar(S, B_L0 + st, (ci / 3) & 1);
        wait_bar(S, B_HR, ci & 1);
        fence_after_sync();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ts(tm + TM_DO, tm + TM_H + 64 * (ks >> 2) + 8 * (ks & 3),
                   sdesc(nw + ks * 2048, 16384, 1024), ID_D, ks > 0);
          mma_commit(saddr(&S.bars[B_D]));
        }
        __syncwarp();
        wait_bar(S, B_DR, ci & 1);
        fence_after_sync();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts(tm + TM_H, tm + TM_U + 32 * (ks >> 1) + 8 * (ks & 1),
                   sdesc(khs + ks * 2048, 8192, 1024), ID_DH, ks > 0);
          mma_commit(saddr(&S.bars[B_H]));
          mma_commit(saddr(&S.bars[B_F0 + st]));
        }
        __syncwarp();
        if (__any_sync(0xffffffffu, aborted(S))) break;
      }
    }
    auto sq = [&](int ci) {
      if (leader) {
        const uint32_t kq = saddr(S.kq[ci & 1]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t d = sdesc(kq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
          mma_ss(tm + TM_SQ, d, d, ID_SQ, ks > 0);
        }
        mma_commit(saddr(&S.bars[B_SQ]));
      }
      __syncwarp();
    };
    if (MODE != kSumML && MODE != kEmitR && nch > 0) {
      wait_bar(S, B_L0, 0);
      sq(0);
      if (nch > 1) {  // the SQ columns are reused once the first gram has read them
        wait_bar(S, B_E2, 0);
        wait_bar(S, B_L1, 0);
        sq(1);
      }
    }
    // kEmitR, per chunk c: [D | q h] (c); O2, Dh (c); Q K^T (c + 1).  Q K^T takes Q^T (MN-major
    // A; only its 64 rows t are read out) and the record's fp16 K.
    const uint32_t ID_SQR = idesc_f16(128, 64, 1, 0);   // Q K^T
    const uint32_t ID_DQ = idesc_f16(128, 128, 0, 1);   // h^T [-w^T | Q^T]
    auto sqr = [&](int ci) {
      const int st = ci & 1;
      wait_bar(S, B_CV, ci & 1);
      wait_bar(S, B_RL0 + st, (ci >> 1) & 1);
      fence_after_sync();
      if (leader) {
        const uint32_t qt = saddr(S.kq[st]) + 8192, khs = saddr(S.kh[st]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(tm + TM_SQ, sdesc(qt + (ks >> 2) * 16384 + (ks & 3) * 2048, 8192, 1024),
                 sdesc(khs + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), ID_SQR, ks > 0);
        mma_commit(saddr(&S.bars[B_SQ]));
      }
      __syncwarp();
    };
    if (MODE == kEmitR && nch > 0) sqr(0);
    for (int ci = 0; MODE == kEmitR && ci < nch; ++ci) {
      const int st = ci & 1;
      wait_bar(S, B_HR, ci & 1);  // (the record and Q^T were waited for by Q K^T)
      fence_after_sync();
      if (leader) {  // D^T (delta^T less u^T) and (q h)^T in one product
        const uint32_t b = saddr(S.kq[st]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tm + TM_DO, tm + TM_H + 64 * (ks >> 2) + 8 * (ks & 3),
                 sdesc(b + (ks >> 2) * 16384 + (ks & 3) * 2048, 8192, 1024), ID_DQ, ks > 0);
        mma_commit(saddr(&S.bars[B_D]));
      }
      __syncwarp();
      wait_bar(S, B_DR, ci & 1);
      wait_bar(S, B_E2, ci & 1);  // attn_i is written and the Q K^T columns are read
      fence_after_sync();
      if (leader) {  // (attn_i delta)^T into its own columns; then the record stage is free
        const uint32_t att = saddr(S.att[st]), khs = saddr(S.kh[st]);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t col = 32 * (ks >> 1) + 8 * (ks & 1);
          mma_ts(tm + TM_W, tm + TM_DO + col, sdesc(att + ks * 32, 16, 1024), ID_O2, ks > 0);
          mma_ts(tm + TM_H, tm + TM_U + col, sdesc(khs + ks * 2048, 8192, 1024), ID_DH, ks > 0);
        }
        mma_commit(saddr(&S.bars[B_H]));
        mma_commit(saddr(&S.bars[B_RF0 + st]));
      }
      __syncwarp();
      if (ci + 1 < nch) sqr(ci + 1);
      if (__any_sync(0xffffffffu, aborted(S))) break;
    }
    for (int ci = 0; MODE != kSumML && MODE != kEmitR && ci < nch; ++ci) {
      const uint32_t khs = saddr(S.kh[ci & 1]), vv = saddr(S.v[ci & 1]);
      // w^T = K^T T_w^T ;  u^T = V^T T_u^T; then the stage is free for the loader
      wait_bar(S, B_T, ci & 1);
      wait_bar(S, B_CV, ci & 1);
      if (leader) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ss(tm + TM_W, sdesc(khs + ks * 2048, 8192, 1024),
                 sdesc(saddr(S.tw) + ks * 32, 16, 1024), ID_WU, ks > 0);
        if (MODE != kSumM) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss(tm + TM_DO, sdesc(vv + ks * 2048, 8192, 1024),
                   sdesc(saddr(S.tu) + ks * 32, 16, 1024), ID_WU, ks > 0);
        }
        mma_commit(saddr(&S.bars[B_WU]));
        if (MODE != kEmit) mma_commit(saddr(&S.bars[B_F0 + (ci & 1)]));
      }
      __syncwarp();
      if (MODE == kEmit) {  // o^T = h^T q_g^T starts the O accumulator; then the stage is free
        wait_bar(S, B_HR, ci & 1);
        fence_after_sync();
        if (leader) {
          const uint32_t qg = saddr(S.kq[ci & 1]) + 8192;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ts(tm + TM_DO + 64, tm + TM_H + 64 * (ks >> 2) + 8 * (ks & 3),
                   sdesc(qg + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), ID_QH, ks > 0);
          mma_commit(saddr(&S.bars[B_F0 + (ci & 1)]));
        }
        __syncwarp();
      }
      // delta^T = u^T + h^T (-w)^T
      wait_bar(S, B_WR, ci & 1);
      if (MODE != kEmit) wait_bar(S, B_HR, ci & 1);
      fence_after_sync();
      if (leader) {
        const uint32_t nw = saddr(nw_tile(ci));
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tm + TM_DO, tm + TM_H + 64 * (ks >> 2) + 8 * (ks & 3),
                 sdesc(nw + ks * 2048, 16384, 1024), ID_D, MODE != kSumM || ks > 0);
        mma_commit(saddr(&S.bars[B_D]));
      }
      __syncwarp();
      // o^T += delta^T attn_i^T ;  Dh^T = delta'^T K
      wait_bar(S, B_DR, ci & 1);
      fence_after_sync();
      if (leader) {
        const uint32_t att = saddr(S.att[ci & 1]);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t col = 32 * (ks >> 1) + 8 * (ks & 1);
          if (MODE == kEmit)
            mma_ts(tm + TM_DO + 64, tm + TM_DO + col, sdesc(att + ks * 32, 16, 1024), ID_O2, 1);
          mma_ts(tm + TM_H, tm + TM_U + col, sdesc(khs + ks * 2048, 8192, 1024), ID_DH, ks > 0);
        }
        mma_commit(saddr(&S.bars[B_H]));
        mma_commit(saddr(&S.bars[B_KF0 + (ci & 1)]));
      }
      __syncwarp();
      // [S ; QK] two chunks ahead, once the gram of the next chunk has read the columns
      if (ci + 2 < nch) {
        wait_bar(S, B_E2, (ci + 1) & 1);
        wait_bar(S, B_L0 + (ci & 1), ((ci + 2) >> 1) & 1);
        sq(ci + 2);
      }
      if (__any_sync(0xffffffffu, aborted(S))) break;
    }
    // every product issued has completed before the TMEM is released
    if (leader) mma_commit(saddr(&S.bars[B_END]));
    __syncwarp();
    wait_bar_drain(S, B_END, 0);  // (also after an abort: committed products land first)
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
  CUtensorMap mk, mq, mv;
  const bool empty = a.T == 0;
  if ((e = make_map(&mk, empty || MODE == kSumML || MODE == kEmitR ? nullptr : a.k, a.T, a.hk)) !=
      cudaSuccess)
    return e;
  if ((e = make_map(&mq, empty || (MODE != kEmit && MODE != kEmitR) ? nullptr : a.q, a.T,
                    a.hk)) != cudaSuccess)
    return e;
  if ((e = make_map(&mv, empty || MODE == kSumM || MODE == kSumML || MODE == kEmitR ? nullptr : a.v,
                    a.T, a.hv)) !=
      cudaSuccess)
    return e;
  tc5_chunk_kernel<MODE><<<grid, kThreads, smem, s>>>(a, mk, mq, mv);
  return cudaGetLastError();
}

}  // namespace

size_t tc5_smem_bytes() { return sizeof(Smem) + 1024; }

// one record per (64-token window of the packed token axis, plus one per sequence, value head)
size_t tc5_records_bytes(int64_t T, int N, int hv) {
  return ((size_t)(T / C) + (size_t)N + 1) * (size_t)hv * kRecBytes;
}

// With records (a.wy), the U half runs first and stores each chunk's -w^T, fp16 K and decay,
// and the M half only loads them; without, each half computes its own factors.
cudaError_t tc5_summary(const Args& a, cudaStream_t s, cudaEvent_t mid) {
  if (a.wy) {  // the U half also runs on the last segment: phase 3 reads its records
    Args ua = a;
    ua.skip_last_summary = false;
    cudaError_t e = launch5<kSumU>(ua, s);
    if (e == cudaSuccess && mid) e = cudaEventRecord(mid, s);
    if (e != cudaSuccess) return e;
    return launch5<kSumML>(a, s);
  }
  cudaError_t e = launch5<kSumM>(a, s);
  if (e == cudaSuccess && mid) e = cudaEventRecord(mid, s);
  if (e != cudaSuccess) return e;
  return launch5<kSumU>(a, s);
}

cudaError_t tc5_emit(const Args& a, cudaStream_t s) {
  return a.wy ? launch5<kEmitR>(a, s) : launch5<kEmit>(a, s);
}

}  // namespace gdn
