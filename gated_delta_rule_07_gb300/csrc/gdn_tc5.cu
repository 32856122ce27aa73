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
//   (K, Q, V stay bf16 as loaded; where they meet a computed operand, that operand is split
//   into bf16 hi + lo parts, x = hi + lo to 2^-16, and the two products accumulate)
//   delta^T   = u^T + h^T (-w)^T                  (128 x 64, K = 128; h^T read from TMEM)
//   O1^T      = h^T Q^T                           (128 x 64, K = 128)
//   O2^T      = delta^T attn_i^T                  (128 x 64, K = 64; delta^T from TMEM)
//   Dh^T      = (diag(e^{G_last - G}) delta)^T K  (128 x 128, K = 64)
// with Q pre-scaled to q_g = diag(e^G) Q after [S ; QK], so o = O1 + O2 accumulates in one
// (double-buffered) TMEM region, and h <- gamma h + Dh.  The state h^T lives in registers
// (fp32) of the chain warps; its fp16 copy, delta and delta' are written back into TMEM as the
// A operands of the next products.  T = (I + A)^-1 is blocked by 16 x 16: the diagonal
// inverses by fp32 forward substitution in registers, the off-diagonal blocks
// T_ab = -T_aa sum_m A_am T_mb with warp-level mma.sync (fp16 operands, fp32 accumulation).
//
// Warp roles (448 threads):
//   warps 0-7  chain:   TMEM lane = state row c; warps w and w + 4 split the columns.  Besides
//                       delta and the state update they build the next chunk's decay tables
//                       and turn its q into fp16 q_g
//   warps 8-11 prepare: masked gram and attn_i, the triangular solve, -w
//   warp 12    MMA:     the whole warp waits, one thread issues every tcgen05.mma and commit
//   warp 13    loader:  TMA boxes of K, Q, V and cp.async of g, beta into the free stage
// Hand-offs use mbarriers; every wait is bounded and a wait that gives up records
// GDN_ERR_DEVICE_TIMEOUT, and all roles leave their loops (group decisions are made uniform
// with barrier reductions) so the CTA always reaches its TMEM release.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"
#include "gdn_warp_mma.cuh"

namespace gdn {
namespace {

using namespace sm100;
using namespace warp_mma;

constexpr int C = kChunk;  // 64
constexpr int KD = 128, VD = 128;
constexpr int kChainThreads = 256, kPrepThreads = 128;
constexpr int kThreads = kChainThreads + kPrepThreads + 64;  // + MMA warp + loader warp
constexpr uint32_t kWaitLimit = 1u << 24;  // polls of ~40-100 ns: a second or more
constexpr float kHalfMax = 65504.f;

enum Mode { kEmit = 0, kSumM = 1, kSumU = 2 };

// TMEM columns (512 allocated)
constexpr uint32_t TM_SQ = 0;    // [S ; QK]          64 fp32
constexpr uint32_t TM_W = 64;    // w^T               64 fp32
constexpr uint32_t TM_U = 128;   // u^T -> delta^T    64 fp32, then fp16 delta / delta'
constexpr uint32_t TM_O = 192;   // o^T, two buffers  2 x 64 fp32 (chunk parity)
constexpr uint32_t TM_DL = 320;  // lo part of delta'  32 bf16 pairs
constexpr uint32_t TM_H = 384;   // Dh^T              128 fp32, then fp16 h^T

// mbarriers
enum Bar { B_SQ = 0, B_T, B_WU, B_WR, B_HR, B_D, B_DR, B_H, B_L0, B_L1, B_QS, kNumBars };

struct Smem {
  uint8_t kq[2][2 * 128 * 128];  // per stage: [kblk][128 rows: K 0-63, Q 64-127][128 B]
  uint8_t v[2][2 * 64 * 128];    // per stage: [kblk][64 rows][128 B]
  uint8_t att[2][64 * 128];      // attn_i [t][s], K-major B
  uint8_t twh[64 * 128];         // T diag(beta e^G) [t][s], K-major B, bf16 hi part
  uint8_t twl[64 * 128];         //   ... and lo part
  uint8_t tuh[64 * 128];         // T diag(beta) [t][s], K-major B, bf16 hi part
  uint8_t tul[64 * 128];         //   ... and lo part
  uint8_t nw[128 * 128];         // -w [i][t], MN-major B
  uint8_t ah[64 * 128];          // masked gram A [t][s], fp16
  uint8_t th[64 * 128];          // blocks of (I + A)^-1 [t][s], fp16 operands
  uint8_t xs[4][16 * 48];        // per-warp 16 x 16 fp16 scratch, 48-byte rows
  float adiag[C][16];            // the diagonal 16 x 16 blocks of A, fp32
  float gst[2][2][C];            // g and beta of a staged chunk
  float G[3][C], eG[3][C], eGLG[3][C], beta[3][C], gamma[3];
  alignas(16) float dec[C * C];  // e^{G_t - G_s} for s <= t, else 0; 16-byte chunks swizzled
  float qsc[C];                  // e^{G_t} of the chunk whose q the chain warps scale
  uint64_t bars[kNumBars];
  uint32_t tmem_base;
  int abort_flag;
  int range_bad;
};

// Members read or written with 16-byte vector accesses, ldmatrix or the tensor core must sit on
// 16-byte (swizzled tiles: 1024-byte) boundaries of the 1024-aligned base.
static_assert(offsetof(Smem, kq) % 1024 == 0 && offsetof(Smem, v) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, att) % 1024 == 0 && offsetof(Smem, twh) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, twl) % 1024 == 0 && offsetof(Smem, tuh) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, tul) % 1024 == 0 && offsetof(Smem, nw) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, ah) % 1024 == 0 && offsetof(Smem, th) % 1024 == 0, "tile alignment");
static_assert(offsetof(Smem, xs) % 16 == 0 && offsetof(Smem, dec) % 16 == 0, "vector alignment");
static_assert(offsetof(Smem, bars) % 8 == 0, "mbarrier alignment");
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory per block");

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
// Warp-uniform bounded wait; `spin` busy-polls (for the MMA warp, whose wake-up delays every
// product behind it).
__device__ __forceinline__ bool warp_wait(Smem& S, int bar, uint32_t parity, bool spin = false) {
  bool ok = !aborted(S) && (spin ? mbar_spin(saddr(&S.bars[bar]), parity, 1u << 28)
                                 : mbar_wait(saddr(&S.bars[bar]), parity, kWaitLimit));
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) set_abort(S);
  return ok;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ bool fits_half(float x) { return fabsf(x) <= kHalfMax; }

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): products with a bf16 operand keep ~16 bits.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ void st_hilo(uint8_t* hi_tile, uint8_t* lo_tile, int r, int c,
                                        float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const uint32_t off = sw128_offset(64, r, c);
  *reinterpret_cast<__nv_bfloat16*>(hi_tile + off) = h;
  *reinterpret_cast<__nv_bfloat16*>(lo_tile + off) = __float2bfloat16_rn(x - __bfloat162float(h));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
// One 64 x 64 box of a [T, heads, 128] bf16 tensor (128-byte swizzle) into shared memory;
// completion is counted in bytes on the mbarrier.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int head,
                                        int t0, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(head), "r"(t0), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile(
      "{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
          mbar),
      "r"(bytes)
      : "memory");
}

// Position of element (t, s) of the 64 x 64 fp32 decay matrix: 16-byte chunks of a row are
// XOR-permuted by (t & 15) so that a warp reading 32 rows at one column is conflict-free.
__device__ __forceinline__ int dec_idx(int t, int s) {
  return t * 64 + ((((s >> 2) ^ (t & 15))) << 2) + (s & 3);
}

__device__ __forceinline__ void st_half(uint8_t* tile, int r, int c, float x) {
  *reinterpret_cast<__half*>(tile + sw128_offset(64, r, c)) = __float2half_rn(x);
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
__global__ void __launch_bounds__(kThreads, 1)
    tc5_chunk_kernel(Args a, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_v) {
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
    for (int b = 0; b < kNumBars; ++b)  // loads: the byte count plus 32 cp.async arrivals
      mbar_init(saddr(&S.bars[b]), (b == B_L0 || b == B_L1) ? 33 : 1);
    S.abort_flag = 0;
    S.range_bad = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 12) {
    tmem_alloc(saddr(&S.tmem_base), 512);
    tmem_relinquish();
  }
  if (tid == kChainThreads) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    if (MODE == kEmit)
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    if (MODE != kSumM)
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
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
    // q (bf16) -> q_g = e^{G_t} q (fp16) of chunk ci, in place, after [S ; QK] has read q
    auto scale_q = [&](int ci) -> bool {
      const int sg = ci & 1;
      if (!group_wait(S, B_SQ, ci & 1, 2, kChainThreads)) return false;
      if (warp == 0) {  // e^{G_t} of chunk ci from its staged g (rows past the end are 0)
        float x0 = S.gst[sg][0][lane], x1 = S.gst[sg][0][lane + 32];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
          const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
          if (lane >= o) { x0 += y0; x1 += y1; }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        S.qsc[lane] = __expf(x0);
        S.qsc[lane + 32] = __expf(x1);
      }
      named_bar(2, kChainThreads);
      {
        const int t = tid >> 2, c0q = 4 * (tid & 3);  // row t, four 16-byte chunks
        const float sc = S.qsc[t];
        uint4* pq[4];
        uint4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          pq[u] = reinterpret_cast<uint4*>(S.kq[sg] + sw128_offset(128, 64 + t, 8 * (c0q + u)));
          x[u] = *pq[u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t* w = reinterpret_cast<uint32_t*>(&x[u]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
            range_ok = range_ok && fits_half(f.x * sc) && fits_half(f.y * sc);
            w[i] = pack_h2(f.x * sc, f.y * sc);
          }
          *pq[u] = x[u];
        }
      }
      fence_async_smem();
      named_bar(2, kChainThreads);
      if (tid == 0) mbar_arrive(saddr(&S.bars[B_QS]));
      return true;
    };
    bool go = nch > 0;
    if (go && MODE == kEmit) go = scale_q(0);
    if (go) {
      publish_h();
      fence_before_sync();
      named_bar(2, kChainThreads);
      if (tid == 0) mbar_arrive(saddr(&S.bars[B_HR]));
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    for (int ci = 0; go && ci < nch; ++ci) {
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
        {  // delta' = e^{G_last - G_t} delta as bf16 hi + lo (it meets bf16 K)
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int t = 32 * hf + 2 * q;
            split_bf16(d0[2 * q] * S.eGLG[gb][t], d0[2 * q + 1] * S.eGLG[gb][t + 1], ph[q], pl[q]);
            split_bf16(d1[2 * q] * S.eGLG[gb][t + 16], d1[2 * q + 1] * S.eGLG[gb][t + 17],
                       ph[q + 8], pl[q + 8]);
          }
          tmem_st16(tm + lane_bits + TM_U + 32 * hf + 16, ph);
          tmem_st16(tm + lane_bits + TM_DL + 16 * hf, pl);
        }
      }
      fence_before_sync();
      named_bar(2, kChainThreads);
      if (tid == 0) mbar_arrive(saddr(&S.bars[B_DR]));

      // ---- the state update first (it gates the next chunk), the outputs after it
      if (!group_wait(S, B_H, ci & 1, 2, kChainThreads)) break;
      fence_after_sync();
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
      if (ci + 1 < nch) publish_h();
      fence_before_sync();
      named_bar(2, kChainThreads);
      if (tid == 0 && ci + 1 < nch) mbar_arrive(saddr(&S.bars[B_HR]));
      if (MODE == kEmit) {
        // o^T buffer ci & 1 is rewritten only after the next chunk's state hand-off
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          float o[16];
          tmem_ld16(tm + lane_bits + TM_O + 64 * (ci & 1) + 32 * hf + 16 * piece, o);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int t = 32 * hf + 16 * piece + q;
            if (t < L) out[((t0 + t) * a.hv + j) * VD + c] = __float2bfloat16_rn(o[q]);
          }
        }
      }
      if (MODE == kEmit && ci + 1 < nch && !scale_q(ci + 1)) break;
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
    const int wb = warp - 8;                  // 0..3: this warp's 16-row block of T
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    const int g8 = lane >> 2, q4 = lane & 3;
    bool range_ok = true;
    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(a.v);
    const uint32_t ah_s = saddr(S.ah), th_s = saddr(S.th), xs_s = saddr(S.xs[wb]);

    // the strictly upper blocks of T diag(.) are zero for every chunk
    for (int e = pt; e < 64 * 128 / 16; e += kPrepThreads) {
      reinterpret_cast<uint4*>(S.twh)[e] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(S.twl)[e] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(S.tuh)[e] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(S.tul)[e] = make_uint4(0u, 0u, 0u, 0u);
    }

    // decay tables and the decay matrix of chunk ci (g, beta staged by the loader)
    auto tables = [&](int ci) -> bool {
      const int sg = ci & 1, gb = ci % 3;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      if (!group_wait(S, B_L0 + sg, (ci >> 1) & 1, 1, kPrepThreads)) return false;
      if (pt < 32) {  // within-chunk inclusive scan of g; rows >= L decay by nothing
        float x0 = S.gst[sg][0][pt], x1 = S.gst[sg][0][pt + 32];
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
        S.eG[gb][pt] = __expf(x0);
        S.eG[gb][pt + 32] = __expf(x1);
        S.eGLG[gb][pt] = __expf(GL - x0);
        S.eGLG[gb][pt + 32] = __expf(GL - x1);
        S.beta[gb][pt] = S.gst[sg][1][pt];
        S.beta[gb][pt + 32] = S.gst[sg][1][pt + 32];
        if (pt == 0) S.gamma[gb] = __expf(GL);
      }
      named_bar(1, kPrepThreads);
      {  // the decay matrix: row t, columns 32 (pt >> 6) .. + 31
        const int t = pt & 63, s0 = 32 * (pt >> 6);
        const float Gt = S.G[gb][t];
#pragma unroll
        for (int c4 = 0; c4 < 32; c4 += 4) {
          float4 d;
          const int s1 = s0 + c4;
          d.x = s1 <= t ? __expf(Gt - S.G[gb][s1]) : 0.f;
          d.y = s1 + 1 <= t ? __expf(Gt - S.G[gb][s1 + 1]) : 0.f;
          d.z = s1 + 2 <= t ? __expf(Gt - S.G[gb][s1 + 2]) : 0.f;
          d.w = s1 + 3 <= t ? __expf(Gt - S.G[gb][s1 + 3]) : 0.f;
          *reinterpret_cast<float4*>(&S.dec[dec_idx(t, s1)]) = d;
        }
      }
      named_bar(1, kPrepThreads);
      return true;
    };

    // T_ab = -T_aa sum_{m=b}^{a-1} A_am T_mb for one 16 x 16 block, by one warp: the sum on
    // mma.sync from the fp16 tiles, then the product with T_aa through the warp's scratch.
    auto off_diag_block = [&](int ab, int bb, int gb) {
      float x[2][4] = {};
      for (int m = bb; m < ab; ++m) {
        uint32_t af[4], bf[4];
        load_a<64>(ah_s, 16 * ab, 16 * m, af);
        load_b_kn<64>(th_s, 16 * m, 16 * bb, bf);
        mma16816(x[0], af, bf[0], bf[1]);
        mma16816(x[1], af, bf[2], bf[3]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<uint32_t*>(S.xs[wb] + g8 * 48 + (8 * nt + 2 * q4) * 2) =
            pack_h2(x[nt][0], x[nt][1]);
        *reinterpret_cast<uint32_t*>(S.xs[wb] + (g8 + 8) * 48 + (8 * nt + 2 * q4) * 2) =
            pack_h2(x[nt][2], x[nt][3]);
      }
      __syncwarp();
      float y[2][4] = {};
      {
        uint32_t af[4], bf[4];
        load_a<64>(th_s, 16 * ab, 16 * ab, af);
        const int mi = lane >> 3, rr = lane & 7;
        ldsm_x4_t(xs_s + (rr + ((mi & 1) << 3)) * 48 + ((mi >> 1) << 3) * 2, bf);
        mma16816(y[0], af, bf[0], bf[1]);
        mma16816(y[1], af, bf[2], bf[3]);
      }
      __syncwarp();
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
          uint32_t hi, lo;
          split_bf16(v0 * w0, v1 * w1, hi, lo);
          *reinterpret_cast<uint32_t*>(S.twh + off) = hi;
          *reinterpret_cast<uint32_t*>(S.twl + off) = lo;
          split_bf16(v0 * u0, v1 * u1, hi, lo);
          *reinterpret_cast<uint32_t*>(S.tuh + off) = hi;
          *reinterpret_cast<uint32_t*>(S.tul + off) = lo;
          range_ok = range_ok && fits_half(v0) && fits_half(v1);
        }
    };

    for (int ci = 0; ci < nch; ++ci) {
      const int gb = ci % 3;
      if (ci == 0 && !tables(0)) break;
      // ---- masked gram A and attn_i from [S ; QK]
      if (!group_wait(S, B_SQ, ci & 1, 1, kPrepThreads)) break;
      fence_after_sync();
      {
        const bool is_s = pt < 64;
        const int t = pt & 63, ab = t >> 4;
        const float bt = is_s ? S.beta[gb][t] : 1.f;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float sv[32];
          tmem_ld32(tm + lane_bits + TM_SQ + 32 * hb, sv);
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4) {
            const int s1 = 32 * hb + c4;
            const float4 d = *reinterpret_cast<const float4*>(&S.dec[dec_idx(t, s1)]);
            // A keeps s < t (times beta_t); attn_i keeps s <= t (the matrix is 0 above)
            sv[c4 + 0] *= bt * (is_s && s1 + 0 == t ? 0.f : d.x);
            sv[c4 + 1] *= bt * (is_s && s1 + 1 == t ? 0.f : d.y);
            sv[c4 + 2] *= bt * (is_s && s1 + 2 == t ? 0.f : d.z);
            sv[c4 + 3] *= bt * (is_s && s1 + 3 == t ? 0.f : d.w);
          }
          if (is_s) {
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if (((32 * hb + q) >> 4) == ab) S.adiag[t][q & 15] = sv[q];
          }
          if (is_s || MODE == kEmit) {
            uint8_t* dst = is_s ? S.ah : S.att[ci & 1];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              uint4 pk;
              pk.x = pack_h2(sv[8 * ch + 0], sv[8 * ch + 1]);
              pk.y = pack_h2(sv[8 * ch + 2], sv[8 * ch + 3]);
              pk.z = pack_h2(sv[8 * ch + 4], sv[8 * ch + 5]);
              pk.w = pack_h2(sv[8 * ch + 6], sv[8 * ch + 7]);
              *reinterpret_cast<uint4*>(dst + sw128_offset(64, t, 32 * hb + 8 * ch)) = pk;
            }
          }
        }
        if (MODE == kEmit && !is_s) fence_async_smem();  // attn_i feeds the tensor core
      }
      fence_before_sync();
      named_bar(1, kPrepThreads);
      // ---- T = (I + A)^-1.  Diagonal block wb by forward substitution in registers:
      // lane (c, rh) holds rows 8 rh .. 8 rh + 7 of column c of the block inverse.
      {
        const int c = lane & 15, rh = lane >> 4;
        const float* Ab = &S.adiag[16 * wb][0];
        float tc[8];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) tc[k2] = (8 * rh + k2 == c) ? 1.f : 0.f;
        if (rh == 0) {
#pragma unroll
          for (int rr = 1; rr < 8; ++rr) {
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < rr; ++s2) {
              if (s2 & 1) x1 += Ab[rr * 16 + s2] * tc[s2];
              else x0 += Ab[rr * 16 + s2] * tc[s2];
            }
            if (rr > c) tc[rr] = -(x0 + x1);
          }
        }
        float y[8];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) y[k2] = __shfl_sync(0xffffffffu, tc[k2], c);
        if (rh == 1) {
#pragma unroll
          for (int rr = 8; rr < 16; ++rr) {
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < 8; ++s2) {
              if (s2 & 1) x1 += Ab[rr * 16 + s2] * y[s2];
              else x0 += Ab[rr * 16 + s2] * y[s2];
            }
#pragma unroll
            for (int s2 = 8; s2 < rr; ++s2) {
              if (s2 & 1) x1 += Ab[rr * 16 + s2] * tc[s2 - 8];
              else x0 += Ab[rr * 16 + s2] * tc[s2 - 8];
            }
            if (rr > c) tc[rr - 8] = -(x0 + x1);
          }
        }
        const int col = 16 * wb + c;
        const float u = S.beta[gb][col], w = u * S.eG[gb][col];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
          const int row = 16 * wb + 8 * rh + k2;
          st_half(S.th, row, col, tc[k2]);
          st_hilo(S.twh, S.twl, row, col, tc[k2] * w);
          st_hilo(S.tuh, S.tul, row, col, tc[k2] * u);
        }
      }
      named_bar(1, kPrepThreads);
      if (wb < 3) off_diag_block(wb + 1, wb, gb);
      named_bar(1, kPrepThreads);
      if (wb < 2) off_diag_block(wb + 2, wb, gb);
      named_bar(1, kPrepThreads);
      if (wb == 0) off_diag_block(3, 0, gb);
      fence_async_smem();
      named_bar(1, kPrepThreads);
      if (pt == 0) mbar_arrive(saddr(&S.bars[B_T]));
      // ---- while w and u are computed: the next chunk's decay tables (E2 of this chunk,
      // the only reader of the decay matrix, is done)
      if (ci + 1 < nch && !tables(ci + 1)) break;
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
    }
    if (!range_ok) S.range_bad = 1;
  } else if (warp == 13) {
    // =============================================================== loader (1 warp)
    for (int ci = 0; ci < nch; ++ci) {
      const int sg = ci & 1;
      // the stage was last used by chunk ci - 2: wait for its last MMA
      if (ci >= 2 && !warp_wait(S, B_H, (ci - 2) & 1)) break;
      const int64_t t0 = sb + (c0 + ci) * C;
      const int L = (int)((se - t0) < C ? (se - t0) : C);
      const uint32_t bar = saddr(&S.bars[B_L0 + sg]);
      if (lane == 0) {  // rows past T read zeros; rows in [L, 64) only meet zero weights
        const uint32_t kq = saddr(S.kq[sg]), vv = saddr(S.v[sg]);
        const uint32_t bytes =
            (MODE == kEmit ? 4u : 2u) * 8192u + (MODE != kSumM ? 2u : 0u) * 8192u;
        mbar_expect_tx(bar, bytes);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          tma_box(kq + kb * 16384, &tm_k, 64 * kb, kh, (int)t0, bar);
          if (MODE == kEmit) tma_box(kq + kb * 16384 + 8192, &tm_q, 64 * kb, kh, (int)t0, bar);
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
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
  } else {
    // =============================================================== MMA (warp 12)
    // every lane waits; lane 0 issues the MMAs and commits
    const bool leader = lane == 0;
    const uint32_t ID_SQ = idesc_f16(128, 64, 0, 0, 1);     // bf16 [K ; Q] K^T
    const uint32_t ID_WU = idesc_f16(128, 64, 1, 0, 1);     // bf16 K^T, V^T x T parts
    const uint32_t ID_D = idesc_f16(128, 64, 0, 1);         // fp16 h^T (-w)^T
    const uint32_t ID_O = idesc_f16(128, 64, 0, 0);         // fp16 h^T q_g^T, delta^T attn^T
    const uint32_t ID_DH = idesc_f16(128, 128, 0, 1, 1);    // bf16 delta'^T K
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
    auto wu = [&](int ci) {
      if (leader) {
        const uint32_t kq = saddr(S.kq[ci & 1]), vv = saddr(S.v[ci & 1]);
        const uint32_t tiles_w[2] = {saddr(S.twh), saddr(S.twl)};
        const uint32_t tiles_u[2] = {saddr(S.tuh), saddr(S.tul)};
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss(tm + TM_W, sdesc(kq + ks * 2048, 16384, 1024),
                   sdesc(tiles_w[part] + ks * 32, 16, 1024), ID_WU, part > 0 || ks > 0);
        if (MODE != kSumM) {
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ss(tm + TM_U, sdesc(vv + ks * 2048, 8192, 1024),
                     sdesc(tiles_u[part] + ks * 32, 16, 1024), ID_WU, part > 0 || ks > 0);
        }
        mma_commit(saddr(&S.bars[B_WU]));
      }
      __syncwarp();
    };
    if (nch > 0) {
      bool ok = warp_wait(S, B_L0, 0, true);
      if (ok) sq(0);
      ok = ok && warp_wait(S, B_T, 0, true);
      if (ok) wu(0);
      for (int ci = 0; ok && ci < nch; ++ci) {
        const uint32_t kq = saddr(S.kq[ci & 1]);
        // delta^T (+)= h^T (-w)^T ;  o^T = h^T q_g^T
        ok = warp_wait(S, B_WR, ci & 1, true) && warp_wait(S, B_HR, ci & 1, true) &&
             (MODE != kEmit || warp_wait(S, B_QS, ci & 1, true));
        if (!ok) break;
        fence_after_sync();
        if (leader) {
          const uint32_t nw = saddr(S.nw);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t ah = tm + TM_H + 64 * (ks >> 2) + 8 * (ks & 3);
            mma_ts(tm + TM_U, ah, sdesc(nw + ks * 2048, 16384, 1024), ID_D,
                   (MODE != kSumM) || ks > 0);
            if (MODE == kEmit)
              mma_ts(tm + TM_O + 64 * (ci & 1), ah,
                     sdesc(kq + (ks >> 2) * 16384 + 64 * 128 + (ks & 3) * 32, 16, 1024), ID_O,
                     ks > 0);
          }
          mma_commit(saddr(&S.bars[B_D]));
        }
        __syncwarp();
        // the next chunk's [S ; QK] as soon as its data is in (R_sq was read before T)
        if (ci + 1 < nch) {
          ok = warp_wait(S, B_L0 + ((ci + 1) & 1), ((ci + 1) >> 1) & 1, true);
          if (!ok) break;
          sq(ci + 1);
        }
        // o^T += delta^T attn_i^T ;  Dh^T = delta'^T K  (delta' as hi + lo)
        ok = warp_wait(S, B_DR, ci & 1, true);
        if (!ok) break;
        fence_after_sync();
        if (leader) {
          const uint32_t att = saddr(S.att[ci & 1]);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t col = TM_U + 32 * (ks >> 1) + 8 * (ks & 1);
            if (MODE == kEmit)
              mma_ts(tm + TM_O + 64 * (ci & 1), tm + col, sdesc(att + ks * 32, 16, 1024), ID_O,
                     1);
            const uint64_t bk = sdesc(kq + ks * 2048, 16384, 1024);
            mma_ts(tm + TM_H, tm + col + 16, bk, ID_DH, ks > 0);
            mma_ts(tm + TM_H, tm + TM_DL + 16 * (ks >> 1) + 8 * (ks & 1), bk, ID_DH, 1);
          }
          mma_commit(saddr(&S.bars[B_H]));
        }
        __syncwarp();
        if (ci + 1 < nch) {
          ok = warp_wait(S, B_T, (ci + 1) & 1, true);
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

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against libcuda).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// [T, heads, 128] bf16 tensor read as 64 (features) x 1 (head) x 64 (tokens) boxes with the
// 128-byte swizzle; tokens past T read as zeros.
cudaError_t make_map(CUtensorMap* m, const void* base, int64_t T, int heads) {
  EncodeTiled fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)(T > 0 ? T : 1)};
  const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  static const uint16_t dummy[64] __attribute__((aligned(16))) = {};
  void* addr = const_cast<void*>(base ? base : static_cast<const void*>(dummy));
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, addr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
  if ((e = make_map(&mk, empty ? nullptr : a.k, a.T, a.hk)) != cudaSuccess) return e;
  if ((e = make_map(&mq, empty || MODE != kEmit ? nullptr : a.q, a.T, a.hk)) != cudaSuccess)
    return e;
  if ((e = make_map(&mv, empty || MODE == kSumM ? nullptr : a.v, a.T, a.hv)) != cudaSuccess)
    return e;
  tc5_chunk_kernel<MODE><<<grid, kThreads, smem, s>>>(a, mk, mq, mv);
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
