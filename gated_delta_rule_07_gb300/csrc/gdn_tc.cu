// gdn_tc.cu -- tensor-core kernels (bf16 operands, fp32 accumulation, fp32 state) for the
// chunked gated delta rule forward with K = V = 128 and C = 64.
//
// One CTA owns one (segment, value head) and walks the segment's chunks in order.  The
// K x V state (or, in phase 1, one half of X = [M | U]) lives in registers as fp32 MMA
// accumulators: warp w holds state rows [16w, 16w + 16) across all 128 columns.  Per
// chunk ("Add context parallelism to the Gated Delta Net", sections "Why" and
// "Implementation"):
//   prepare  S = K K^T, A = mask(beta_t e^{G_t - G_s} S) (s < t), T = (I + A)^-1 (blocked
//            forward substitution in fp32), w = T diag(beta e^G) K, u = T diag(beta) V
//   chain    delta = u - w h, h <- gamma h + K^T diag(e^{G_last - G}) delta
//   emit     o = diag(e^G) Q h + attn_i delta, attn_i = mask(e^{G_t - G_s} Q K^T) (s <= t)
//   phase 1  the same chain on X = [M | U] from [I | 0] (u = 0 for the M half), which is the
//            low-rank composition M <- gamma M - k_tilde^T (w M).
// Every decay factor is applied elementwise with a non-positive exponent.
//
// MMA operands are fp16 (11-bit significand): the bf16 inputs are converted in shared memory
// (exact for |x| >= 2^-14, and below that the absolute error is < 2^-25), and the computed
// operands (T, w, the state copy, delta, attn_i) keep 8x the precision bf16 would.  The bf16
// output rounding alone costs up to 2^-9 max|o|, so the inner operands must be finer than
// bf16 to keep max|err| / rms(o) inside 2e-2.  A value outside the fp16 range is reported
// as GDN_ERR_DEVICE_RANGE.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_warp_mma.cuh"

namespace gdn {
namespace {

using namespace warp_mma;

constexpr int C = kChunk;  // 64
constexpr int KD = 128;
constexpr int VD = 128;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int FP = C + 1;  // fp32 row pitch of the 64 x 64 solve buffers

enum Mode { kEmit = 0, kSumM = 1, kSumU = 2 };

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // src-size 0 zero-fills the 16 bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

constexpr float kHalfMax = 65504.f;

// Converts, in place, the 16-byte chunk at p from 8 bf16 to 8 fp16; returns false when a
// value does not fit the fp16 range.
__device__ __forceinline__ bool bf16_chunk_to_f16(char* p) {
  uint4 x = *reinterpret_cast<uint4*>(p);
  uint32_t* w = reinterpret_cast<uint32_t*>(&x);
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
    ok = ok && fabsf(f.x) <= kHalfMax && fabsf(f.y) <= kHalfMax;
    w[i] = pack_h2(f.x, f.y);
  }
  *reinterpret_cast<uint4*>(p) = x;
  return ok;
}

// ------------------------------------------------------------ swizzled bf16 tiles
//
// A tile is `rows` x RL 16-bit values (fp16), row-major, with the 16-byte chunks of each row XOR-permuted by
// (row & 7) so that the eight row addresses of an ldmatrix hit eight different bank groups.

// Stores the accumulator of an m16n8 tile at (m0, n0) as fp16, row g scaled by s0 and row
// g + 8 by s1.  Returns false when a stored value overflows the fp16 range.
template <int RL>
__device__ __forceinline__ bool store_acc_h(char* base, int m0, int n0, const float (&d)[4],
                                            float s0, float s1) {
  const int l = threadIdx.x & 31, g = l >> 2, q = l & 3;
  const int r0 = m0 + g, r1 = m0 + g + 8;
  const float a = d[0] * s0, b = d[1] * s0, c = d[2] * s1, e = d[3] * s1;
  *reinterpret_cast<uint32_t*>(base + tile_off<RL>(r0, n0) + 4 * q) = pack_h2(a, b);
  *reinterpret_cast<uint32_t*>(base + tile_off<RL>(r1, n0) + 4 * q) = pack_h2(c, e);
  return fmaxf(fmaxf(fabsf(a), fabsf(b)), fmaxf(fabsf(c), fabsf(e))) <= kHalfMax;
}

// ------------------------------------------------------------ shared memory plan

struct Smem {
  __half q[C * KD];    // [t][i]
  __half k[C * KD];    // [t][i]
  __half v[C * VD];    // [t][c]
  __half nw[C * KD];   // -w  [t][i]
  __half h[KD * VD];   // state as an operand [i][c]
  __half d[C * VD];    // delta [t][c]
  __half dp[C * VD];   // diag(e^{G_last - G_t}) delta [t][c]
  __half att[C * C];   // attn_i [t][s]
  __half tw[C * C];    // T diag(beta e^G) [t][s]
  __half tu[C * C];    // T diag(beta) [t][s]
  float A[C * FP];            // masked gram, fp32
  float Ti[C * FP];           // (I + A)^-1, fp32
  float X[C * FP];            // solve scratch
  float G[C];                 // inclusive cumulative log decay
  float beta[C];
};

// ------------------------------------------------------------ the chunk loop

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) tc_chunk_kernel(Args a) {
  extern __shared__ __align__(128) char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, q4 = lane & 3;
  const int seg = blockIdx.x, j = blockIdx.y;
  const int n = seg / a.P, r = seg % a.P;
  if (MODE != kEmit && r == a.P - 1 && a.skip_last_summary) return;  // not needed by the scan
  const int kh = j / (a.hv / a.hk);
  int64_t sb, se;
  if (!seq_bounds(a.cu, n, a.T, a.status, sb, se)) return;
  int64_t c0, c1;
  segment_chunks(se - sb, a.P, r, c0, c1);

  const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(a.v);
  __nv_bfloat16* gout = static_cast<__nv_bfloat16*>(a.out);

  const uint32_t sq = smem_addr(S.q), sk = smem_addr(S.k), sv = smem_addr(S.v);
  const uint32_t snw = smem_addr(S.nw), shh = smem_addr(S.h), sd = smem_addr(S.d);
  const uint32_t sdp = smem_addr(S.dp), satt = smem_addr(S.att);
  const uint32_t stw = smem_addr(S.tw), stu = smem_addr(S.tu);

  bool range_ok = true;  // every fp16 operand stayed finite

  // ---- the state: rows [16 warp, +16), all 128 columns, as 16 m16n8 accumulators
  float hacc[16][4];
  {
    const float* src = nullptr;
    if (MODE == kEmit) src = a.h_in ? a.h_in + ((int64_t)seg * a.hv + j) * KD * VD : nullptr;
    for (int nt = 0; nt < 16; ++nt)
      for (int e = 0; e < 4; ++e) {
        const int i = warp * 16 + g8 + ((e >> 1) << 3), c = nt * 8 + 2 * q4 + (e & 1);
        float x = 0.f;
        if (MODE == kEmit) x = src ? src[i * VD + c] : 0.f;
        if (MODE == kSumM) x = (i == c) ? 1.f : 0.f;
        hacc[nt][e] = x;
      }
  }

  for (int64_t ch = c0; ch < c1; ++ch) {
    const int64_t t0 = sb + ch * C;
    const int L = (int)((se - t0) < C ? (se - t0) : C);

    // ---- (0) publish the state as a bf16 operand; stage q, k, v, g, beta
    __syncthreads();  // previous chunk finished reading every buffer
    for (int nt = 0; nt < 16; ++nt)
      range_ok &= store_acc_h<VD>(reinterpret_cast<char*>(S.h), warp * 16, nt * 8, hacc[nt], 1.f,
                                  1.f);
    for (int e = tid; e < C * 16; e += kThreads) {
      const int t = e >> 4, cc = (e & 15) << 3;
      const bool ok = t < L;
      const int64_t tt = ok ? t0 + t : sb;
      cp_async16(sk + tile_off<KD>(t, cc), gk + (tt * a.hk + kh) * KD + cc, ok);
      if (MODE == kEmit) cp_async16(sq + tile_off<KD>(t, cc), gq + (tt * a.hk + kh) * KD + cc, ok);
      if (MODE != kSumM) cp_async16(sv + tile_off<VD>(t, cc), gv + (tt * a.hv + j) * VD + cc, ok);
    }
    if (warp == 0) {  // inclusive scan of g over the chunk (rows >= L decay by 0)
      float x0 = lane < L ? a.g[(t0 + lane) * a.hv + j] : 0.f;
      float x1 = lane + 32 < L ? a.g[(t0 + lane + 32) * a.hv + j] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
        const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (lane >= o) { x0 += y0; x1 += y1; }
      }
      x1 += __shfl_sync(0xffffffffu, x0, 31);
      S.G[lane] = x0;
      S.G[lane + 32] = x1;
      S.beta[lane] = lane < L ? a.beta[(t0 + lane) * a.hv + j] : 0.f;
      S.beta[lane + 32] = lane + 32 < L ? a.beta[(t0 + lane + 32) * a.hv + j] : 0.f;
    }
    cp_async_wait_all();
    // bf16 -> fp16 in place, each thread on the chunks it copied
    for (int e = tid; e < C * 16; e += kThreads) {
      const int t = e >> 4, cc = (e & 15) << 3;
      range_ok &= bf16_chunk_to_f16(reinterpret_cast<char*>(S.k) + tile_off<KD>(t, cc));
      if (MODE == kEmit)
        range_ok &= bf16_chunk_to_f16(reinterpret_cast<char*>(S.q) + tile_off<KD>(t, cc));
      if (MODE != kSumM)
        range_ok &= bf16_chunk_to_f16(reinterpret_cast<char*>(S.v) + tile_off<VD>(t, cc));
    }
    __syncthreads();
    const float GL = S.G[L - 1];
    const float gamma = __expf(GL);

    // ---- (1) S = K K^T (and Q K^T when emitting): warp tile rows 16(w%4), cols 32(w/4)
    {
      const int m0 = (warp & 3) * 16, nb = (warp >> 2) * 32;
      float sacc[4][4] = {}, qacc[4][4] = {};
#pragma unroll
      for (int k0 = 0; k0 < KD; k0 += 16) {
        uint32_t ak[4], aq[4], b01[4], b23[4];
        load_a<KD>(sk, m0, k0, ak);
        if (MODE == kEmit) load_a<KD>(sq, m0, k0, aq);
        load_b_nk<KD>(sk, k0, nb, b01);
        load_b_nk<KD>(sk, k0, nb + 16, b23);
        mma16816(sacc[0], ak, b01[0], b01[1]);
        mma16816(sacc[1], ak, b01[2], b01[3]);
        mma16816(sacc[2], ak, b23[0], b23[1]);
        mma16816(sacc[3], ak, b23[2], b23[3]);
        if (MODE == kEmit) {
          mma16816(qacc[0], aq, b01[0], b01[1]);
          mma16816(qacc[1], aq, b01[2], b01[3]);
          mma16816(qacc[2], aq, b23[0], b23[1]);
          mma16816(qacc[3], aq, b23[2], b23[3]);
        }
      }
      for (int nt = 0; nt < 4; ++nt)
        for (int hf = 0; hf < 2; ++hf) {
          const int t = m0 + g8 + hf * 8, s = nb + nt * 8 + 2 * q4;
          float x[2], y[2];
          for (int e = 0; e < 2; ++e) {
            const int ss = s + e;
            const float dec = __expf(S.G[t] - S.G[ss < t ? ss : t]);  // exponent <= 0
            x[e] = ss < t ? S.beta[t] * dec * sacc[nt][2 * hf + e] : 0.f;
            y[e] = ss <= t ? dec * qacc[nt][2 * hf + e] : 0.f;
          }
          S.A[t * FP + s] = x[0];
          S.A[t * FP + s + 1] = x[1];
          if (MODE == kEmit)
            *reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(S.att) + tile_off<C>(t, s) +
                                         (s & 7) * 2) = pack_h2(y[0], y[1]);
        }
    }
    __syncthreads();

    // ---- (2) T = (I + A)^-1, blocked forward substitution over four 16-row blocks, fp32.
    // (a) diagonal blocks: warp b inverts block b, two lanes per column.
    if (warp < 4) {
      const int b = warp * 16, c = lane & 15, half = lane >> 4;
      for (int t = 0; t < 16; ++t) S.Ti[(b + t) * FP + b + c] = (t == c) ? 1.f : 0.f;
      __syncwarp();
      for (int t = 1; t < 16; ++t) {
        float x = 0.f;
        for (int s = half; s < t; s += 2) x += S.A[(b + t) * FP + b + s] * S.Ti[(b + s) * FP + b + c];
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        if (half == 0 && t > c) S.Ti[(b + t) * FP + b + c] = -x;
        __syncwarp();
      }
    }
    __syncthreads();
    // (b) off-diagonal blocks, one sub-diagonal at a time:
    //     T_ab = -T_aa * sum_{m=b}^{a-1} A_am T_mb     (a > b)
    for (int dist = 1; dist < 4; ++dist) {
      const int nblk = 4 - dist;
      // X_ab = sum_m A_am T_mb
      for (int e = tid; e < nblk * 256; e += kThreads) {
        const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
        const int bb = blk, aa = blk + dist;
        float x = 0.f;
        for (int m = bb; m < aa; ++m)
          for (int s = 0; s < 16; ++s)
            x += S.A[(aa * 16 + rr) * FP + m * 16 + s] * S.Ti[(m * 16 + s) * FP + bb * 16 + cc];
        S.X[(aa * 16 + rr) * FP + bb * 16 + cc] = x;
      }
      __syncthreads();
      for (int e = tid; e < nblk * 256; e += kThreads) {
        const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
        const int bb = blk, aa = blk + dist;
        float x = 0.f;
        for (int s = 0; s <= rr; ++s)
          x += S.Ti[(aa * 16 + rr) * FP + aa * 16 + s] * S.X[(aa * 16 + s) * FP + bb * 16 + cc];
        S.Ti[(aa * 16 + rr) * FP + bb * 16 + cc] = -x;
      }
      __syncthreads();
    }
    // T diag(beta e^G) and T diag(beta) as bf16 operands (zero above the diagonal)
    for (int e = tid; e < C * C / 2; e += kThreads) {
      const int t = e >> 5, s = (e & 31) * 2;
      const float t0v = s <= t ? S.Ti[t * FP + s] : 0.f;
      const float t1v = s + 1 <= t ? S.Ti[t * FP + s + 1] : 0.f;
      const float b0 = S.beta[s], b1 = S.beta[s + 1];
      const uint32_t off = tile_off<C>(t, s & ~7) + (s & 7) * 2;
      *reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(S.tw) + off) =
          pack_h2(t0v * b0 * __expf(S.G[s]), t1v * b1 * __expf(S.G[s + 1]));
      *reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(S.tu) + off) =
          pack_h2(t0v * b0, t1v * b1);
    }
    __syncthreads();

    // ---- (3) -w = -T_w K (to smem) and u = T_u V (kept as the delta accumulator).
    // Warp tile: rows 16(w%4), columns 64(w/4).
    const int m0 = (warp & 3) * 16, n0 = (warp >> 2) * 64;
    float dacc[8][4];
    {
      float wacc[8][4] = {};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
        for (int e = 0; e < 4; ++e) dacc[nt][e] = 0.f;
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16) {
        uint32_t aw[4], au[4];
        load_a<C>(stw, m0, k0, aw);
        if (MODE != kSumM) load_a<C>(stu, m0, k0, au);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bk[4];
          load_b_kn<KD>(sk, k0, n0 + np * 16, bk);
          mma16816(wacc[2 * np], aw, bk[0], bk[1]);
          mma16816(wacc[2 * np + 1], aw, bk[2], bk[3]);
          if (MODE != kSumM) {
            uint32_t bv[4];
            load_b_kn<VD>(sv, k0, n0 + np * 16, bv);
            mma16816(dacc[2 * np], au, bv[0], bv[1]);
            mma16816(dacc[2 * np + 1], au, bv[2], bv[3]);
          }
        }
      }
      for (int nt = 0; nt < 8; ++nt)
        range_ok &= store_acc_h<KD>(reinterpret_cast<char*>(S.nw), m0, n0 + nt * 8, wacc[nt], -1.f,
                                    -1.f);
    }
    __syncthreads();

    // ---- (4) delta = u - w h  (and, emitting, Q h): same warp tile.
    float oacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
      for (int e = 0; e < 4; ++e) oacc[nt][e] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < KD; k0 += 16) {
      uint32_t aw[4], aq[4];
      load_a<KD>(snw, m0, k0, aw);
      if (MODE == kEmit) load_a<KD>(sq, m0, k0, aq);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bh[4];
        load_b_kn<VD>(shh, k0, n0 + np * 16, bh);
        mma16816(dacc[2 * np], aw, bh[0], bh[1]);
        mma16816(dacc[2 * np + 1], aw, bh[2], bh[3]);
        if (MODE == kEmit) {
          mma16816(oacc[2 * np], aq, bh[0], bh[1]);
          mma16816(oacc[2 * np + 1], aq, bh[2], bh[3]);
        }
      }
    }
    {
      const int t0r = m0 + g8, t1r = m0 + g8 + 8;
      const float s0 = __expf(GL - S.G[t0r]), s1 = __expf(GL - S.G[t1r]);
      for (int nt = 0; nt < 8; ++nt) {
        if (MODE == kEmit)
          range_ok &= store_acc_h<VD>(reinterpret_cast<char*>(S.d), m0, n0 + nt * 8, dacc[nt], 1.f,
                                      1.f);
        range_ok &= store_acc_h<VD>(reinterpret_cast<char*>(S.dp), m0, n0 + nt * 8, dacc[nt], s0,
                                    s1);
      }
    }
    __syncthreads();

    // ---- (5) o = diag(e^G) Q h + attn_i delta, stored for the chunk's valid rows.
    if (MODE == kEmit) {
      const int t0r = m0 + g8, t1r = m0 + g8 + 8;
      const float e0 = __expf(S.G[t0r]), e1 = __expf(S.G[t1r]);
      for (int nt = 0; nt < 8; ++nt) {
        oacc[nt][0] *= e0; oacc[nt][1] *= e0;
        oacc[nt][2] *= e1; oacc[nt][3] *= e1;
      }
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16) {
        uint32_t aa[4];
        load_a<C>(satt, m0, k0, aa);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bd[4];
          load_b_kn<VD>(sd, k0, n0 + np * 16, bd);
          mma16816(oacc[2 * np], aa, bd[0], bd[1]);
          mma16816(oacc[2 * np + 1], aa, bd[2], bd[3]);
        }
      }
      for (int nt = 0; nt < 8; ++nt) {
        const int c = n0 + nt * 8 + 2 * q4;
        if (t0r < L)
          *reinterpret_cast<__nv_bfloat162*>(gout + ((t0 + t0r) * a.hv + j) * VD + c) =
              __floats2bfloat162_rn(oacc[nt][0], oacc[nt][1]);
        if (t1r < L)
          *reinterpret_cast<__nv_bfloat162*>(gout + ((t0 + t1r) * a.hv + j) * VD + c) =
              __floats2bfloat162_rn(oacc[nt][2], oacc[nt][3]);
      }
    }

    // ---- (6) h <- gamma h + K^T delta'   (warp rows 16w of the state, all columns)
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      for (int e = 0; e < 4; ++e) hacc[nt][e] *= gamma;
#pragma unroll
    for (int k0 = 0; k0 < C; k0 += 16) {
      uint32_t ak[4];
      load_a_t<KD>(sk, warp * 16, k0, ak);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t bd[4];
        load_b_kn<VD>(sdp, k0, np * 16, bd);
        mma16816(hacc[2 * np], ak, bd[0], bd[1]);
        mma16816(hacc[2 * np + 1], ak, bd[2], bd[3]);
      }
    }
  }

  if (!range_ok) set_status(a.status, GDN_ERR_DEVICE_RANGE);

  // ---- write the state out
  float* dst = nullptr;
  if (MODE == kEmit) {
    if (a.h_final && r == a.P - 1) dst = a.h_final + ((int64_t)n * a.hv + j) * KD * VD;
  } else if (MODE == kSumM) {
    dst = a.M_out + ((int64_t)seg * a.hv + j) * KD * KD;
  } else {
    dst = a.U_out + ((int64_t)seg * a.hv + j) * KD * VD;
  }
  if (dst)
    for (int nt = 0; nt < 16; ++nt) {
      const int i0 = warp * 16 + g8, c = nt * 8 + 2 * q4;
      *reinterpret_cast<float2*>(dst + i0 * VD + c) = make_float2(hacc[nt][0], hacc[nt][1]);
      *reinterpret_cast<float2*>(dst + (i0 + 8) * VD + c) = make_float2(hacc[nt][2], hacc[nt][3]);
    }
}

template <int MODE>
cudaError_t launch_chunk(const Args& a, dim3 grid, cudaStream_t s) {
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  const size_t smem = sizeof(Smem);
  cudaError_t e = cudaFuncSetAttribute(tc_chunk_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_chunk_kernel<MODE><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(const Args& a) { return a.bf16 && a.K == KD && a.V == VD; }

// The tensor-core kernels recompute the chunk factors on chip; materialised factors (the
// stage entry points) go through the SIMT kernels.
cudaError_t tc_prepare(const Args& a, cudaStream_t s) { return simt_prepare(a, s); }
cudaError_t tc_scan(const Args& a, cudaStream_t s) { return simt_scan(a, s); }

cudaError_t tc_summary(const Args& a, bool fused_prepare, cudaStream_t s) {
  if (!fused_prepare) return simt_summary(a, s);
  const dim3 grid((unsigned)(a.N * a.P), a.hv, 1);
  cudaError_t e = launch_chunk<kSumM>(a, grid, s);
  if (e != cudaSuccess) return e;
  return launch_chunk<kSumU>(a, grid, s);
}

cudaError_t tc_emit(const Args& a, bool fused_prepare, cudaStream_t s) {
  if (!fused_prepare) return simt_emit(a, s);
  return launch_chunk<kEmit>(a, dim3((unsigned)(a.N * a.P), a.hv, 1), s);
}

}  // namespace gdn
