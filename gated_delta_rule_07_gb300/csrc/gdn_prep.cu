// gdn_prep.cu -- the chunk preparation of the gated delta rule forward as one fully parallel
// tcgen05 kernel (bf16 I/O, K = 128, C = 64).
//
// For every chunk and value head it forms the UT transform of the page "Add context
// parallelism to the Gated Delta Net" (section "Why": the w, u of the chunk map are T diag(.) K
// and T diag(.) V with T = (I + A)^-1) and stores the two scaled inverses the products need:
//     A[t][s] = beta_t exp(G_t - G_s) (k_t . k_s)   (s < t),   T = (I + A)^-1,
//     T_w = T diag(beta exp(G)),   T_u = T diag(beta),
// as fp16 64 x 64 tiles in the 128-byte-swizzle layout the chain kernels' tensor-core products
// read (a record of 16 KB per chunk and value head: T_w, then T_u).  Nothing here depends on a
// state, so all chunks run at once; the chain kernels then load the record instead of solving
// on their own critical path ("Implementation": phase 3 reuses the WY factors).
//
// Work item: a pair of consecutive chunk slots of one value head.  A CTA (9 warps) walks a
// strided range of pairs of one value head:
//   * warp 8 (producer) loads the pair's bf16 keys by TMA and issues the gram
//     [K_0 ; K_1] [K_0 ; K_1]^T as one tcgen05.mma of M = N = 128 into TMEM (its two diagonal
//     64 x 64 blocks are the chunks' grams), one pair ahead of the others: the next pair's load
//     and product run while the current pair is solved;
//   * warps 0-7 read 32 gram entries of one row each, apply beta and the decay (every exponent
//     G_t - G_s <= 0 for s <= t when g <= 0) and write A as fp16 plus its diagonal 16 x 16
//     blocks in fp32; then warps 0-3 solve chunk 0 and warps 4-7 chunk 1: each 16 x 16 diagonal
//     block of T by fp32 forward substitution (two 8 x 8 halves side by side), the off-diagonal
//     blocks by doubling on warp-level mma.sync (T_ab = -T_aa A_ab T_bb, then the lower-left
//     32 x 32 block from the two 32-blocks), written straight to the record.
// Waits are bounded: a wait that gives up records GDN_ERR_DEVICE_TIMEOUT in the status word, and
// the producer still waits (again bounded) for its own copy and product before the TMEM is
// released.
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
constexpr int kWorkers = 256;                // warps 0-7: masked gram and solves
constexpr int kThreads = kWorkers + 32;      // + warp 8: loads and the gram product
constexpr uint32_t kTileBytes = 64 * 128;  // a 64 x 64 fp16 tile
constexpr long long kWaitCycles = 2000000000LL;  // about a second

// Per-chunk solve scratch.
struct SolveTiles {
  uint8_t ah[kTileBytes];            // A [t][s] fp16 (swizzled rows)
  uint8_t th[kTileBytes];            // T [t][s] fp16: the operand of the doubling products
};
struct Solve {
  uint8_t xs[4][16 * 48];            // 16 x 16 fp16 blocks for mma.sync, 48-byte rows
  alignas(16) float adiag[C][20];    // the diagonal 16 x 16 blocks of A, fp32 (padded rows)
  float wd[4][16 * 17];              // per-warp fp32 16 x 16 block of T (padded rows)
};
// Decay and write-strength tables of a chunk.
struct Tables {
  float G[C];                        // inclusive within-chunk cumulative sum of g
  float sw[C], su[C];                // column scales of T_w (beta e^G) and T_u (beta)
};

struct Smem {
  uint8_t k[2 * 128 * 128];  // [feature block][chunk 0 rows 0-63 | chunk 1 rows 64-127][128 B]
  SolveTiles st[2];
  Solve sv[2];
  Tables tb[2][2];           // [pair parity][chunk]
  uint64_t bar_load, bar_mma, bar_tfree;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(offsetof(Smem, k) % 1024 == 0 && offsetof(Smem, st) % 1024 == 0, "tile alignment");
static_assert(sizeof(SolveTiles) % 1024 == 0 && offsetof(Smem, sv) % 16 == 0, "alignment");
static_assert(sizeof(Solve) % 16 == 0 && offsetof(Solve, adiag) % 16 == 0, "alignment");
static_assert(offsetof(Smem, bar_load) % 8 == 0, "alignment");
static_assert(2 * (sizeof(Smem) + 2048) <= 233472, "two CTAs per SM");

__device__ __forceinline__ void arrive_bar(uint32_t bar) { mbar_arrive(bar); }

// Bounded wait (about `cycles` SM cycles) for the phase with the given parity.  Returns false,
// after recording the abort flag, when it gives up or (honour_abort) another thread gave up.
__device__ __noinline__ bool wait_bounded(Smem& S, uint32_t bar, uint32_t parity,
                                          long long cycles, bool honour_abort) {
  const long long t_end = clock64() + cycles;
  while (!mbar_try(bar, parity)) {
    if (clock64() > t_end || (honour_abort && *reinterpret_cast<volatile int*>(&S.abort_flag))) {
      *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
      return false;
    }
  }
  return true;
}

// The zero blocks above the diagonal of a 64 x 64 lower-triangular record tile, 16 bytes per
// thread of the solve group.
__device__ __forceinline__ void zero_upper_blocks(uint8_t* tile, int gt) {
  for (int e = gt; e < 6 * 32; e += 128) {
    const int b = e >> 5, row_in = (e >> 1) & 15, half = e & 1;
    const int rb = b < 3 ? 0 : (b < 5 ? 1 : 2);
    const int cb = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
    const int row = 16 * rb + row_in, c8 = 2 * cb + half;
    *reinterpret_cast<uint4*>(tile + row * 128 + ((c8 ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
  }
}

// T = (I + A)^-1 of one chunk by the solve group (4 warps, 16-row block wb each), from A in
// V.ah (fp16) and V.adiag (fp32); writes T into V.th and T_w, T_u into the record tiles gw, gu.
__device__ __forceinline__ void solve_chunk(SolveTiles& VT, Solve& V, const Tables& TB, int wb,
                                            int lane, int bar_id, uint8_t* gw, uint8_t* gu) {
  const int g8 = lane >> 2, q4 = lane & 3;
  const uint32_t ah_s = saddr(VT.ah), th_s = saddr(VT.th);
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
      *reinterpret_cast<uint32_t*>(V.xs[tile] + g8 * 48 + (8 * nt + 2 * q4) * 2) =
          pack_h2(x[nt][0], x[nt][1]);
      *reinterpret_cast<uint32_t*>(V.xs[tile] + (g8 + 8) * 48 + (8 * nt + 2 * q4) * 2) =
          pack_h2(x[nt][2], x[nt][3]);
    }
  };
  // y += T_blk(a_r, a_c) xs[tile]
  auto mma_xs = [&](float (&y)[2][4], int a_r, int a_c, int tile) {
    uint32_t af[4], bf[4];
    load_a<64>(th_s, a_r, a_c, af);
    const int mi = lane >> 3, rr = lane & 7;
    ldsm_x4_t(saddr(V.xs[tile]) + (rr + ((mi & 1) << 3)) * 48 + ((mi >> 1) << 3) * 2, bf);
    mma16816(y[0], af, bf[0], bf[1]);
    mma16816(y[1], af, bf[2], bf[3]);
  };
  // T_ab = -y into th and the record's T_w, T_u
  auto store_t = [&](const float (&y)[2][4], int ab, int bb) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = 16 * ab + g8 + 8 * hr, col = 16 * bb + 8 * nt + 2 * q4;
        const float v0 = -y[nt][2 * hr], v1 = -y[nt][2 * hr + 1];
        const uint32_t off = sw128_offset(64, row, col);
        *reinterpret_cast<uint32_t*>(VT.th + off) = pack_h2(v0, v1);
        *reinterpret_cast<uint32_t*>(gw + off) = pack_h2(v0 * TB.sw[col], v1 * TB.sw[col + 1]);
        *reinterpret_cast<uint32_t*>(gu + off) = pack_h2(v0 * TB.su[col], v1 * TB.su[col + 1]);
      }
  };

  {  // Diagonal block wb = [[P, 0], [R, Q]] (8 x 8 parts): P^-1 and Q^-1 by forward
     // substitution side by side (lane c < 8: column c of P^-1, 8 <= c < 16: column c - 8 of
     // Q^-1), then the lower left block -Q^-1 (R P^-1) by all lanes, in fp32 in wd.
    float* W = V.wd[wb];
    const float* Ab = &V.adiag[16 * wb][0];
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
    {  // row r = lane / 2, columns 8 (lane & 1) .. + 7 of the block into th, T_w, T_u
      const int r = lane >> 1, col0 = 16 * wb + 8 * (lane & 1);
      const float* wr = W + r * 17 + 8 * (lane & 1);
      uint32_t ph[4], pw[4], pu[4];
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float v0 = wr[j], v1 = wr[j + 1];
        ph[j >> 1] = pack_h2(v0, v1);
        pw[j >> 1] = pack_h2(v0 * TB.sw[col0 + j], v1 * TB.sw[col0 + j + 1]);
        pu[j >> 1] = pack_h2(v0 * TB.su[col0 + j], v1 * TB.su[col0 + j + 1]);
      }
      const uint32_t off = sw128_offset(64, 16 * wb + r, col0);
      *reinterpret_cast<uint4*>(VT.th + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      *reinterpret_cast<uint4*>(gw + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(gu + off) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
    }
  }
  named_bar(bar_id, 128);
  // The off-diagonal blocks by doubling: T_10 and T_32 join the 16-blocks into 32-blocks
  // (T_ab = -T_aa A_ab T_bb), then the lower left 32-block is -T_BB X with X = A_BA T_AA
  // (A = blocks 0-1, B = blocks 2-3), whose products with the diagonal blocks of T_AA are
  // started meanwhile.
  float x[2][4] = {}, x2[2][4] = {};
  const int rw = 2 + (wb >> 1);  // warps 0, 2: row block of X
  if (wb & 1) {
    mma_blk(x, ah_s, 16 * wb, 16 * (wb - 1), th_s, 16 * (wb - 1), 16 * (wb - 1));
    frag_to_xs(x, wb);
    __syncwarp();
    float y[2][4] = {};
    mma_xs(y, 16 * wb, 16 * wb, wb);
    store_t(y, wb, wb - 1);
  } else {
    mma_blk(x, ah_s, 16 * rw, 0, th_s, 0, 0);      // A_r0 T_00
    mma_blk(x2, ah_s, 16 * rw, 16, th_s, 16, 16);  // X_r1 = A_r1 T_11
  }
  named_bar(bar_id, 128);
  if (!(wb & 1)) {
    mma_blk(x, ah_s, 16 * rw, 16, th_s, 16, 0);    // X_r0 = A_r0 T_00 + A_r1 T_10
    frag_to_xs(x, wb);                              // X_20, X_21, X_30, X_31 -> xs[0..3]
    frag_to_xs(x2, wb + 1);
  }
  named_bar(bar_id, 128);
  {  // warp wb: T_{r c}, r = 2 + wb / 2, c = wb % 2:  T_2c = -T_22 X_2c,
     // T_3c = -(T_32 X_2c + T_33 X_3c)
    float y[2][4] = {};
    if (rw == 3) mma_xs(y, 48, 32, wb & 1);
    mma_xs(y, 16 * rw, 16 * rw, wb);
    store_t(y, rw, wb & 1);
  }
}

// Chunks of one pair: whether each slot holds a chunk, its first token and its rows in range.
struct Pair {
  bool ok0, ok1;
  int t0, t1, L0, L1;
};
__device__ __forceinline__ Pair pair_info(const Args& a, int64_t pair) {
  Pair P;
  int n = 0;
  int64_t cg = 0, sb = 0, se = 0;
  P.ok0 = slot_to_chunk(a.cu, a.N, a.T, 2 * pair, n, cg) && seq_bounds(a.cu, n, a.T, nullptr, sb, se);
  P.t0 = P.ok0 ? (int)(sb + C * cg) : 0;
  P.L0 = P.ok0 ? (int)((se - P.t0) < C ? (se - P.t0) : C) : 0;
  P.ok1 = slot_to_chunk(a.cu, a.N, a.T, 2 * pair + 1, n, cg) &&
          seq_bounds(a.cu, n, a.T, nullptr, sb, se);
  P.t1 = P.ok1 ? (int)(sb + C * cg) : 0;
  P.L1 = P.ok1 ? (int)((se - P.t1) < C ? (se - P.t1) : C) : 0;
  return P;
}

__global__ void __launch_bounds__(kThreads, 2)
    tc5_prep_kernel(Args a, uint8_t* rec, int64_t npairs, const __grid_constant__ CUtensorMap tm_k) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.y, kh = j / (a.hv / a.hk);
  const int64_t first = blockIdx.x, stride = gridDim.x;
  if (first >= npairs) return;
  const long long wl = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;  // this call's limit
  const int iters = (int)((npairs - first + stride - 1) / stride);

  if (tid == 0) {
    mbar_init(saddr(&S.bar_load), 1);
    mbar_init(saddr(&S.bar_mma), 1);
    mbar_init(saddr(&S.bar_tfree), kWorkers);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 8) {
    tmem_alloc(saddr(&S.tmem_base), 128);
    tmem_relinquish();
  }
  // the fp32 scratch of each diagonal block's upper right 8 x 8 stays zero
#pragma unroll
  for (int h = 0; h < 2; ++h)
    for (int e = tid; e < 4 * 16 * 17; e += kThreads) (&S.sv[h].wd[0][0])[e] = 0.f;
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = S.tmem_base;
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&S.abort_flag) != 0; };

  // g and beta of chunk h of a pair (warp h, two rows per lane; rows past the sequence read 0),
  // then its tables: load first, scan later, so that the loads overlap other work
  auto tables_load = [&](const Pair& P, int h, float (&x)[2], float (&b)[2]) {
    const bool okh = h ? P.ok1 : P.ok0;
    const int Lh = h ? P.L1 : P.L0, th0 = h ? P.t1 : P.t0;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = lane + 32 * r;
      const bool in = okh && t < Lh;
      const int64_t tt = (int64_t)th0 + t;
      x[r] = in ? a.g[tt * a.hv + j] : 0.f;
      b[r] = in ? a.beta[tt * a.hv + j] : 0.f;
    }
  };
  auto tables_store = [&](Tables& TB, float (&x)[2], const float (&b)[2]) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_up_sync(0xffffffffu, x[0], o);
      const float y1 = __shfl_up_sync(0xffffffffu, x[1], o);
      if (lane >= o) { x[0] += y0; x[1] += y1; }
    }
    x[1] += __shfl_sync(0xffffffffu, x[0], 31);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = lane + 32 * r;
      TB.G[t] = x[r];
      TB.sw[t] = b[r] * __expf(x[r]);
      TB.su[t] = b[r];
    }
  };

  if (warp == 8) {
    // ============================================================ producer (one lane issues)
    // copies and products issued so far (a pending one completes phase issued - 1)
    int loads = 0, mmas = 0;
    bool load_pending = false, mma_pending = false;
    if (lane == 0) {
      auto issue_load = [&](int64_t pr) {
        const Pair P = pair_info(a, pr);
        const uint32_t bar = saddr(&S.bar_load);
        mbar_expect_tx(bar, (P.ok0 ? 2u : 0u) * 8192u + (P.ok1 ? 2u : 0u) * 8192u);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          if (P.ok0) tma_box(saddr(S.k) + kb * 16384, &tm_k, 64 * kb, kh, P.t0, bar);
          if (P.ok1) tma_box(saddr(S.k) + kb * 16384 + 8192, &tm_k, 64 * kb, kh, P.t1, bar);
        }
      };
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
      issue_load(first);
      ++loads;
      load_pending = true;
      const uint32_t id = idesc_f16(128, 128, 0, 0, 1);
      for (int it = 0; it < iters; ++it) {
        // the workers have read the previous gram out of TMEM
        if (it > 0 && !wait_bounded(S, saddr(&S.bar_tfree), (it - 1) & 1, wl, true)) break;
        if (!wait_bounded(S, saddr(&S.bar_load), it & 1, wl, true)) break;
        load_pending = false;
        fence_after_sync();
        const uint32_t kq = saddr(S.k);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t d = sdesc(kq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
          mma_ss(tm, d, d, id, ks > 0);
        }
        mma_commit(saddr(&S.bar_mma));
        ++mmas;
        mma_pending = true;
        // the keys are dead once the product has read them: load the next pair's
        if (!wait_bounded(S, saddr(&S.bar_mma), it & 1, wl, true)) break;
        mma_pending = false;
        if (it + 1 < iters) {
          issue_load(first + (it + 1) * stride);
          ++loads;
          load_pending = true;
        }
      }
      // a producer that gave up still lets its own copy and product land before the TMEM goes
      if (load_pending) wait_bounded(S, saddr(&S.bar_load), (loads - 1) & 1, kWaitCycles / 10, false);
      if (mma_pending) wait_bounded(S, saddr(&S.bar_mma), (mmas - 1) & 1, kWaitCycles / 10, false);
    }
    __syncwarp();
  } else {
    // ============================================================ workers (warps 0-7)
    float x[2] = {0.f, 0.f}, b[2] = {0.f, 0.f};
    if (warp < 2) {
      tables_load(pair_info(a, first), warp, x, b);
      tables_store(S.tb[0][warp], x, b);
    }
    named_bar(3, kWorkers);
    for (int it = 0; it < iters; ++it) {
      const int64_t pr = first + it * stride;
      const Pair P = pair_info(a, pr);
      const Tables* TBp = S.tb[it & 1];
      bool go = wait_bounded(S, saddr(&S.bar_mma), it & 1, wl, true);
      fence_after_sync();
      go = named_bar_and(3, kWorkers, go);
      if (!go) break;
      // ---- masked gram: thread (row r = 32 (warp % 4) + lane, column half warp / 4)
      {
        const int q = warp & 3, hb = warp >> 2;
        const int r = 32 * q + lane, h = r >> 6, t = r & 63;
        float sv[32];
        tmem_ld32(tm + ((uint32_t)(32 * q) << 16) + 64 * h + 32 * hb, sv);
        if (h ? P.ok1 : P.ok0) {
          const Tables& TB = TBp[h];
          Solve& V = S.sv[h];
          const float Gt = TB.G[t], bt = TB.su[t];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int s = 32 * hb + i;
            sv[i] = s < t ? bt * __expf(Gt - TB.G[s]) * sv[i] : 0.f;
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 pk;
            pk.x = pack_h2(sv[8 * ch + 0], sv[8 * ch + 1]);
            pk.y = pack_h2(sv[8 * ch + 2], sv[8 * ch + 3]);
            pk.z = pack_h2(sv[8 * ch + 4], sv[8 * ch + 5]);
            pk.w = pack_h2(sv[8 * ch + 6], sv[8 * ch + 7]);
            *reinterpret_cast<uint4*>(S.st[h].ah + sw128_offset(64, t, 32 * hb + 8 * ch)) = pk;
          }
          if (hb == (t >> 5)) {  // row t of its own diagonal 16-block, in fp32
            const bool upper = (t & 16) != 0;  // (selects, not run-time indices)
#pragma unroll
            for (int k4 = 0; k4 < 16; k4 += 4)
              *reinterpret_cast<float4*>(&V.adiag[t][k4]) =
                  upper ? make_float4(sv[16 + k4], sv[17 + k4], sv[18 + k4], sv[19 + k4])
                        : make_float4(sv[k4], sv[1 + k4], sv[2 + k4], sv[3 + k4]);
          }
        }
      }
      fence_before_sync();
      arrive_bar(saddr(&S.bar_tfree));  // the producer may put the next gram into TMEM
      named_bar(3, kWorkers);           // A and its diagonal blocks are complete
      // the next pair's g and beta, loaded now and scanned after the solve
      const bool has_next = it + 1 < iters;
      if (warp < 2 && has_next) tables_load(pair_info(a, pr + stride), warp, x, b);
      // ---- the solves: warps 4h .. 4h + 3 take chunk h
      {
        const int h = warp >> 2, wb = warp & 3;
        if (h ? P.ok1 : P.ok0) {
          const int64_t slot = 2 * pr + h;
          uint8_t* gw = rec + (slot * a.hv + j) * (int64_t)(2 * kTileBytes);
          uint8_t* gu = gw + kTileBytes;
          zero_upper_blocks(gw, tid & 127);
          zero_upper_blocks(gu, tid & 127);
          solve_chunk(S.st[h], S.sv[h], TBp[h], wb, lane, 1 + h, gw, gu);
        }
      }
      if (warp < 2 && has_next) tables_store(S.tb[(it + 1) & 1][warp], x, b);
      if (!named_bar_and(3, kWorkers, !aborted())) break;  // tables ready; scratch free
    }
  }

  // ---- teardown
  fence_before_sync();
  __syncthreads();
  if (tid == 0 && aborted()) set_status(a.status, GDN_ERR_DEVICE_TIMEOUT);
  if (warp == 8) {
    fence_after_sync();
    tmem_dealloc(tm, 128);
  }
}

}  // namespace

size_t prep_records_bytes(int64_t T, int N, int hv) {
  return ((size_t)(T / C) + (size_t)N + 2) * (size_t)hv * 2 * kTileBytes;
}

cudaError_t prep_launch(const Args& a, void* rec, cudaStream_t s) {
  const int64_t slots = a.T / C + a.N + 1;
  const int64_t npairs = (slots + 1) / 2;
  if (a.T == 0 || a.hv == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // one wave of two CTAs per SM, each walking a strided range of pairs of one value head
  int64_t per_head = (2 * (int64_t)sms) / a.hv;
  if (per_head < 1) per_head = 1;
  if (per_head > npairs) per_head = npairs;
  const dim3 grid((unsigned)per_head, a.hv, 1);
  const size_t smem = sizeof(Smem) + 1024;
  e = cudaFuncSetAttribute(tc5_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  CUtensorMap mk;
  if ((e = make_map(&mk, a.k, a.T, a.hk)) != cudaSuccess) return e;
  tc5_prep_kernel<<<grid, kThreads, smem, s>>>(a, static_cast<uint8_t*>(rec), npairs, mk);
  return cudaGetLastError();
}

}  // namespace gdn
