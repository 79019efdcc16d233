// Backward pass of exact attention on the 5th-generation tensor cores.
//
// "Chapter 33: inference compute optimisation" §33.3, eqs. 33.6-33.8: the
// probabilities are not stored; each block recomputes them from the scores
// and the row's saved lse (P = exp(S - lse)), then
//
//   G_V = P^T G_O,  G_P = G_O V^T,  G_S = P (G_P - D),  D_i = g_o,i . o_i,
//   G_Q = scale G_S K,  G_K = scale G_S^T Q.
//
// D is eq. 33.7's row sum sum_k P_ik (G_P)_ik in the form Exercise 33.4
// derives for attention (g_o . o), computed once per row before the products.
//
// Three kernels, all on the call's stream:
//  1. row facts: D and lse in base-2 units per row; the largest row end
//     min(pos + 1, len) of each 128-row query tile.
//  2. dQ: one CTA per 128-row query tile of one head, walking the key tiles
//     its rows see.  Per tile: S = Q K^T and G_P = G_O V^T (smem x smem ->
//     TMEM), the rows form G_S in bf16 in columns of its own (two buffers by
//     tile parity), then G_Q += G_S K (A from TMEM, K as an N-major B
//     operand).
//  3. dK/dV: one CTA per 128-key tile of one KV head, walking the query
//     tiles of its G query heads that see any of its keys.  Per tile:
//     S^T = K Q^T and G_P^T = V G_O^T; the key rows form P^T and G_S^T in
//     bf16 over those columns; then G_V += P^T G_O and G_K += G_S^T Q.
// Both products into one accumulator stay in one CTA, so no atomics and a
// fixed summation order: the results are deterministic.  The price is that
// S and G_P are formed twice (7 products of 128 x 128 x 128 per tile pair
// instead of 5).
//
// Roles in kernel 2 (352 threads): warps 0-7 one thread per TMEM lane and
// half tile: group g = warp / 4 owns key columns [64 g, 64 g + 64) of every
// tile, lane quarter warp % 4; warp 8 the TMA producer; warp 9 TMEM
// allocation and the thread that issues the accumulating products; warp 10
// the thread that issues the S and G_P products.  Kernel 3 (608 threads) has
// 16 row warps: group g = warp / 4 owns query columns [32 g, 32 g + 32) (half
// g / 2), then the producer (16), the accumulating thread (17) and the score
// thread (18); each group writes its P^T and G_S^T into the first 16 of its
// own 32 columns, so the A operand of half h is two 16-column pieces 32
// columns apart.  (One thread issues a product every ~75 cycles; an N = 64
// product's math takes ~32, and two issuing threads get one every ~49.)
// In dQ, S and G_P are whole-tile products (N = 128) and the rows read them
// out of TMEM at once: the next tile's S (G_P) is issued as soon as every row
// warp has read this tile's, so the tensor core works on tile j + 1 while
// the rows form tile j's P and G_S; nothing waits for G_Q += G_S K but the
// reuse of its G_S buffer two tiles later.  K_j is read by S_j and, one tile
// later, by G_Q += G_S K_j, so the dQ kernel keeps three K slots (two for V):
// with two, the copy of K_{j+2} could start only once G_Q's product of tile
// j had completed, and the copies' latency set the kernel's pace.
// In dK/dV (tensor memory full: S^T, G_P^T, G_V, G_K) the products of a tile
// are issued by half (N = 64 for S^T and G_P^T, K = 64 for the accumulating
// ones), each half with its own barriers, so one half's exponentials
// overlap the tensor core's work on the other half.  The next tile's half g
// overwrites the columns the accumulating products of half g read, so its
// S^T and G_P^T wait until those products have completed (a barrier per
// half).  The stages are split further: the key rows
// form P^T as soon as S^T is in (G_P^T may still be in the pipe) and G_V's
// products start on it while the rows form G_S^T; the next S^T waits only
// for G_V, the next G_P^T for G_K.  The accumulating products come from one thread in
// a fixed order, so the sums stay deterministic.  Every wait is bounded
// (error flag, then an orderly exit).
//
// Visibility is the forward's (length, position, bias, and with the WIN
// instantiations a sliding window; select, not add): invisible entries get
// P = 0 and G_S = 0 exactly.  With a window, dQ blocks start at their rows'
// earliest visible key tile and dK/dV blocks skip the query tiles whose
// windows end before them.  Cache rows past the last
// key a CTA's rows see may hold anything (NaN): the dQ kernel zeroes those K
// rows in shared memory before G_S K reads them.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace blkattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int BT = 128;  // rows of a query tile, keys of a key tile (TMEM lanes)
constexpr int HT = 64;   // half tile: the columns of one group
constexpr int D = 128;   // head dim
constexpr int STAGES = 2;
constexpr int kBox = 128 * 128;       // one 64-dim (128-byte) box of 128 rows: 16 KB
constexpr int kTileBytes = 2 * kBox;  // 128 rows x 128 dims, bf16
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;    // the accumulating products (and TMEM allocation)
constexpr int kScoreWarp = 10; // the S and G_P products
constexpr int kThreads = 352;
// dK/dV kernel: 16 row warps (a lane quarter and 32 query columns each; the
// four warps of a quarter-group g own columns [32 g, 32 g + 32), half g / 2),
// then the producer, the accumulating thread (and TMEM allocation) and the
// score thread
constexpr int kKvRowWarps = 16;
constexpr int kKvTmaWarp = 16;
constexpr int kKvMmaWarp = 17;
constexpr int kKvScoreWarp = 18;
constexpr int kKvThreads = 32 * 19;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescHalf = tc::idesc_bf16(128, HT, 0, 0);  // S half: both K-major, N = 64
constexpr uint32_t kIdescTN = tc::idesc_bf16(128, 128, 0, 1);   // A in TMEM, B N-major, N = 128
constexpr uint32_t kIdescFull = tc::idesc_bf16(128, 128, 0, 0); // S whole: both K-major, N = 128
constexpr uint32_t kColDS = 384;  // dQ: G_S of tiles with even / odd index at +0 / +64 (bf16 pairs)

// Shared memory: two stationary tiles, two 2-stage rings, barriers, facts.
constexpr int kOffA0 = 0;                             // dQ: Q    | dK/dV: K
constexpr int kOffA1 = kTileBytes;                    // dQ: G_O  | dK/dV: V
constexpr int kOffR0 = 2 * kTileBytes;                // dQ: K ring | dK/dV: Q ring
constexpr int kOffR1 = kOffR0 + STAGES * kTileBytes;  // dQ: V ring | dK/dV: G_O ring
constexpr int kOffBar = kOffR1 + STAGES * kTileBytes;
constexpr int kNumBars = 24;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffFacts = kOffMisc + 128;                     // dK/dV: float4 [2][128] (-L, -D, end, start)
constexpr int kMaxQTiles = 1024;                              // query tiles per sequence (T_q <= 131072)
constexpr int kOffEnds = kOffFacts + 2 * 128 * 16;            // dK/dV: int [kMaxQTiles] row ends per query tile
constexpr int kOffStarts = kOffEnds + kMaxQTiles * 4;         // dK/dV (window): smallest row start per query tile
constexpr int kSmemBytes = kOffStarts + kMaxQTiles * 4 + 1024;  // + slack to align to 1024
// dQ kernel: Q and G_O, a 3-slot K ring (K_j is read by S_j and, a tile
// later, by G_Q += G_S K_j, so its slot is held longer than V_j's), a 2-slot
// V ring, barriers.  (No row facts: the rows read their own.)
constexpr int KST = 3;
constexpr int kDqOffQ = 0;
constexpr int kDqOffG = kTileBytes;
constexpr int kDqOffK = 2 * kTileBytes;
constexpr int kDqOffV = kDqOffK + KST * kTileBytes;
constexpr int kDqOffBar = kDqOffV + STAGES * kTileBytes;
constexpr int kDqOffMisc = kDqOffBar + kNumBars * 8;
constexpr int kDqSmemBytes = kDqOffMisc + 128 + 1024;  // + slack to align to 1024
static_assert(kDqSmemBytes <= 227 * 1024, "dQ shared memory");
// Epilogue staging (in a ring the finished products no longer read): per
// compute warp its 32 rows of one group's 64 columns, a row padded to 68
// floats (conflict-free both ways); group g's warps in ring g.
constexpr int kStageRow = HT + 4;
constexpr int kStageWarp = 32 * kStageRow * 4;
static_assert(4 * kStageWarp <= STAGES * kTileBytes, "staging fits a ring");

// One compute warp's 32 rows x 64 columns of an fp32 accumulator (TMEM
// columns col, col + 32) times mul, to rows dst0 + r * row_stride of global
// memory, the first `rows` of them: staged through shared memory so that the
// global stores are 16 lanes to a row, 256 contiguous bytes each.
__device__ __forceinline__ void store_rows(uint32_t col, float mul, float* stg, float* dst0, int64_t row_stride,
                                           int rows, int lane) {
#pragma unroll 1
  for (int q2 = 0; q2 < 2; ++q2) {
    uint32_t r[32];
    tc::ld32(col + 32 * q2, r);
    tc::wait_ld();
#pragma unroll
    for (int c = 0; c < 32; c += 4)
      *reinterpret_cast<float4*>(stg + lane * kStageRow + 32 * q2 + c) =
          make_float4(__uint_as_float(r[c]) * mul, __uint_as_float(r[c + 1]) * mul, __uint_as_float(r[c + 2]) * mul,
                      __uint_as_float(r[c + 3]) * mul);
  }
  __syncwarp();
#pragma unroll 4
  for (int it = 0; it < 16; ++it) {
    const int r = 2 * it + (lane >> 4);
    if (r < rows)
      *reinterpret_cast<float4*>(dst0 + r * row_stride + 4 * (lane & 15)) =
          *reinterpret_cast<const float4*>(stg + r * kStageRow + 4 * (lane & 15));
  }
  __syncwarp();  // the staging rows are read before they are written again
}

static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// One warp's 32 rows x 32 columns of an fp32 accumulator (TMEM columns
// col..col + 31) times mul, to rows dst0 + r * row_stride, the first `rows`
// of them: staged through shared memory (rows padded to 36 floats) so that
// the global stores are 8 lanes to a row, 128 contiguous bytes each.
constexpr int kStage32Row = 32 + 4;
constexpr int kStage32Warp = 32 * kStage32Row;  // floats
static_assert(kKvRowWarps * kStage32Warp * 4 <= 2 * STAGES * kTileBytes, "dK/dV staging fits the rings");
__device__ __forceinline__ void store_rows32(uint32_t col, float mul, float* stg, float* dst0, int64_t row_stride,
                                             int rows, int lane) {
  uint32_t r[32];
  tc::ld32(col, r);
  tc::wait_ld();
#pragma unroll
  for (int c = 0; c < 32; c += 4)
    *reinterpret_cast<float4*>(stg + lane * kStage32Row + c) =
        make_float4(__uint_as_float(r[c]) * mul, __uint_as_float(r[c + 1]) * mul, __uint_as_float(r[c + 2]) * mul,
                    __uint_as_float(r[c + 3]) * mul);
  __syncwarp();
#pragma unroll 4
  for (int it = 0; it < 8; ++it) {
    const int rr = 4 * it + (lane >> 3);
    if (rr < rows)
      *reinterpret_cast<float4*>(dst0 + rr * row_stride + 4 * (lane & 7)) =
          *reinterpret_cast<const float4*>(stg + rr * kStage32Row + 4 * (lane & 7));
  }
  __syncwarp();  // the staging rows are read before they are written again
}



// Half g of S = A B^T over d = 128: A = 128 rows (all), B = rows [64 g, 64 g
// + 64) of a 128-row tile; both K-major, 128-byte swizzled (rows 64.. start
// 8 KB into each 64-dim box, a whole number of 8-row atoms).
__device__ __forceinline__ void issue_half(uint32_t dcol, uint32_t sa, uint32_t sb, int g) {
  const uint32_t alo = tc::desc_lo(sa, 16);
  const uint32_t blo = tc::desc_lo(sb + (uint32_t)(g * HT * 128), 16);
  constexpr uint32_t kHi = tc::desc_hi(1024);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = (uint32_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4);
    tc::mma_ss(dcol, tc::desc_join(alo + off, kHi), tc::desc_join(blo + off, kHi), kIdescHalf, ks > 0 ? 1u : 0u);
  }
}

// S = A B^T over d = 128 for all 128 rows of both tiles (N = 128): the
// dQ kernel's score products.
__device__ __forceinline__ void issue_full(uint32_t dcol, uint32_t sa, uint32_t sb) {
  const uint32_t alo = tc::desc_lo(sa, 16);
  const uint32_t blo = tc::desc_lo(sb, 16);
  constexpr uint32_t kHi = tc::desc_hi(1024);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = (uint32_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4);
    tc::mma_ss(dcol, tc::desc_join(alo + off, kHi), tc::desc_join(blo + off, kHi), kIdescFull, ks > 0 ? 1u : 0u);
  }
}

// C += A B over the contraction rows [64 g, 64 g + 64): A = 128 lanes x 64
// bf16 (packed pairs in 32 TMEM columns from acol), B = those rows of a
// [128 x 128 dims] tile in shared memory (N-major: two 64-dim boxes 16 KB apart).
__device__ __forceinline__ void issue_acc(uint32_t dcol, uint32_t acol, uint32_t sb, int g, bool accumulate) {
  const uint32_t blo = tc::desc_lo(sb, kBox);
  constexpr uint32_t kHi = tc::desc_hi(1024);
#pragma unroll
  for (int ks = 0; ks < HT / 16; ++ks) {
    const uint64_t bdesc = tc::desc_join(blo + (uint32_t)((g * 4 + ks) * 16 * 128 >> 4), kHi);
    tc::mma_ts(dcol, acol + 8 * ks, bdesc, kIdescTN, (accumulate || ks > 0) ? 1u : 0u);
  }
}

// issue_acc for the dK/dV layout: the A operand of half g (64 contraction
// rows, 32 bf16-pair columns) sits as two 16-column pieces 32 columns
// apart (acol and acol + 32), one per row-warp group of the half.
__device__ __forceinline__ void issue_acc_split(uint32_t dcol, uint32_t acol, uint32_t sb, int g, bool accumulate) {
  const uint32_t blo = tc::desc_lo(sb, kBox);
  constexpr uint32_t kHi = tc::desc_hi(1024);
#pragma unroll
  for (int ks = 0; ks < HT / 16; ++ks) {
    const uint64_t bdesc = tc::desc_join(blo + (uint32_t)((g * 4 + ks) * 16 * 128 >> 4), kHi);
    const uint32_t a = acol + (ks < 2 ? 8 * ks : 32 + 8 * (ks - 2));
    tc::mma_ts(dcol, a, bdesc, kIdescTN, (accumulate || ks > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ int row_end(const BwdParams& p, int b, int i, int len) {
  const int pos = p.qpos[b * p.qp_sb + (int64_t)i * p.qp_si];
  return pos < 0 ? 0 : (pos >= len ? len : pos + 1);
}

// first visible key of row i under the sliding window (0 without one, and
// for pos < 0: such a row sees nothing anyway); pos >= 0 first, no overflow
__device__ __forceinline__ int row_start(const BwdParams& p, int b, int i) {
  if (p.window <= 0) return 0;
  const int pos = p.qpos[b * p.qp_sb + (int64_t)i * p.qp_si];
  return pos < 0 ? 0 : max(0, pos - p.window + 1);
}

__device__ __forceinline__ int seq_len(const BwdParams& p, int b) {
  const int len = p.seqlens[b * p.sl_s];
  return len < 0 ? 0 : (len > p.Tmax ? p.Tmax : len);
}

// ---------------------------------------------------------------- row facts
// One warp per (b, query tile): the largest row end of the tile (and the
// smallest row start, for a sliding window).  Then one warp per row
// (b, h, i): -D = -(g_o . o) (fp32) and -L = -lse log2 e (-inf for an empty
// row, so that 2^(x - L) = 0), negated for the fused multiply-adds that use
// them.
__global__ void __launch_bounds__(256) bwd_facts_kernel(const BwdParams p) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Tq;
  const int64_t warps = (int64_t)gridDim.x * 8;
  const int lane = threadIdx.x & 31;
  // first, one warp per (sequence, query tile): the largest row end of the
  // tile and, over the rows that see keys, the smallest row start
  const int64_t tiles = (int64_t)p.B * p.n_qt;
  for (int64_t e = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); e < tiles; e += warps) {
    const int b = (int)(e / p.n_qt);
    const int qt = (int)(e % p.n_qt);
    const int len = seq_len(p, b);
    int mx = 0, mn = 0x7fffffff;
    const int i1 = min(qt * BT + BT, p.Tq);
    for (int i = qt * BT + lane; i < i1; i += 32) {
      const int e_i = row_end(p, b, i, len), s_i = row_start(p, b, i);
      mx = max(mx, e_i);
      if (e_i > s_i) mn = min(mn, s_i);
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (lane == 0) {
      p.ws_end[e] = mx;
      p.ws_start[e] = mn;
    }
  }
  // two rows per warp and step, every load of both issued before either
  // row's reduction (twice the bytes in flight per warp)
  for (int64_t r0 = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r0 < rows; r0 += 2 * warps) {
    uint2 gw[2];
    float o[2][4], l[2];
    int64_t rr[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t r = r0 + u * warps;
      rr[u] = r;
      gw[u] = make_uint2(0u, 0u);
      o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
      l[u] = 0.f;
      if (r >= rows) continue;
      const int i = (int)(r % p.Tq);
      const int64_t bh = r / p.Tq;
      const int h = (int)(bh % p.Hq);
      const int b = (int)(bh / p.Hq);
      const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(p.dout) + b * p.g_sb + h * p.g_sh + i * p.g_si;
      const int64_t ob = b * p.o_sb + h * p.o_sh + i * p.o_si;
      // lane: dims [4 lane, 4 lane + 4) (g_o rows are 16-byte aligned: one 8-byte load)
      gw[u] = *reinterpret_cast<const uint2*>(g + 4 * lane);
      if (p.out_vec) {  // fp32 rows, unit dim stride, 16-byte aligned: one 16-byte load
        const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(p.out) + ob + 4 * lane);
        o[u][0] = v.x; o[u][1] = v.y; o[u][2] = v.z; o[u][3] = v.w;
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t t = ob + (int64_t)(4 * lane + c) * p.o_sd;
          o[u][c] = p.out_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.out)[t])
                               : static_cast<const float*>(p.out)[t];
        }
      }
      if (lane == 0) l[u] = p.lse[b * p.l_sb + h * p.l_sh + i * p.l_si];
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (rr[u] >= rows) break;
      float acc = bf16lo(gw[u].x) * o[u][0];
      acc = fmaf(bf16hi(gw[u].x), o[u][1], acc);
      acc = fmaf(bf16lo(gw[u].y), o[u][2], acc);
      acc = fmaf(bf16hi(gw[u].y), o[u][3], acc);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) {
        p.ws_D[rr[u]] = -acc;
        p.ws_L[rr[u]] = (l[u] == -__builtin_huge_valf()) ? -__builtin_huge_valf() : -l[u] * kLog2e;
      }
    }
  }
}

// L2 prefetch of one box of a 4-D tensor map (no shared memory, no
// completion): the later tiled load of the same box then hits L2.
__device__ __forceinline__ void tma_prefetch_l2_4d(const void* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// TMEM set-up shared by the two tensor-core kernels (after thread 0 has
// initialised the barriers): warp 9 allocates, everyone reads the base.
__device__ __forceinline__ uint32_t setup_tmem(int* misc, int warp, int alloc_warp = kMmaWarp) {
  if (warp == alloc_warp) {
    tc::alloc(reinterpret_cast<uint32_t*>(&misc[0]), kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  return static_cast<uint32_t>(misc[0]);
}

// dQ, step 1: P of one row over 32 keys from its scores s in TMEM words:
// P = 2^(s scale log2 e + m log2 e - L), 0 by select where the key is
// invisible; P replaces s in place (fp32 bits).  Returns the visibility bits
// (bit c: key + c is visible).  MASK = false: every key of the half is
// visible (no bias, the whole half tile before the row end).
template <bool BIAS, bool MASK, bool WIN = false>
__device__ __forceinline__ uint32_t dq_p(uint32_t (&rs)[32], int key, int my_end, float2 c2, float2 nl2,
                                         const float* brow, int64_t bi_sj, int Tmax, int my_start) {
  uint32_t vis = 0xffffffffu;
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float2 x = __ffma2_rn(make_float2(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1])), c2, nl2);
    bool v0 = true, v1 = true;
    if constexpr (MASK) {
      v0 = key + c < my_end;
      v1 = key + c + 1 < my_end;
      if constexpr (WIN) {  // sliding window: keys before the row's first visible key
        v0 = v0 && key + c >= my_start;
        v1 = v1 && key + c + 1 >= my_start;
      }
    }
    if constexpr (BIAS) {
      const float m0 = key + c < Tmax ? brow[(int64_t)(key + c) * bi_sj] : 0.f;
      const float m1 = key + c + 1 < Tmax ? brow[(int64_t)(key + c + 1) * bi_sj] : 0.f;
      v0 = v0 && m0 != -__builtin_huge_valf();
      v1 = v1 && m1 != -__builtin_huge_valf();
      x = __ffma2_rn(make_float2(m0, m1), make_float2(kLog2e, kLog2e), x);
    }
    float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
    if constexpr (MASK || BIAS) {
      p0 = v0 ? p0 : 0.f;
      p1 = v1 ? p1 : 0.f;
      vis &= ~((v0 ? 0u : 1u) << c) & ~((v1 ? 0u : 1u) << (c + 1));
    }
    rs[c] = __float_as_uint(p0);
    rs[c + 1] = __float_as_uint(p1);
  }
  return vis;
}

// dQ, step 2: G_S = P (G_P - D) over the same 32 keys, packed to bf16 pairs,
// by select where the key is invisible (a masked G_P may be NaN).
template <bool SEL>
__device__ __forceinline__ void dq_ds(const uint32_t (&pr)[32], const uint32_t (&rp)[32], uint32_t vis, float2 nd2,
                                      uint32_t (&ds)[16]) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const float2 gp = __fadd2_rn(make_float2(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1])), nd2);
    const float2 g = __fmul2_rn(make_float2(__uint_as_float(pr[c]), __uint_as_float(pr[c + 1])), gp);
    if constexpr (SEL)
      ds[c >> 1] = pack_bf16(((vis >> c) & 1u) ? g.x : 0.f, ((vis >> (c + 1)) & 1u) ? g.y : 0.f);
    else
      ds[c >> 1] = pack_bf16(g.x, g.y);
  }
}

// dK/dV: 32 entries of one key's row (a key over 32 query rows) in two
// steps, so that P^T can go to its products before G_P^T has arrived.
// Step 1: P^T of 32 rows from S^T and the rows' facts f (-L, -D, end,
// start), packed to bf16 pairs, by select where the row does not see the
// key; returns the visibility bits of the 32 rows (bit c: row c sees the
// key).  MASK = false: the key is visible to every row of the half (no bias,
// before every end).
template <bool BIAS, bool MASK, bool WIN = false>
__device__ __forceinline__ uint32_t dkv_p(const uint32_t (&rs)[32], const float4* f, int key, float2 c2,
                                          const float* bcol, int64_t bi_si, int rows_left, bool kin,
                                          uint32_t (&pp)[16]) {
  uint32_t vis = 0xffffffffu;
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const float4 f0 = f[c], f1 = f[c + 1];
    float2 x = __ffma2_rn(make_float2(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1])), c2,
                          make_float2(f0.x, f1.x));
    bool v0 = true, v1 = true;
    if constexpr (MASK) {
      v0 = key < __float_as_int(f0.z);
      v1 = key < __float_as_int(f1.z);
      if constexpr (WIN) {  // sliding window: the row's first visible key in .w
        v0 = v0 && key >= __float_as_int(f0.w);
        v1 = v1 && key >= __float_as_int(f1.w);
      }
    }
    if constexpr (BIAS) {
      const float m0 = (kin && c < rows_left) ? bcol[(int64_t)c * bi_si] : 0.f;
      const float m1 = (kin && c + 1 < rows_left) ? bcol[(int64_t)(c + 1) * bi_si] : 0.f;
      v0 = v0 && m0 != -__builtin_huge_valf();
      v1 = v1 && m1 != -__builtin_huge_valf();
      x = __ffma2_rn(make_float2(m0, m1), make_float2(kLog2e, kLog2e), x);
    }
    float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
    if constexpr (MASK || BIAS) {
      p0 = v0 ? p0 : 0.f;
      p1 = v1 ? p1 : 0.f;
      vis &= ~((v0 ? 0u : 1u) << c) & ~((v1 ? 0u : 1u) << (c + 1));
    }
    pp[c >> 1] = pack_bf16(p0, p1);
  }
  return vis;
}

// Step 2: G_S^T = P (G_P - D) of the 32 rows from G_P^T and step 1's P (the
// bf16 pairs: G_S^T is rounded to bf16 for its product anyway), by select
// where the row does not see the key (a masked G_P may be NaN).
template <bool SEL>
__device__ __forceinline__ void dkv_ds(const uint32_t (&rp)[32], const uint32_t (&pp)[16], uint32_t vis,
                                       const float4* f, uint32_t (&ds)[16]) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const float2 pv = make_float2(__uint_as_float(pp[c >> 1] << 16), __uint_as_float(pp[c >> 1] & 0xffff0000u));
    const float2 g = __fmul2_rn(pv, __fadd2_rn(make_float2(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1])),
                                               make_float2(f[c].y, f[c + 1].y)));
    if constexpr (SEL)
      ds[c >> 1] = pack_bf16(((vis >> c) & 1u) ? g.x : 0.f, ((vis >> (c + 1)) & 1u) ? g.y : 0.f);
    else
      ds[c >> 1] = pack_bf16(g.x, g.y);
  }
}

// The first key tile of a dQ block whose first row is at position q0 under
// a sliding window (rows at their own index, the prefill layout).
__device__ __forceinline__ int dq_spec_first_tile(int q0, int window) {
  const int64_t s0 = (int64_t)q0 - (int64_t)window + 1;
  return s0 > 0 ? (int)(s0 / BT) : 0;
}

// ---------------------------------------------------------------- dQ
template <bool BIAS, bool WIN>
__device__ __forceinline__ void dq_body(const BwdParams& p, const CUtensorMap& tmq, const CUtensorMap& tmg,
                                        const CUtensorMap& tmk, const CUtensorMap& tmv, int blk) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kDqOffBar);
  uint64_t* q_full = bars;            // Q and G_O tiles
  uint64_t* k_full = bars + 1;        // [KST]
  uint64_t* v_full = bars + 4;        // [STAGES]
  uint64_t* k_empty = bars + 6;       // [KST]
  uint64_t* v_empty = bars + 9;       // [STAGES]
  uint64_t* s_full = bars + 11;       // S of the tile is in TMEM
  uint64_t* gp_full = bars + 12;      // G_P of the tile is in TMEM
  uint64_t* s_free = bars + 13;       // the 8 row warps have read S (its columns are free)
  uint64_t* gp_free = bars + 14;      // the 8 row warps have read G_P
  uint64_t* p_full = bars + 15;       // [2] G_S of tiles with even / odd index is in TMEM (8 warps)
  uint64_t* acc_done = bars + 17;     // [2] G_Q += G_S K of tiles with even / odd index has completed
  uint64_t* drain = bars + 19;        // every product has completed (both issuing threads)
  int* misc = reinterpret_cast<int*>(sm + kDqOffMisc);  // [0] TMEM base, [1] CTA end

  // Groups of p.hg_q (sequence, head) pairs whose K/V fit in L2 together;
  // within a group the longest query tiles first (causal: the last tiles see
  // the most keys), the group's heads side by side.
  const int per_group = p.n_qt * p.hg_q;
  const int r_in = blk % per_group;
  const int qt = p.n_qt - 1 - r_in / p.hg_q;
  const int bh = (blk / per_group) * p.hg_q + r_in % p.hg_q;
  if (bh >= p.B * p.Hq) return;  // padding of the last group (the whole CTA)
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int hk = h / p.G;
  const int i0 = qt * BT;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    misc[1] = 0;
    if constexpr (WIN) misc[2] = 0x7fffffff;
    mbar_init(q_full, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(gp_full, 1);
    mbar_init(s_free, 8);
    mbar_init(gp_free, 8);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&p_full[x], 8);
      mbar_init(&acc_done[x], 1);
    }
    mbar_init(drain, 2);
    fence_barrier_init();
  }
  const uint32_t tb = setup_tmem(misc, warp);
  const uint64_t pol = policy_evict_first();
  const uint64_t pol_ring = policy_evict_last();  // K/V tiles: re-read by the head's other query tiles
  if (warp == kTmaWarp && lane == 0) {
    // the query-side tiles and the first key tile (T_max >= 1) right away
    mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
    tma_load_4d(sm + kDqOffQ, &tmq, 0, i0, h, b, q_full, pol);
    tma_load_4d(sm + kDqOffQ + kBox, &tmq, 64, i0, h, b, q_full, pol);
    tma_load_4d(sm + kDqOffG, &tmg, 0, i0, h, b, q_full, pol);
    tma_load_4d(sm + kDqOffG + kBox, &tmg, 64, i0, h, b, q_full, pol);
    // with a window the first key tile follows from the positions: the copy
    // goes to the tile rows at their own index start at (ring position 0;
    // another first tile moves the block's tiles one ring position on)
    const int key_first = WIN ? dq_spec_first_tile(i0, p.window) * BT : 0;
    mbar_arrive_expect_tx(&k_full[0], kTileBytes);
    tma_load_4d(sm + kDqOffK, &tmk, 0, key_first, hk, b, &k_full[0], pol_ring);
    tma_load_4d(sm + kDqOffK + kBox, &tmk, 64, key_first, hk, b, &k_full[0], pol_ring);
    mbar_arrive_expect_tx(&v_full[0], kTileBytes);
    tma_load_4d(sm + kDqOffV, &tmv, 0, key_first, hk, b, &v_full[0], pol_ring);
    tma_load_4d(sm + kDqOffV + kBox, &tmv, 64, key_first, hk, b, &v_full[0], pol_ring);
  }

  const int len = seq_len(p, b);
  const int row_i = i0 + (int)(threadIdx.x & 127);
  const bool my_row = warp < 8 && row_i < p.Tq;
  const int my_end = my_row ? row_end(p, b, row_i, len) : 0;
  int my_start = 0;
  if constexpr (WIN) {
    my_start = my_row ? row_start(p, b, row_i) : 0;
    if (my_row && warp < 4 && my_end > my_start) {
      atomicMax(&misc[1], my_end);
      atomicMin(&misc[2], my_start);
    }
  } else {
    if (my_row && warp < 4) atomicMax(&misc[1], my_end);
  }
  __syncthreads();
  // key tiles [j_lo, j_lo + n) (j_lo = 0 without a window); ring slots and
  // phases count from j_lo
  const int cta_end = misc[1];
  int j_lo = 0, n = (cta_end + BT - 1) / BT;
  if constexpr (WIN) {
    j_lo = misc[2] != 0x7fffffff ? misc[2] / BT : 0;
    n = max(0, n - j_lo);
  }
  // ring position of key tile j: j + ro (ro = 1 when the early copy holds another tile)
  const int ro = (WIN && j_lo != dq_spec_first_tile(i0, p.window)) ? 1 : 0;
  const uint32_t sQ = smem_u32(sm + kDqOffQ), sG = smem_u32(sm + kDqOffG);
  const uint32_t sK = smem_u32(sm + kDqOffK), sV = smem_u32(sm + kDqOffV);
  const int grp = (warp >> 2) & 1;  // column half of a compute warp
  float* dq_row = p.dq + (int64_t)b * p.dq_sb + (int64_t)h * p.dq_sh + (int64_t)row_i * p.dq_si + grp * HT;

  if (n == 0) {
    // no row of the tile sees a key: G_Q = 0; the first copies must land
    if (my_row)
      for (int c = 0; c < HT; c += 4) *reinterpret_cast<float4*>(dq_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp == kTmaWarp && lane == 0) {
      bool landed = mbar_wait(q_full, 0);
      landed = mbar_wait(&k_full[0], 0) && landed;
      landed = mbar_wait(&v_full[0], 0) && landed;
      if (!landed) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kTmaWarp) {
    if (lane == 0) {
      // Q, G_O and ring position 0 are in flight already; positions issued
      int k_issued = 1, v_issued = 1;
      bool ok = true;
      if (ro == 1) {
        // position 0 holds another tile: it lands, then its slots are released
        ok = mbar_wait(&k_full[0], 0) && mbar_wait(&v_full[0], 0);
        mbar_arrive(&k_empty[0]);
        mbar_arrive(&v_empty[0]);
      }
      for (int j = 1 - ro; j < n && ok; ++j) {
        const int u = j + ro;
        const int sk = u % KST, sv = u % STAGES;
        const int key0 = (j_lo + j) * BT;
        if (u >= KST && !mbar_wait(&k_empty[sk], ((u / KST) - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[sk], kTileBytes);
        tma_load_4d(sm + kDqOffK + sk * kTileBytes, &tmk, 0, key0, hk, b, &k_full[sk], pol_ring);
        tma_load_4d(sm + kDqOffK + sk * kTileBytes + kBox, &tmk, 64, key0, hk, b, &k_full[sk], pol_ring);
        k_issued = u + 1;
        if (u >= STAGES && !mbar_wait(&v_empty[sv], ((u / STAGES) - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&v_full[sv], kTileBytes);
        tma_load_4d(sm + kDqOffV + sv * kTileBytes, &tmv, 0, key0, hk, b, &v_full[sv], pol_ring);
        tma_load_4d(sm + kDqOffV + sv * kTileBytes + kBox, &tmv, 64, key0, hk, b, &v_full[sv], pol_ring);
        v_issued = u + 1;
        if (j + 1 < n && u + 1 >= STAGES) {
          // the next tile's copies wait for slots: bring it into L2 now
          tma_prefetch_l2_4d(&tmk, 0, key0 + BT, hk, b);
          tma_prefetch_l2_4d(&tmk, 64, key0 + BT, hk, b);
          tma_prefetch_l2_4d(&tmv, 0, key0 + BT, hk, b);
          tma_prefetch_l2_4d(&tmv, 64, key0 + BT, hk, b);
        }
      }
      // every issued copy lands before the CTA exits
      if (!mbar_wait(q_full, 0)) ok = false;
      for (int j = k_issued - KST < 0 ? 0 : k_issued - KST; j < k_issued; ++j)
        if (!mbar_wait(&k_full[j % KST], (j / KST) & 1)) ok = false;
      for (int j = v_issued - STAGES < 0 ? 0 : v_issued - STAGES; j < v_issued; ++j)
        if (!mbar_wait(&v_full[j % STAGES], (j / STAGES) & 1)) ok = false;
      if (!ok) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kScoreWarp) {
    // ---------------- S and G_P products (one thread) ----------------
    if (lane == 0) {
      auto tile_ready = [&](int j) -> bool {
        const int u = j + ro;
        const bool r = mbar_wait(&k_full[u % KST], (u / KST) & 1) && mbar_wait(&v_full[u % STAGES], (u / STAGES) & 1);
        tc::fence_after();
        return r;
      };
      bool ok = mbar_wait(q_full, 0) && tile_ready(0);
      if (ok) {
        issue_full(tb + 0, sQ, sK + (ro % KST) * kTileBytes);
        tc::commit(s_full);
        issue_full(tb + 128, sG, sV + (ro % STAGES) * kTileBytes);
        tc::commit(gp_full);
        tc::commit(&v_empty[ro % STAGES]);
      }
      for (int j = 0; ok && j + 1 < n; ++j) {
        // tile j + 1's S (G_P) overwrites tile j's as soon as the rows have
        // read it; G_S has columns of its own
        const int s1 = (j + 1 + ro) % STAGES;
        if (!tile_ready(j + 1)) { ok = false; break; }
        if (!mbar_wait(s_free, j & 1)) { ok = false; break; }
        tc::fence_after();
        issue_full(tb + 0, sQ, sK + ((j + 1 + ro) % KST) * kTileBytes);
        tc::commit(s_full);
        if (!mbar_wait(gp_free, j & 1)) { ok = false; break; }
        tc::fence_after();
        issue_full(tb + 128, sG, sV + s1 * kTileBytes);
        tc::commit(gp_full);
        tc::commit(&v_empty[s1]);  // V_{j+1} once its product is done
      }
      if (!ok) record_error(p.err, kErrTimeout);
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ---------------- G_Q += G_S K (one thread; a fixed order) ----------------
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; ok && j < n; ++j) {
        const int s = (j + ro) % KST;
        const int par = j & 1;
        if (!mbar_wait(&p_full[par], (j >> 1) & 1)) { ok = false; break; }
        tc::fence_after();
        issue_acc(tb + 256, tb + kColDS + 64 * par, sK + s * kTileBytes, 0, j > 0);
        issue_acc(tb + 256, tb + kColDS + 64 * par + 32, sK + s * kTileBytes, 1, true);
        tc::commit(&acc_done[par]);
        tc::commit(&k_empty[s]);  // K_j is free: its S completed before its G_S was written
      }
      if (!ok) record_error(p.err, kErrTimeout);
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) record_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- rows x half tile: P, G_S ----------------
    const uint32_t tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quarter
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    const int64_t fact = ((int64_t)b * p.Hq + h) * p.Tq + (my_row ? row_i : 0);
    const float nLrow = my_row ? p.ws_L[fact] : -__builtin_huge_valf();  // -L (base 2)
    const float nDrow = my_row ? p.ws_D[fact] : 0.f;                     // -D
    const float* brow = nullptr;
    if constexpr (BIAS)
      brow = p.bias + (int64_t)b * p.bi_sb + (int64_t)h * p.bi_sh + (int64_t)(my_row ? row_i : 0) * p.bi_si;
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 nl2 = make_float2(nLrow, nLrow);
    const float2 nd2 = make_float2(nDrow, nDrow);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int par = j & 1;
      if (!wait_all(s_full, j & 1)) { ok = false; break; }
      tc::fence_after();
      const int key0 = (j_lo + j) * BT + grp * HT;  // first key of this half
      // (warp-uniform) every row of the warp sees every key of the half
      const bool whole = !BIAS && __all_sync(0xffffffffu, key0 + HT <= my_end && (!WIN || key0 >= my_start));
      // This half of S, then its columns are free for the next tile's S, and
      // P while G_P is in the pipe.  With a bias, S and P go chunk by chunk
      // after G_P has arrived instead (the bias loads would hold too many
      // registers across the wait).
      uint32_t pr[2][32];
      uint32_t vis[2] = {0u, 0u};
      if constexpr (!BIAS) {
        tc::ld32(tl + HT * grp, pr[0]);
        tc::ld32(tl + HT * grp + 32, pr[1]);
        tc::wait_ld();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          if (whole)
            vis[q2] = dq_p<false, false, WIN>(pr[q2], key0 + 32 * q2, my_end, c2, nl2, brow, p.bi_sj, p.Tmax, my_start);
          else
            vis[q2] = dq_p<false, true, WIN>(pr[q2], key0 + 32 * q2, my_end, c2, nl2, brow, p.bi_sj, p.Tmax, my_start);
        }
      }
      if (!wait_all(gp_full, j & 1)) { ok = false; break; }
      // G_S of tile j goes where tile j - 2's was: its product must have completed
      if (j >= 2 && !wait_all(&acc_done[par], ((j >> 1) - 1) & 1)) { ok = false; break; }
      tc::fence_after();
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        if constexpr (BIAS) {  // (whole is false with a bias)
          tc::ld32(tl + HT * grp + 32 * q2, pr[q2]);
          tc::wait_ld();
          if (q2 == 1) {
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
          }
          vis[q2] = dq_p<true, true, WIN>(pr[q2], key0 + 32 * q2, my_end, c2, nl2, brow, p.bi_sj, p.Tmax, my_start);
        }
        uint32_t rp[32], ds[16];
        tc::ld32(tl + 128 + HT * grp + 32 * q2, rp);
        tc::wait_ld();
        if (q2 == 1) {  // G_P's columns are free for the next tile's G_P
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(gp_free);
        }
        if (whole)
          dq_ds<false>(pr[q2], rp, vis[q2], nd2, ds);
        else
          dq_ds<true>(pr[q2], rp, vis[q2], nd2, ds);
        tc::st16(tl + kColDS + 64 * par + 32 * grp + 16 * q2, ds);
      }
      if ((j_lo + j) * BT + BT > cta_end) {
        // last tile: the K rows of this half past every visible key of the
        // CTA are zeroed before G_S K reads them (they may hold anything)
        const int s = (j + ro) % KST;
        if (!wait_all(&k_full[s], ((j + ro) / KST) & 1)) { ok = false; break; }
        unsigned char* kt = sm + kDqOffK + s * kTileBytes;
        const int z0 = max(cta_end - (j_lo + j) * BT, grp * HT);
        const int t = (int)(threadIdx.x & 127);
        for (int idx = t; idx < (grp * HT + HT - z0) * 16; idx += 128) {
          const int r = z0 + (idx >> 4);
          const int c = idx & 15;
          *reinterpret_cast<uint4*>(kt + (c >> 3) * kBox + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[par]);
    }
    if (ok && !wait_all(drain, 0)) ok = false;
    if (!ok) {
      if (lane == 0) record_error(p.err, kErrTimeout);
    } else {
      // G_Q: this group stores dims [64 g, 64 g + 64) of the warp's rows,
      // staged in the K/V rings (every product has completed)
      tc::fence_after();
      const int r0 = i0 + 32 * (warp & 3);
      store_rows(tl + 256 + HT * grp, p.scale,
                 reinterpret_cast<float*>(sm + kDqOffK + (grp * 4 + (warp & 3)) * kStageWarp),
                 p.dq + (int64_t)b * p.dq_sb + (int64_t)h * p.dq_sh + (int64_t)r0 * p.dq_si + grp * HT, p.dq_si,
                 min(32, p.Tq - r0), lane);
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tb, kTmemCols);
}

// ---------------------------------------------------------------- dK / dV
// The (query head, query tile) pairs a key tile visits: for each of the G
// heads of its KV head, the query tiles whose largest row end passes the
// tile's first key (and, with a sliding window, whose smallest row start
// comes before its last key).  Every role walks the same sequence.
struct Visit {
  int g, qt;
};
template <bool WIN>
__device__ __forceinline__ bool next_visit(const BwdParams& p, const int* ends, const int* starts, int k0,
                                           Visit& v) {
  // advance from v (exclusive); v.g = -1 starts
  int g = v.g, qt = v.qt + 1;
  if (g < 0) {
    g = 0;
    qt = 0;
  }
  while (g < p.G) {
    while (qt < p.n_qt && (ends[qt] <= k0 || (WIN && starts[qt] >= k0 + BT))) ++qt;
    if (qt < p.n_qt) {
      v.g = g;
      v.qt = qt;
      return true;
    }
    ++g;
    qt = 0;
  }
  return false;
}

template <bool BIAS, bool WIN>
__device__ __forceinline__ void dkv_body(const BwdParams& p, const CUtensorMap& tmq, const CUtensorMap& tmg,
                                         const CUtensorMap& tmk, const CUtensorMap& tmv, int blk) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* kv_full = bars;          // K and V tiles
  uint64_t* qg_full = bars + 1;      // [STAGES] Q and G_O tiles
  uint64_t* qg_empty = bars + 3;     // [STAGES]
  uint64_t* s_full = bars + 5;       // [2] half g of S^T in TMEM
  uint64_t* gp_full = bars + 7;      // [2] half g of G_P^T in TMEM
  uint64_t* pt_full = bars + 9;      // [2] half g of P^T in TMEM (4 warps of group g)
  uint64_t* ds_full = bars + 11;     // [2] half g of G_S^T in TMEM (4 warps of group g)
  uint64_t* dv_done = bars + 13;     // [2] G_V += P^T G_O over half g has completed
  uint64_t* dk_done = bars + 15;     // [2] G_K += G_S^T Q over half g has completed
  uint64_t* drain = bars + 17;       // every product has completed (both issuing threads)
  int* misc = reinterpret_cast<int*>(sm + kOffMisc);
  float4* facts = reinterpret_cast<float4*>(sm + kOffFacts);  // [2][128]: L, D, end (int bits), -
  int* ends = reinterpret_cast<int*>(sm + kOffEnds);          // this sequence's row end per query tile
  int* starts = reinterpret_cast<int*>(sm + kOffStarts);      // (window) smallest row start per query tile

  // Groups of p.hg_kv (sequence, KV head) pairs whose query-side tiles fit in
  // L2 together; within a group the longest key tiles first (causal: the
  // first tiles are seen by the most rows), the group's heads side by side.
  const int per_group = p.n_kt * p.hg_kv;
  const int r_in = blk % per_group;
  const int kt = r_in / p.hg_kv;
  const int bk = (blk / per_group) * p.hg_kv + r_in % p.hg_kv;
  if (bk >= p.B * p.Hkv) return;  // padding of the last group (the whole CTA)
  const int b = bk / p.Hkv;
  const int hk = bk % p.Hkv;
  const int k0 = kt * BT;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the visit sequence is walked from shared memory (a global load per step
  // sat on the MMA thread's path between visits); published by the barrier
  // in setup_tmem
  for (int i = threadIdx.x; i < p.n_qt; i += kKvThreads) {
    ends[i] = p.ws_end[(int64_t)b * p.n_qt + i];
    if constexpr (WIN) starts[i] = p.ws_start[(int64_t)b * p.n_qt + i];
  }

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&qg_full[s], 1);
      mbar_init(&qg_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&gp_full[g], 1);
      mbar_init(&pt_full[g], 8);  // the 8 row warps of half g
      mbar_init(&ds_full[g], 8);
      mbar_init(&dv_done[g], 1);
      mbar_init(&dk_done[g], 1);
    }
    mbar_init(drain, 2);
    fence_barrier_init();
  }
  const uint32_t tb = setup_tmem(misc, warp, kKvMmaWarp);
  const uint32_t sK = smem_u32(sm + kOffA0), sV = smem_u32(sm + kOffA1);
  const uint32_t sQ = smem_u32(sm + kOffR0), sG = smem_u32(sm + kOffR1);
  const uint64_t pol = policy_evict_first();
  const uint64_t pol_ring = policy_evict_last();  // Q/G_O tiles: re-read by the head's other key tiles
  Visit first{-1, -1};
  const bool any = next_visit<WIN>(p, ends, starts, k0, first);

  if (warp == kKvTmaWarp) {
    if (lane == 0 && any) {
      bool ok = true;
      mbar_arrive_expect_tx(kv_full, 2 * kTileBytes);
      tma_load_4d(sm + kOffA0, &tmk, 0, k0, hk, b, kv_full, pol);
      tma_load_4d(sm + kOffA0 + kBox, &tmk, 64, k0, hk, b, kv_full, pol);
      tma_load_4d(sm + kOffA1, &tmv, 0, k0, hk, b, kv_full, pol);
      tma_load_4d(sm + kOffA1 + kBox, &tmv, 64, k0, hk, b, kv_full, pol);
      Visit v = first;
      int t = 0;
      do {
        const int s = t % STAGES;
        if (t >= STAGES && !mbar_wait(&qg_empty[s], ((t / STAGES) - 1) & 1)) { ok = false; break; }
        const int h = hk * p.G + v.g;
        const int row = v.qt * BT;
        mbar_arrive_expect_tx(&qg_full[s], 2 * kTileBytes);
        tma_load_4d(sm + kOffR0 + s * kTileBytes, &tmq, 0, row, h, b, &qg_full[s], pol_ring);
        tma_load_4d(sm + kOffR0 + s * kTileBytes + kBox, &tmq, 64, row, h, b, &qg_full[s], pol_ring);
        tma_load_4d(sm + kOffR1 + s * kTileBytes, &tmg, 0, row, h, b, &qg_full[s], pol_ring);
        tma_load_4d(sm + kOffR1 + s * kTileBytes + kBox, &tmg, 64, row, h, b, &qg_full[s], pol_ring);
        ++t;
        Visit vn = v;
        if (t >= STAGES && next_visit<WIN>(p, ends, starts, k0, vn)) {
          // the next visit's copies wait for a slot: bring its tiles into L2 now
          const int hn = hk * p.G + vn.g, rn = vn.qt * BT;
          tma_prefetch_l2_4d(&tmq, 0, rn, hn, b);
          tma_prefetch_l2_4d(&tmq, 64, rn, hn, b);
          tma_prefetch_l2_4d(&tmg, 0, rn, hn, b);
          tma_prefetch_l2_4d(&tmg, 64, rn, hn, b);
        }
      } while (next_visit<WIN>(p, ends, starts, k0, v));
      if (!mbar_wait(kv_full, 0)) ok = false;
      for (int u = t - STAGES < 0 ? 0 : t - STAGES; u < t; ++u)
        if (!mbar_wait(&qg_full[u % STAGES], (u / STAGES) & 1)) ok = false;
      if (!ok) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kKvScoreWarp) {
    // ---------------- S^T and G_P^T products (one thread) ----------------
    if (lane == 0 && any) {
      // S^T (G_P^T) of the query rows [64 g, 64 g + 64) of visit t
      auto half_s = [&](int t, int g) {
        issue_half(tb + HT * g, sK, sQ + (t % STAGES) * kTileBytes, g);
        tc::commit(&s_full[g]);
      };
      auto half_gp = [&](int t, int g) {
        issue_half(tb + 128 + HT * g, sV, sG + (t % STAGES) * kTileBytes, g);
        tc::commit(&gp_full[g]);
      };
      auto visit_ready = [&](int t) -> bool {
        const bool r = mbar_wait(&qg_full[t % STAGES], (t / STAGES) & 1);
        tc::fence_after();
        return r;
      };
      bool ok = mbar_wait(kv_full, 0) && visit_ready(0);
      if (ok) {
        half_s(0, 0);
        half_gp(0, 0);
        half_s(0, 1);
        half_gp(0, 1);
      }
      Visit v = first;
      for (int t = 0; ok && next_visit<WIN>(p, ends, starts, k0, v); ++t) {
        // S^T of visit t + 1 overwrites the P^T columns G_V of visit t read,
        // G_P^T the G_S^T columns G_K read: each waits for those products
        if (!visit_ready(t + 1)) { ok = false; break; }
        const uint32_t ph = t & 1;
        if (!mbar_wait(&dv_done[0], ph)) { ok = false; break; }
        tc::fence_after();
        half_s(t + 1, 0);
        if (!mbar_wait(&dk_done[0], ph)) { ok = false; break; }
        tc::fence_after();
        half_gp(t + 1, 0);
        if (!mbar_wait(&dv_done[1], ph)) { ok = false; break; }
        tc::fence_after();
        half_s(t + 1, 1);
        if (!mbar_wait(&dk_done[1], ph)) { ok = false; break; }
        tc::fence_after();
        half_gp(t + 1, 1);
      }
      if (!ok) record_error(p.err, kErrTimeout);
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kKvMmaWarp) {
    // ---------------- G_V += P^T G_O, G_K += G_S^T Q (one thread; a fixed order) ----------------
    if (lane == 0 && any) {
      bool ok = true;
      Visit v = first;
      for (int t = 0; ok; ++t) {
        const int s = t % STAGES;
        const bool next = next_visit<WIN>(p, ends, starts, k0, v);
        const uint32_t ph = t & 1;
        // G_V over half 0 as soon as its P^T is in, G_K once its G_S^T is,
        // then half 1 (this order every visit)
        if (!mbar_wait(&pt_full[0], ph)) { ok = false; break; }
        tc::fence_after();
        issue_acc_split(tb + 256, tb + 0, sG + s * kTileBytes, 0, t > 0);
        tc::commit(&dv_done[0]);
        if (!mbar_wait(&ds_full[0], ph)) { ok = false; break; }
        tc::fence_after();
        issue_acc_split(tb + 384, tb + 128, sQ + s * kTileBytes, 0, t > 0);
        tc::commit(&dk_done[0]);
        if (!mbar_wait(&pt_full[1], ph)) { ok = false; break; }
        tc::fence_after();
        issue_acc_split(tb + 256, tb + HT, sG + s * kTileBytes, 1, true);
        tc::commit(&dv_done[1]);
        if (!mbar_wait(&ds_full[1], ph)) { ok = false; break; }
        tc::fence_after();
        issue_acc_split(tb + 384, tb + 128 + HT, sQ + s * kTileBytes, 1, true);
        tc::commit(&dk_done[1]);
        // the visit's Q and G_O slot is free: its halves completed before its P^T was written
        tc::commit(&qg_empty[s]);
        if (!next) break;
      }
      if (!ok) record_error(p.err, kErrTimeout);
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) record_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- keys x 32 query columns: P^T, G_S^T ----------------
    const int grp = warp >> 2;  // columns [32 grp, 32 grp + 32): half hf = grp / 2
    const int hf = grp >> 1;
    const int key = k0 + 32 * (warp & 3) + lane;
    const uint32_t tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    const int len = seq_len(p, b);
    const int t128 = (int)(threadIdx.x & 127);  // thread within the group
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    bool ok = true;
    if (any) {
      Visit v = first;
      for (int t = 0;; ++t) {
        const int h = hk * p.G + v.g;
        float4* f = facts + (t & 1) * 128 + grp * 32;
        if (t128 < 32) {
          // the facts of this group's query rows, one row per thread
          const int i = v.qt * BT + grp * 32 + t128;
          float4 e = make_float4(-__builtin_huge_valf(), 0.f, __int_as_float(0), __int_as_float(0));
          if (i < p.Tq) {
            const int64_t r = ((int64_t)b * p.Hq + h) * p.Tq + i;
            e = make_float4(p.ws_L[r], p.ws_D[r], __int_as_float(row_end(p, b, i, len)),
                            __int_as_float(WIN ? row_start(p, b, i) : 0));
          }
          f[t128] = e;
          // the smallest row end (and largest row start) of the group's rows
          const int mn = __reduce_min_sync(0xffffffffu, __float_as_int(e.z));
          if (lane == 0) misc[4 + (t & 1) * 4 + grp] = mn;
          if constexpr (WIN) {
            const int mx = __reduce_max_sync(0xffffffffu, __float_as_int(e.w));
            if (lane == 0) misc[12 + (t & 1) * 4 + grp] = mx;
          }
        }
        // (the barrier also publishes the facts; the answer is the same for
        // the group's 128 threads, so none is left at a later barrier)
        if (!bar_and(1 + grp, 128, wait_all(&s_full[hf], t & 1))) { ok = false; break; }
        tc::fence_after();
        const float* bcol = nullptr;
        if constexpr (BIAS)
          bcol = p.bias + (int64_t)b * p.bi_sb + (int64_t)h * p.bi_sh +
                 (int64_t)(v.qt * BT + grp * 32) * p.bi_si + (int64_t)key * p.bi_sj;
        // (warp-uniform) every row of the group sees every key of the warp
        const int mn = misc[4 + (t & 1) * 4 + grp];
        const int mx = misc[12 + (t & 1) * 4 + grp];
        const bool whole = !BIAS && __all_sync(0xffffffffu, key < mn && (!WIN || key >= mx));
        const int rows_left = p.Tq - (v.qt * BT + grp * 32);  // rows of the group inside T_q
        // step 1: P^T from S^T (G_P^T may still be in the tensor pipe), into
        // the first 16 of this group's own 32 columns
        uint32_t pk[16], vis;
        {
          uint32_t rs[32];
          tc::ld32(tl + 32 * grp, rs);
          tc::wait_ld();
          if (whole)
            vis = dkv_p<BIAS, false, WIN>(rs, f, key, c2, bcol, p.bi_si, rows_left, key < p.Tmax, pk);
          else
            vis = dkv_p<BIAS, true, WIN>(rs, f, key, c2, bcol, p.bi_si, rows_left, key < p.Tmax, pk);
          tc::st16(tl + 32 * grp, pk);
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pt_full[hf]);
        // step 2: G_S^T from G_P^T and P, likewise over G_P^T's columns
        if (!bar_and(1 + grp, 128, wait_all(&gp_full[hf], t & 1))) { ok = false; break; }
        tc::fence_after();
        {
          uint32_t rp[32], ds[16];
          tc::ld32(tl + 128 + 32 * grp, rp);
          tc::wait_ld();
          if (whole)
            dkv_ds<false>(rp, pk, vis, f, ds);
          else
            dkv_ds<true>(rp, pk, vis, f, ds);
          tc::st16(tl + 128 + 32 * grp, ds);
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ds_full[hf]);
        if (!next_visit<WIN>(p, ends, starts, k0, v)) break;
      }
      if (ok && !wait_all(drain, 0)) ok = false;
    }
    float* dv_row = p.dv + (int64_t)b * p.dv_sb + (int64_t)hk * p.dv_sh + (int64_t)key * p.dv_sj + grp * 32;
    float* dk_row = p.dk + (int64_t)b * p.dk_sb + (int64_t)hk * p.dk_sh + (int64_t)key * p.dk_sj + grp * 32;
    if (!ok) {
      if (lane == 0) record_error(p.err, kErrTimeout);
    } else if (!any) {
      if (key < p.Tmax)
        for (int c = 0; c < 32; c += 4) {
          *reinterpret_cast<float4*>(dv_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(dk_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    } else {
      // this warp stores dims [32 grp, 32 grp + 32) of G_V and G_K for its
      // keys, staged in the Q/G_O rings (every product has completed; the
      // tensor-memory loads are warp-collective: every lane takes part)
      tc::fence_after();
      const int key_w = k0 + 32 * (warp & 3);
      float* stg = reinterpret_cast<float*>(sm + kOffR0) + warp * kStage32Warp;
      const int rows = min(32, p.Tmax - key_w);
      store_rows32(tl + 256 + 32 * grp, 1.f, stg,
                   p.dv + (int64_t)b * p.dv_sb + (int64_t)hk * p.dv_sh + (int64_t)key_w * p.dv_sj + grp * 32, p.dv_sj,
                   rows, lane);
      store_rows32(tl + 384 + 32 * grp, p.scale, stg,
                   p.dk + (int64_t)b * p.dk_sb + (int64_t)hk * p.dk_sh + (int64_t)key_w * p.dk_sj + grp * 32, p.dk_sj,
                   rows, lane);
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kKvMmaWarp) tc::dealloc(tb, kTmemCols);
}

template <bool BIAS, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmg,
              const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  dq_body<BIAS, WIN>(p, tmq, tmg, tmk, tmv, (int)blockIdx.x);
}
template <bool BIAS, bool WIN>
__global__ void __launch_bounds__(kKvThreads, 1)
    dkv_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmg,
               const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  dkv_body<BIAS, WIN>(p, tmq, tmg, tmk, tmv, (int)blockIdx.x);
}
template <bool BIAS, bool WIN>
cudaError_t launch_pair(const BwdParams& p, const CUtensorMap& tmq, const CUtensorMap& tmg, const CUtensorMap& tmk,
                        const CUtensorMap& tmv, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute((const void*)dq_kernel<BIAS, WIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute((const void*)dkv_kernel<BIAS, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.hg_q < 1 || p.hg_kv < 1 || p.n_qt > kMaxQTiles) return cudaErrorInvalidValue;
  const int64_t dq_blocks = ((int64_t)p.B * p.Hq + p.hg_q - 1) / p.hg_q * p.hg_q * p.n_qt;
  const int64_t dkv_blocks = ((int64_t)p.B * p.Hkv + p.hg_kv - 1) / p.hg_kv * p.hg_kv * p.n_kt;
  if (dq_blocks > 0x7fffffff || dkv_blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (dq_blocks > 0) {
    dq_kernel<BIAS, WIN><<<(unsigned)dq_blocks, kThreads, kDqSmemBytes, stream>>>(p, tmq, tmg, tmk, tmv);
    if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  }
  dkv_kernel<BIAS, WIN><<<(unsigned)dkv_blocks, kKvThreads, kSmemBytes, stream>>>(p, tmq, tmg, tmk, tmv);
  return cudaGetLastError();
}

}  // namespace

int backward_smem_bytes() { return kDqSmemBytes > kSmemBytes ? kDqSmemBytes : kSmemBytes; }

cudaError_t launch_backward(const BwdParams& p, const CUtensorMap& tmq, const CUtensorMap& tmg,
                            const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Tq;
  int64_t fb = (rows + 7) / 8;
  if (fb < 1) fb = 1;
  if (fb > 4096) fb = 4096;
  bwd_facts_kernel<<<(unsigned)fb, 256, 0, stream>>>(p);
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  if (p.window > 0)
    return p.bias != nullptr ? launch_pair<true, true>(p, tmq, tmg, tmk, tmv, stream)
                             : launch_pair<false, true>(p, tmq, tmg, tmk, tmv, stream);
  return p.bias != nullptr ? launch_pair<true, false>(p, tmq, tmg, tmk, tmv, stream)
                           : launch_pair<false, false>(p, tmq, tmg, tmk, tmv, stream);
}

}  // namespace blkattn
