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
//     TMEM), then the rows form G_S in bf16 over G_P's columns, then
//     G_Q += G_S K (A from TMEM, K as an N-major B operand).
//  3. dK/dV: one CTA per 128-key tile of one KV head, walking the query
//     tiles of its G query heads that see any of its keys.  Per tile:
//     S^T = K Q^T and G_P^T = V G_O^T; the key rows form P^T and G_S^T in
//     bf16 over their columns; then G_V += P^T G_O and G_K += G_S^T Q.
// Both products into one accumulator stay in one CTA, so no atomics and a
// fixed summation order: the results are deterministic.  The price is that
// S and G_P are formed twice (7 products of 128 x 128 x 128 per tile pair
// instead of 5).
//
// Roles in kernels 2 and 3 (192 threads): warps 0-3 one thread per TMEM lane
// (a query row in 2, a key in 3), warp 4 the TMA producer, warp 5 TMEM
// allocation and the single MMA-issuing thread.  Products execute in issue
// order, so the next tile's S may overwrite the columns the previous tile's
// products read.  Every wait is bounded (error flag, then an orderly exit).
//
// Visibility is the forward's (length, position, bias; select, not add):
// invisible entries get P = 0 and G_S = 0 exactly.  Cache rows past the last
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
constexpr int D = 128;   // head dim
constexpr int STAGES = 2;
constexpr int kBox = 128 * 128;       // one 64-dim (128-byte) box of 128 rows: 16 KB
constexpr int kTileBytes = 2 * kBox;  // 128 rows x 128 dims, bf16
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescKK = tc::idesc_bf16(128, 128, 0, 0);  // both operands K-major
constexpr uint32_t kIdescTN = tc::idesc_bf16(128, 128, 0, 1);  // A in TMEM, B N-major

// Shared memory: two stationary tiles, two 2-stage rings, barriers, facts.
constexpr int kOffA0 = 0;                             // dQ: Q    | dK/dV: K
constexpr int kOffA1 = kTileBytes;                    // dQ: G_O  | dK/dV: V
constexpr int kOffR0 = 2 * kTileBytes;                // dQ: K ring | dK/dV: Q ring
constexpr int kOffR1 = kOffR0 + STAGES * kTileBytes;  // dQ: V ring | dK/dV: G_O ring
constexpr int kOffBar = kOffR1 + STAGES * kTileBytes;
constexpr int kNumBars = 16;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffFacts = kOffMisc + 64;                   // dK/dV: [2][3][128] (L, D, end)
constexpr int kSmemBytes = kOffFacts + 2 * 3 * 128 * 4 + 1024;  // + slack to align to 1024

static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// S (or S^T) = A B^T over d = 128: both operands K-major, 128-byte swizzled.
__device__ __forceinline__ void issue_kk(uint32_t dcol, uint32_t sa, uint32_t sb) {
  const uint32_t alo = tc::desc_lo(sa, 16);
  const uint32_t blo = tc::desc_lo(sb, 16);
  constexpr uint32_t kHi = tc::desc_hi(1024);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = (uint32_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4);
    tc::mma_ss(dcol, tc::desc_join(alo + off, kHi), tc::desc_join(blo + off, kHi), kIdescKK, ks > 0 ? 1u : 0u);
  }
}

// C += A B with A = 128 lanes x 128 bf16 (packed pairs in 64 TMEM columns
// from acol) and B = a [128 rows (the contraction) x 128 dims] tile in shared
// memory (N-major: two 64-dim boxes 16 KB apart).
__device__ __forceinline__ void issue_tn(uint32_t dcol, uint32_t acol, uint32_t sb, bool accumulate) {
  const uint32_t blo = tc::desc_lo(sb, kBox);
  constexpr uint32_t kHi = tc::desc_hi(1024);
#pragma unroll
  for (int ks = 0; ks < BT / 16; ++ks) {
    const uint64_t bdesc = tc::desc_join(blo + (uint32_t)(ks * 16 * 128 >> 4), kHi);
    tc::mma_ts(dcol, acol + 8 * ks, bdesc, kIdescTN, (accumulate || ks > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ int row_end(const BwdParams& p, int b, int i, int len) {
  const int pos = p.qpos[b * p.qp_sb + (int64_t)i * p.qp_si];
  return pos < 0 ? 0 : (pos >= len ? len : pos + 1);
}

__device__ __forceinline__ int seq_len(const BwdParams& p, int b) {
  const int len = p.seqlens[b * p.sl_s];
  return len < 0 ? 0 : (len > p.Tmax ? p.Tmax : len);
}

// ---------------------------------------------------------------- row facts
// One warp per row (b, h, i): D = g_o . o (fp32), L = lse * log2 e (+inf for
// an empty row, so that 2^(x - L) = 0).  Then one thread per (b, query tile):
// the largest row end of the tile.
__global__ void __launch_bounds__(256) bwd_facts_kernel(const BwdParams p) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Tq;
  const int64_t warps = (int64_t)gridDim.x * 8;
  const int lane = threadIdx.x & 31;
  for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += warps) {
    const int i = (int)(r % p.Tq);
    const int64_t bh = r / p.Tq;
    const int h = (int)(bh % p.Hq);
    const int b = (int)(bh / p.Hq);
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(p.dout) + b * p.g_sb + h * p.g_sh + i * p.g_si;
    const int64_t ob = b * p.o_sb + h * p.o_sh + i * p.o_si;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      const int t = lane + 32 * c;
      const float o = p.out_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.out)[ob + t * p.o_sd])
                                 : static_cast<const float*>(p.out)[ob + t * p.o_sd];
      acc = fmaf(__bfloat162float(g[t]), o, acc);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const float l = p.lse[b * p.l_sb + h * p.l_sh + i * p.l_si];
      p.ws_D[r] = acc;
      p.ws_L[r] = (l == -__builtin_huge_valf()) ? __builtin_huge_valf() : l * kLog2e;
    }
  }
  const int64_t tiles = (int64_t)p.B * p.n_qt;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < tiles; e += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(e / p.n_qt);
    const int qt = (int)(e % p.n_qt);
    const int len = seq_len(p, b);
    int mx = 0;
    for (int i = qt * BT; i < min(qt * BT + BT, p.Tq); ++i) mx = max(mx, row_end(p, b, i, len));
    p.ws_end[e] = mx;
  }
}

// ---------------------------------------------------------------- dQ
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmg,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* q_full = bars;            // Q and G_O tiles
  uint64_t* k_full = bars + 1;        // [STAGES]
  uint64_t* v_full = bars + 3;        // [STAGES]
  uint64_t* k_empty = bars + 5;       // [STAGES]
  uint64_t* v_empty = bars + 7;       // [STAGES]
  uint64_t* sp_full = bars + 9;       // S and G_P of the tile are in TMEM
  uint64_t* ds_full = bars + 10;      // G_S of the tile is in TMEM (4 row warps)
  uint64_t* drain = bars + 11;        // every product has completed
  int* misc = reinterpret_cast<int*>(sm + kOffMisc);  // [0] TMEM base, [1] CTA end

  // longest query tiles first (causal: the last tiles see the most keys)
  const int per = p.B * p.Hq;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x / per);
  const int bh = (int)(blockIdx.x % per);
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int hk = h / p.G;
  const int i0 = qt * BT;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    misc[1] = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(sp_full, 1);
    mbar_init(ds_full, 4);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::alloc(reinterpret_cast<uint32_t*>(&misc[0]), kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint64_t pol_q = policy_evict_first();
  if (warp == kTmaWarp && lane == 0) {
    // the query-side tiles and the first key tile (T_max >= 1) right away
    mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
    tma_load_4d(sm + kOffA0, &tmq, 0, i0, h, b, q_full, pol_q);
    tma_load_4d(sm + kOffA0 + kBox, &tmq, 64, i0, h, b, q_full, pol_q);
    tma_load_4d(sm + kOffA1, &tmg, 0, i0, h, b, q_full, pol_q);
    tma_load_4d(sm + kOffA1 + kBox, &tmg, 64, i0, h, b, q_full, pol_q);
    mbar_arrive_expect_tx(&k_full[0], kTileBytes);
    tma_load_4d(sm + kOffR0, &tmk, 0, 0, hk, b, &k_full[0], pol_q);
    tma_load_4d(sm + kOffR0 + kBox, &tmk, 64, 0, hk, b, &k_full[0], pol_q);
    mbar_arrive_expect_tx(&v_full[0], kTileBytes);
    tma_load_4d(sm + kOffR1, &tmv, 0, 0, hk, b, &v_full[0], pol_q);
    tma_load_4d(sm + kOffR1 + kBox, &tmv, 64, 0, hk, b, &v_full[0], pol_q);
  }

  const int len = seq_len(p, b);
  const int row_i = i0 + (int)(threadIdx.x & 127);
  const bool my_row = warp < 4 && row_i < p.Tq;
  const int my_end = my_row ? row_end(p, b, row_i, len) : 0;
  if (my_row) atomicMax(&misc[1], my_end);
  __syncthreads();
  const int cta_end = misc[1];
  const int n = (cta_end + BT - 1) / BT;
  const uint32_t tb = static_cast<uint32_t>(misc[0]);
  const uint32_t sQ = smem_u32(sm + kOffA0), sG = smem_u32(sm + kOffA1);
  const uint32_t sK = smem_u32(sm + kOffR0), sV = smem_u32(sm + kOffR1);
  float* dq_row = p.dq + (int64_t)b * p.dq_sb + (int64_t)h * p.dq_sh + (int64_t)row_i * p.dq_si;

  if (n == 0) {
    // no row of the tile sees a key: G_Q = 0; the first copies must land
    if (my_row)
      for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(dq_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp == kTmaWarp && lane == 0) {
      bool landed = mbar_wait(q_full, 0);
      landed = mbar_wait(&k_full[0], 0) && landed;
      landed = mbar_wait(&v_full[0], 0) && landed;
      if (!landed) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kTmaWarp) {
    if (lane == 0) {
      // Q, G_O and K/V tile 0 are in flight already
      int k_issued = 1, v_issued = 1;
      bool ok = true;
      for (int j = 1; j < n && ok; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = ((j / STAGES) - 1) & 1;
        if (j >= STAGES && !mbar_wait(&k_empty[s], ph)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[s], kTileBytes);
        tma_load_4d(sm + kOffR0 + s * kTileBytes, &tmk, 0, j * BT, hk, b, &k_full[s], pol_q);
        tma_load_4d(sm + kOffR0 + s * kTileBytes + kBox, &tmk, 64, j * BT, hk, b, &k_full[s], pol_q);
        k_issued = j + 1;
        if (j >= STAGES && !mbar_wait(&v_empty[s], ph)) { ok = false; break; }
        mbar_arrive_expect_tx(&v_full[s], kTileBytes);
        tma_load_4d(sm + kOffR1 + s * kTileBytes, &tmv, 0, j * BT, hk, b, &v_full[s], pol_q);
        tma_load_4d(sm + kOffR1 + s * kTileBytes + kBox, &tmv, 64, j * BT, hk, b, &v_full[s], pol_q);
        v_issued = j + 1;
      }
      // every issued copy lands before the CTA exits
      if (!mbar_wait(q_full, 0)) ok = false;
      for (int j = k_issued - STAGES < 0 ? 0 : k_issued - STAGES; j < k_issued; ++j)
        if (!mbar_wait(&k_full[j % STAGES], (j / STAGES) & 1)) ok = false;
      for (int j = v_issued - STAGES < 0 ? 0 : v_issued - STAGES; j < v_issued; ++j)
        if (!mbar_wait(&v_full[j % STAGES], (j / STAGES) & 1)) ok = false;
      if (!ok) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0);
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = (j / STAGES) & 1;
        if (!mbar_wait(&k_full[s], ph)) { ok = false; break; }
        tc::fence_after();
        issue_kk(tb + 0, sQ, sK + s * kTileBytes);          // S = Q K^T
        if (!mbar_wait(&v_full[s], ph)) { ok = false; break; }
        tc::fence_after();
        issue_kk(tb + 128, sG, sV + s * kTileBytes);        // G_P = G_O V^T
        tc::commit(sp_full);
        tc::commit(&v_empty[s]);
        if (!mbar_wait(ds_full, j & 1)) { ok = false; break; }
        tc::fence_after();
        issue_tn(tb + 256, tb + 128, sK + s * kTileBytes, j > 0);  // G_Q += G_S K
        tc::commit(&k_empty[s]);
      }
      if (!ok) record_error(p.err, kErrTimeout);
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) record_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- rows: P, G_S ----------------
    const uint32_t tl = tb + ((uint32_t)(32 * warp) << 16);  // this warp's lane quarter
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    const int64_t fact = ((int64_t)b * p.Hq + h) * p.Tq + (my_row ? row_i : 0);
    const float Lrow = my_row ? p.ws_L[fact] : __builtin_huge_valf();
    const float Drow = my_row ? p.ws_D[fact] : 0.f;
    const float* brow = (p.bias != nullptr && my_row)
                            ? p.bias + (int64_t)b * p.bi_sb + (int64_t)h * p.bi_sh + (int64_t)row_i * p.bi_si
                            : nullptr;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!wait_all(sp_full, j & 1)) { ok = false; break; }
      tc::fence_after();
      const int key0 = j * BT;
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t rs[32], rp[32], ds[16];
        tc::ld32(tl + 32 * q4, rs);
        tc::ld32(tl + 128 + 32 * q4, rp);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float g2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = key0 + 32 * q4 + c + e;
            float x = __uint_as_float(rs[c + e]) * p.scale_log2;
            bool vis = key < my_end;
            if (brow != nullptr) {
              const float m = key < p.Tmax ? brow[(int64_t)key * p.bi_sj] : 0.f;
              vis = vis && m != -__builtin_huge_valf();
              x = fmaf(m, kLog2e, x);
            }
            const float pr = fast_exp2(x - Lrow);
            g2[e] = vis ? pr * (__uint_as_float(rp[c + e]) - Drow) : 0.f;
          }
          ds[c >> 1] = pack_bf16(g2[0], g2[1]);
        }
        tc::st16(tl + 128 + 16 * q4, ds);  // G_S over G_P's first 64 columns
      }
      if (key0 + BT > cta_end) {
        // last tile: K rows past every visible key of the CTA are zeroed
        // before G_S K reads them (they may hold anything)
        const int s = j % STAGES;
        if (!wait_all(&k_full[s], (j / STAGES) & 1)) { ok = false; break; }
        unsigned char* kt = sm + kOffR0 + s * kTileBytes;
        const int z0 = cta_end - key0;
        for (int idx = (int)threadIdx.x; idx < (BT - z0) * 16; idx += 128) {
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
      if (lane == 0) mbar_arrive(ds_full);
    }
    if (ok && !wait_all(drain, 0)) ok = false;
    if (!ok) {
      if (lane == 0) record_error(p.err, kErrTimeout);
    } else {
      tc::fence_after();
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t r[32];
        tc::ld32(tl + 256 + 32 * q4, r);
        tc::wait_ld();
        if (my_row) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(dq_row + 32 * q4 + c) =
                make_float4(__uint_as_float(r[c]) * p.scale, __uint_as_float(r[c + 1]) * p.scale,
                            __uint_as_float(r[c + 2]) * p.scale, __uint_as_float(r[c + 3]) * p.scale);
        }
      }
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
// tile's first key.  Every role walks the same sequence.
struct Visit {
  int g, qt;
};
__device__ __forceinline__ bool next_visit(const BwdParams& p, const int* ends, int k0, Visit& v) {
  // advance from v (exclusive); v.g = -1 starts
  int g = v.g, qt = v.qt + 1;
  if (g < 0) {
    g = 0;
    qt = 0;
  }
  while (g < p.G) {
    while (qt < p.n_qt && ends[qt] <= k0) ++qt;
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

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkv_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmg,
                   const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* kv_full = bars;          // K and V tiles
  uint64_t* qg_full = bars + 1;      // [STAGES] Q and G_O tiles
  uint64_t* qg_empty = bars + 3;     // [STAGES]
  uint64_t* sp_full = bars + 5;      // S^T and G_P^T in TMEM
  uint64_t* p_full = bars + 6;       // P^T and G_S^T in TMEM (4 key warps)
  uint64_t* drain = bars + 7;
  int* misc = reinterpret_cast<int*>(sm + kOffMisc);
  float* facts = reinterpret_cast<float*>(sm + kOffFacts);  // [2][3][128]: L, D, end (int bits)

  // longest key tiles first (causal: the first tiles are seen by the most rows)
  const int per = p.B * p.Hkv;
  const int kt = (int)(blockIdx.x / per);
  const int r_in = (int)(blockIdx.x % per);
  const int b = r_in / p.Hkv;
  const int hk = r_in % p.Hkv;
  const int k0 = kt * BT;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int* ends = p.ws_end + (int64_t)b * p.n_qt;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&qg_full[s], 1);
      mbar_init(&qg_empty[s], 1);
    }
    mbar_init(sp_full, 1);
    mbar_init(p_full, 4);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::alloc(reinterpret_cast<uint32_t*>(&misc[0]), kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = static_cast<uint32_t>(misc[0]);
  const uint32_t sK = smem_u32(sm + kOffA0), sV = smem_u32(sm + kOffA1);
  const uint32_t sQ = smem_u32(sm + kOffR0), sG = smem_u32(sm + kOffR1);
  const uint64_t pol = policy_evict_first();
  Visit first{-1, -1};
  const bool any = next_visit(p, ends, k0, first);

  if (warp == kTmaWarp) {
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
        tma_load_4d(sm + kOffR0 + s * kTileBytes, &tmq, 0, row, h, b, &qg_full[s], pol);
        tma_load_4d(sm + kOffR0 + s * kTileBytes + kBox, &tmq, 64, row, h, b, &qg_full[s], pol);
        tma_load_4d(sm + kOffR1 + s * kTileBytes, &tmg, 0, row, h, b, &qg_full[s], pol);
        tma_load_4d(sm + kOffR1 + s * kTileBytes + kBox, &tmg, 64, row, h, b, &qg_full[s], pol);
        ++t;
      } while (next_visit(p, ends, k0, v));
      if (!mbar_wait(kv_full, 0)) ok = false;
      for (int u = t - STAGES < 0 ? 0 : t - STAGES; u < t; ++u)
        if (!mbar_wait(&qg_full[u % STAGES], (u / STAGES) & 1)) ok = false;
      if (!ok) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && any) {
      bool ok = mbar_wait(kv_full, 0);
      Visit v = first;
      int t = 0;
      while (ok) {
        const int s = t % STAGES;
        if (!mbar_wait(&qg_full[s], (t / STAGES) & 1)) { ok = false; break; }
        tc::fence_after();
        issue_kk(tb + 0, sK, sQ + s * kTileBytes);    // S^T = K Q^T
        issue_kk(tb + 128, sV, sG + s * kTileBytes);  // G_P^T = V G_O^T
        tc::commit(sp_full);
        if (!mbar_wait(p_full, t & 1)) { ok = false; break; }
        tc::fence_after();
        issue_tn(tb + 256, tb + 0, sG + s * kTileBytes, t > 0);    // G_V += P^T G_O
        issue_tn(tb + 384, tb + 128, sQ + s * kTileBytes, t > 0);  // G_K += G_S^T Q
        tc::commit(&qg_empty[s]);
        ++t;
        if (!next_visit(p, ends, k0, v)) break;
      }
      if (!ok) record_error(p.err, kErrTimeout);
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) record_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- keys: P^T, G_S^T ----------------
    const int key = k0 + (int)threadIdx.x;
    const uint32_t tl = tb + ((uint32_t)(32 * warp) << 16);
    const int len = seq_len(p, b);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    bool ok = true;
    if (any) {
      Visit v = first;
      int t = 0;
      while (true) {
        const int h = hk * p.G + v.g;
        float* f = facts + (t & 1) * 3 * 128;
        {
          // this tile's row facts, one row per thread
          const int i = v.qt * BT + (int)threadIdx.x;
          float L = __builtin_huge_valf(), Dv = 0.f;
          int e = 0;
          if (i < p.Tq) {
            const int64_t r = ((int64_t)b * p.Hq + h) * p.Tq + i;
            L = p.ws_L[r];
            Dv = p.ws_D[r];
            e = row_end(p, b, i, len);
          }
          f[threadIdx.x] = L;
          f[128 + threadIdx.x] = Dv;
          f[256 + threadIdx.x] = __int_as_float(e);
        }
        // (the barrier also publishes the facts; the verdict is the same
        // for all 128 key threads, so none is left at a later barrier)
        if (!bar_and(1, 128, wait_all(sp_full, t & 1))) { ok = false; break; }
        tc::fence_after();
        const float* brow = p.bias != nullptr
                                ? p.bias + (int64_t)b * p.bi_sb + (int64_t)h * p.bi_sh +
                                      (int64_t)(v.qt * BT) * p.bi_si + (int64_t)key * p.bi_sj
                                : nullptr;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t rs[32], rp[32], pp[16], ds[16];
          tc::ld32(tl + 32 * q4, rs);
          tc::ld32(tl + 128 + 32 * q4, rp);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float pv[2], gv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int col = 32 * q4 + c + e;  // query row within the tile
              float x = __uint_as_float(rs[c + e]) * p.scale_log2;
              bool vis = key < __float_as_int(f[256 + col]);
              if (brow != nullptr) {
                const int i = v.qt * BT + col;
                const float m = (i < p.Tq && key < p.Tmax) ? brow[(int64_t)col * p.bi_si] : 0.f;
                vis = vis && m != -__builtin_huge_valf();
                x = fmaf(m, kLog2e, x);
              }
              const float pr = vis ? fast_exp2(x - f[col]) : 0.f;
              pv[e] = pr;
              gv[e] = vis ? pr * (__uint_as_float(rp[c + e]) - f[128 + col]) : 0.f;
            }
            pp[c >> 1] = pack_bf16(pv[0], pv[1]);
            ds[c >> 1] = pack_bf16(gv[0], gv[1]);
          }
          tc::st16(tl + 16 * q4, pp);         // P^T over S^T's first 64 columns
          tc::st16(tl + 128 + 16 * q4, ds);   // G_S^T over G_P^T's first 64 columns
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        ++t;
        if (!next_visit(p, ends, k0, v)) break;
      }
      if (ok && !wait_all(drain, 0)) ok = false;
    }
    if (!ok) {
      if (lane == 0) record_error(p.err, kErrTimeout);
    } else if (key < p.Tmax) {
      float* dv_row = p.dv + (int64_t)b * p.dv_sb + (int64_t)hk * p.dv_sh + (int64_t)key * p.dv_sj;
      float* dk_row = p.dk + (int64_t)b * p.dk_sb + (int64_t)hk * p.dk_sh + (int64_t)key * p.dk_sj;
      if (!any) {
        for (int c = 0; c < D; c += 4) {
          *reinterpret_cast<float4*>(dv_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(dk_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    if (ok && any) {
      // the tensor-memory loads are warp-collective: every lane takes part
      tc::fence_after();
      float* dv_row = p.dv + (int64_t)b * p.dv_sb + (int64_t)hk * p.dv_sh + (int64_t)key * p.dv_sj;
      float* dk_row = p.dk + (int64_t)b * p.dk_sb + (int64_t)hk * p.dk_sh + (int64_t)key * p.dk_sj;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        float* dst = part == 0 ? dv_row : dk_row;
        const float mul = part == 0 ? 1.f : p.scale;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t r[32];
          tc::ld32(tl + 256 + 128 * part + 32 * q4, r);
          tc::wait_ld();
          if (key < p.Tmax) {
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(dst + 32 * q4 + c) =
                  make_float4(__uint_as_float(r[c]) * mul, __uint_as_float(r[c + 1]) * mul,
                              __uint_as_float(r[c + 2]) * mul, __uint_as_float(r[c + 3]) * mul);
          }
        }
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tb, kTmemCols);
}

}  // namespace

int backward_smem_bytes() { return kSmemBytes; }

cudaError_t launch_backward(const BwdParams& p, const CUtensorMap& tmq, const CUtensorMap& tmg,
                            const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    for (const void* f : {(const void*)bwd_dq_kernel, (const void*)bwd_dkv_kernel}) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  const int64_t rows = (int64_t)p.B * p.Hq * p.Tq;
  int64_t fb = (rows + 7) / 8;
  if (fb < 1) fb = 1;
  if (fb > 4096) fb = 4096;
  bwd_facts_kernel<<<(unsigned)fb, 256, 0, stream>>>(p);
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  const int64_t dq_blocks = (int64_t)p.B * p.Hq * p.n_qt;
  const int64_t dkv_blocks = (int64_t)p.B * p.Hkv * p.n_kt;
  if (dq_blocks > 0x7fffffff || dkv_blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (dq_blocks > 0) {
    bwd_dq_kernel<<<(unsigned)dq_blocks, kThreads, kSmemBytes, stream>>>(p, tmq, tmg, tmk, tmv);
    if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  }
  bwd_dkv_kernel<<<(unsigned)dkv_blocks, kThreads, kSmemBytes, stream>>>(p, tmq, tmg, tmk, tmv);
  return cudaGetLastError();
}

}  // namespace blkattn
