// Causal prefill kernel on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Exact blocked attention ("Chapter 33: inference compute optimisation"
// §33.2, Algorithm 33.1; §33.3 for the on-chip tiling and the skipping of
// fully invisible blocks): a CTA owns TWO query tiles of 128 consecutive rows
// of one head (rows [i0, i0 + 256)) and walks the key tiles of 128 keys that
// hold any key visible to them, keeping per row the statistics (m, l, u) of
// eq. 33.3 with u in tensor memory.  Both query tiles share every K/V tile
// the CTA loads; key tiles beyond the CTA's last visible key are never loaded.
//
//   S_j  = Q K_j^T     tcgen05.mma M=128 N=128 K=16 x 8      (smem x smem -> TMEM)
//   U   += P_j V_j     tcgen05.mma M=128 N=128 K=16 x 8 (x 2 on split tiles; P from TMEM, V smem)
//
// Roles (320 threads): warps 0-3 and 4-7 = one thread per query row of the
// first / second query tile (a TMEM lane each): scores, mask by select,
// online statistics, P; warp 8 = TMA producer (both Q tiles once, K and V
// tiles into 2-stage rings released separately); warp 9 = TMEM allocation
// and the single thread that issues every MMA.  Each query tile has one S
// buffer in TMEM and P_j is written over it.  On a key tile that some row of
// the query tile does not see in full (the diagonal, a window's leading
// edge: where the rows with few keys get most of their weight) P_j goes in
// as bf16 P_hi and P_lo (P = P_hi + P_lo to ~16 bits, two PV products, ~2^-17
// relative accuracy although P is not an input); on the other tiles as one
// bf16 P rounded to nearest, with l summing the rounded values so that u / l
// stays a convex combination of the values (rows that see those tiles see
// at least 128 keys in each, and the rounding errors average out: measured
// well inside the output bar).  The MMA thread tells the two kinds of tile
// apart by the same rule as the rows.  S_{j+1} is issued right after U +=
// P_j V_j (products execute in issue order).  The two query tiles ping-pong: while
// one tile's rows compute P, the tensor core runs the other tile's products.
// Each tile's chain S_j -> P_j -> products -> S_{j+1} passes through the
// MMA thread, so its issue path is kept short: shared-memory descriptors are
// formed once per operand buffer and only their address word moves.
// The epilogue (o = u / l) stages fp32 rows in the freed K / V ring and
// stores them with tiled TMA when the output layout allows it.
//
// Online rescaling is lazy: a row keeps its reference maximum m until a tile
// raises the row maximum by more than 8 (base-2 units); only then is its U
// row rescaled in TMEM.  S_j ready implies U += P_{j-1} V_{j-1} completed, so
// the rescale needs no extra wait.  With any reference m >= (true max - 8)
// the state (m, l, u) still represents the same set (eqs. 33.4-33.5 hold for
// any common reference), and P <= 2^8.
//
// With a sliding window ("Chapter 33" §33.7, the paragraph of eq. 33.16;
// the WIN instantiation) a row at position pos sees keys pos - W < j <= pos:
// each query tile gets a first key tile (its rows' earliest visible key), the
// CTA loads from the smaller of the two, and the leading tiles are masked per
// row.  The unwindowed instantiation is unchanged by this.
//
// Rows with no visible key keep the empty state and get out = 0,
// lse = -inf.  V rows of the last tile past the CTA's last visible key (cache
// padding, possibly NaN) are zero-filled in shared memory before the PV
// product so that 0 * garbage never reaches U.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace blkattn {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLazyRescale = 8.f;  // base-2 units: rescale only when max grows by > 2^8

constexpr int BM = 128;  // query rows per query tile (TMEM lanes)
constexpr int QT = 2;    // query tiles per CTA
constexpr int BN = 128;  // keys per tile
constexpr int D = 128;   // head dim
constexpr int STAGES = 2;
constexpr int kBox = 128 * 128;       // one 64-dim (128-byte) box of 128 rows: 16 KB
constexpr int kTileBytes = 2 * kBox;  // one Q, K or V tile of 128 rows x 128 dims
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + QT * kTileBytes;
constexpr int kOffV = kOffK + STAGES * kTileBytes;
constexpr int kOffBar = kOffV + STAGES * kTileBytes;
// q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[QT], p_full[QT], drain
constexpr int kNumBars = 1 + 4 * STAGES + QT + QT + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align to 1024
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTileCols = 256;  // per query tile: S / P at [0, 128), U at [128, 256)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColPlo = 64;     // P_hi at [0, 64), P_lo at [64, 128) (bf16 pairs)
constexpr uint32_t kColO = 128;
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kIdescQK = tc::idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16(BM, D, 0, 1);   // P (TMEM), V MN-major

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// The first key tile of a CTA whose first row is at position q0 under a
// sliding window (rows at their own index, the prefill layout).
__device__ __forceinline__ int spec_first_tile(int q0, int window) {
  const int64_t s0 = (int64_t)q0 - (int64_t)window + 1;
  return s0 > 0 ? (int)(s0 / BN) : 0;
}

template <bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tmo) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* v_full = k_full + STAGES;
  uint64_t* k_empty = v_full + STAGES;
  uint64_t* v_empty = k_empty + STAGES;
  uint64_t* s_full = v_empty + STAGES;  // [QT]
  uint64_t* p_full = s_full + QT;       // [QT]
  uint64_t* drain = p_full + QT;
  // misc: [0] tmem base, [1 + 2x] end of query tile x, [2 + 2x] min end of x, [5] timeout,
  // (sliding window) [6 + 2x] smallest and [7 + 2x] largest first visible key of x's rows
  int* misc = reinterpret_cast<int*>(sm + kOffMisc);

  // Linear grid in dispatch order: groups of p.head_group (sequence, head)
  // pairs whose K/V fit in L2 together; within a group every head's longest
  // (latest) query-tile pair goes before any shorter one.  The next group's
  // long pairs start while the previous group's short ones finish.
  const int n_pairs = (p.Tq + 2 * BM - 1) / (2 * BM);
  const int hg = p.head_group;
  const int per_group = n_pairs * hg;
  const int group = blockIdx.x / per_group;
  const int r_in = blockIdx.x % per_group;
  const int pair = n_pairs - 1 - r_in / hg;
  const int bh = group * hg + r_in % hg;
  if (bh >= p.Hq * p.B) return;  // padding of the last group
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int hk = h / p.G;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int x = warp >> 2;  // query tile of a row warp (0 or 1)
  const int i0 = (2 * pair + (warp < 8 ? x : 0)) * BM;

  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();  // K/V tiles are re-read by the other query tiles
  // Barriers and tensor memory first: the producer then starts both Q tiles
  // and the first K/V tile (always inside the cache, T_max >= 1) while the
  // rows read their positions.
  if (threadIdx.x == 0) {
    misc[1] = 0; misc[2] = 0x7fffffff;
    misc[3] = 0; misc[4] = 0x7fffffff;
    misc[5] = 0;
    misc[6] = 0x7fffffff; misc[7] = 0;
    misc[8] = 0x7fffffff; misc[9] = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < QT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);  // one arrival per row warp of the query tile
    }
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
  if (warp == kTmaWarp && lane == 0) {
    const int q0 = 2 * pair * BM;
    mbar_arrive_expect_tx(q_full, QT * kTileBytes);
    for (int t = 0; t < QT; ++t) {
      tma_load_4d(sm + kOffQ + t * kTileBytes, &tmq, 0, q0 + t * BM, h, b, q_full, pol_q);
      tma_load_4d(sm + kOffQ + t * kTileBytes + kBox, &tmq, 64, q0 + t * BM, h, b, q_full, pol_q);
    }
    // K/V tile 0 of the CTA's range right away; with a window the range
    // starts at the key tile of the CTA's earliest visible key, known only
    // from the positions, so the copy goes to the tile that rows at positions
    // q0 + r would start at (ring position 0; if the positions say otherwise,
    // the CTA's tiles start at ring position 1 and this copy is dropped)
    const int key_first = WIN ? spec_first_tile(2 * pair * BM, p.window) * BN : 0;
    mbar_arrive_expect_tx(&k_full[0], kTileBytes);
    tma_load_4d(sm + kOffK, &tmk, 0, key_first, hk, b, &k_full[0], pol_kv);
    tma_load_4d(sm + kOffK + kBox, &tmk, 64, key_first, hk, b, &k_full[0], pol_kv);
    mbar_arrive_expect_tx(&v_full[0], kTileBytes);
    tma_load_4d(sm + kOffV, &tmv, 0, key_first, hk, b, &v_full[0], pol_kv);
    tma_load_4d(sm + kOffV + kBox, &tmv, 64, key_first, hk, b, &v_full[0], pol_kv);
  }

  // ---- visibility of the rows (integers) ----
  int len = p.seqlens[b * p.sl_s];
  len = len < 0 ? 0 : (len > p.Tmax ? p.Tmax : len);
  int my_end = 0, my_start = 0;
  bool my_row = false;
  const int row_i = i0 + (int)(threadIdx.x & 127);
  if (warp < 8 && row_i < p.Tq) {
    const int pos = p.qpos[b * p.qp_sb + row_i * p.qp_si];
    my_end = pos < 0 ? 0 : (pos >= len ? len : pos + 1);
    my_row = true;
    if constexpr (WIN) {
      // sliding window: keys pos - W < j <= pos (pos >= 0 first: no overflow)
      my_start = pos < 0 ? 0 : max(0, pos - p.window + 1);
      if (my_end > my_start) {
        atomicMin(&misc[6 + 2 * x], my_start);
        atomicMax(&misc[7 + 2 * x], my_start);
      } else {
        // a window that starts at or past the cache length holds no key: the
        // row is masked by its end on every tile, like a row at pos < 0
        my_end = 0;
      }
    }
    atomicMax(&misc[1 + 2 * x], my_end);
    atomicMin(&misc[2 + 2 * x], my_end);
  }
  __syncthreads();
  // key tiles [f_x, e_x) of query tile x (f_x = 0 without a window), and the
  // CTA's range [j_lo, j_hi) over the query tiles that see any key; ring
  // slots and phases count from j_lo
  int e_t0 = (misc[1] + BN - 1) / BN;
  int e_t1 = (misc[3] + BN - 1) / BN;
  int f_t0 = 0, f_t1 = 0;
  if constexpr (WIN) {
    f_t0 = misc[6] == 0x7fffffff ? e_t0 : misc[6] / BN;
    f_t1 = misc[8] == 0x7fffffff ? e_t1 : misc[8] / BN;
    if (f_t0 >= e_t0) f_t0 = e_t0 = 0;  // no row of the tile sees a key
    if (f_t1 >= e_t1) f_t1 = e_t1 = 0;
  }
  const int n_t0 = e_t0 - f_t0;  // key tiles per query tile
  const int n_t1 = e_t1 - f_t1;
  const int j_lo = !WIN ? 0 : (n_t0 == 0 ? f_t1 : (n_t1 == 0 ? f_t0 : min(f_t0, f_t1)));
  const int j_hi = max(e_t0, e_t1);
  const int n_max = j_hi - j_lo;  // key tiles the CTA loads
  // ring position of the CTA's key tile j: j + ro (ro = 1 when the copy made
  // before the positions were read holds another tile)
  const int ro = (WIN && j_lo != spec_first_tile(2 * pair * BM, p.window)) ? 1 : 0;
  const int cta_end = max(n_t0 > 0 ? misc[1] : 0, n_t1 > 0 ? misc[3] : 0);
  const int64_t out_row = (int64_t)b * p.o_sb + (int64_t)h * p.o_sh + (int64_t)row_i * p.o_si;
  const int64_t lse_idx = (int64_t)b * p.l_sb + (int64_t)h * p.l_sh + (int64_t)row_i * p.l_si;

  auto write_empty_row = [&]() {  // the defined output of a row with no visible key
    for (int d = 0; d < D; ++d) {
      if (p.out_bf16)
        static_cast<__nv_bfloat16*>(p.out)[out_row + (int64_t)d * p.o_sd] = __float2bfloat16_rn(0.f);
      else
        static_cast<float*>(p.out)[out_row + (int64_t)d * p.o_sd] = 0.f;
    }
    p.lse[lse_idx] = kNegInf;
  };
  const uint32_t tb = static_cast<uint32_t>(misc[0]);
  const uint32_t sQ = smem_u32(sm + kOffQ);
  const uint32_t sK = smem_u32(sm + kOffK);
  const uint32_t sV = smem_u32(sm + kOffV);

  if (n_max == 0) {
    // no row of the CTA sees a key: the defined empty output; the first
    // copies must still land before the CTA exits
    if (my_row) write_empty_row();
    if (warp == kTmaWarp && lane == 0) {
      bool landed = mbar_wait(q_full, 0);
      landed = mbar_wait(&k_full[0], 0) && landed;
      landed = mbar_wait(&v_full[0], 0) && landed;
      if (!landed) record_error(p.err, kErrTimeout);
    }
  } else if (warp == kTmaWarp) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // Q and ring position 0 are in flight already; positions issued so far
      int k_issued = 1, v_issued = 1;
      bool ok = true;
      if (ro == 1) {
        // position 0 holds another tile: it lands, then its slot is released
        ok = mbar_wait(&k_full[0], 0) && mbar_wait(&v_full[0], 0);
        mbar_arrive(&k_empty[0]);
        mbar_arrive(&v_empty[0]);
      }
      for (int j = 1 - ro; j < n_max && ok; ++j) {
        const int u = j + ro;
        const int s = u % STAGES;
        const int key0 = (j_lo + j) * BN;
        if (u >= STAGES && !mbar_wait(&k_empty[s], ((u / STAGES) - 1) & 1)) { ok = false; break; }
        unsigned char* kd = sm + kOffK + s * kTileBytes;
        mbar_arrive_expect_tx(&k_full[s], kTileBytes);
        tma_load_4d(kd, &tmk, 0, key0, hk, b, &k_full[s], pol_kv);
        tma_load_4d(kd + kBox, &tmk, 64, key0, hk, b, &k_full[s], pol_kv);
        k_issued = u + 1;
        if (u >= STAGES && !mbar_wait(&v_empty[s], ((u / STAGES) - 1) & 1)) { ok = false; break; }
        unsigned char* vd = sm + kOffV + s * kTileBytes;
        mbar_arrive_expect_tx(&v_full[s], kTileBytes);
        tma_load_4d(vd, &tmv, 0, key0, hk, b, &v_full[s], pol_kv);
        tma_load_4d(vd + kBox, &tmv, 64, key0, hk, b, &v_full[s], pol_kv);
        v_issued = u + 1;
      }
      // every issued copy must land before the CTA can exit
      if (!mbar_wait(q_full, 0)) ok = false;
      for (int j = k_issued - STAGES < 0 ? 0 : k_issued - STAGES; j < k_issued; ++j)
        if (!mbar_wait(&k_full[j % STAGES], (j / STAGES) & 1)) ok = false;
      for (int j = v_issued - STAGES < 0 ? 0 : v_issued - STAGES; j < v_issued; ++j)
        if (!mbar_wait(&v_full[j % STAGES], (j / STAGES) & 1)) ok = false;
      if (!ok) {
        record_error(p.err, kErrTimeout);
        misc[5] = 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0);
      // S_jj = Q_t K_jj^T into query tile t's S buffer
      auto issue_qk = [&](int t, int jj) {
        // descriptors: only the start address moves (split-word form)
        const uint32_t klo = tc::desc_lo(sK + ((jj + ro) % STAGES) * kTileBytes, 16);
        const uint32_t qlo = tc::desc_lo(sQ + t * kTileBytes, 16);
        constexpr uint32_t kHi = tc::desc_hi(1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (uint32_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4);
          const uint64_t adesc = tc::desc_join(qlo + off, kHi);
          const uint64_t bdesc = tc::desc_join(klo + off, kHi);
          tc::mma_ss(tb + t * kTileCols + kColS, adesc, bdesc, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[t]);
      };
      // U_t += P_jj V_jj (P_hi, then P_lo on the tiles that split P);
      // `more`: U_t already holds a tile
      const int min_end[QT] = {misc[2], misc[4]};
      const int win_max[QT] = {WIN ? misc[7] : 0, WIN ? misc[9] : 0};
      auto issue_pv = [&](int t, int jj, bool more) {
        const uint32_t vlo = tc::desc_lo(sV + ((jj + ro) % STAGES) * kTileBytes, kBox);
        constexpr uint32_t kHi = tc::desc_hi(1024);
        const uint32_t tcol = tb + t * kTileCols;
        const int k0 = (j_lo + jj) * BN;
        const bool split = k0 + BN > min_end[t] || (WIN && k0 < win_max[t]);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          if (part == 1 && !split) break;
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            // B = V rows [16ks, 16ks+16) (keys, K) x 128 dims (N, two 64-dim boxes 16 KB apart)
            const uint64_t bdesc = tc::desc_join(vlo + (uint32_t)(ks * 16 * 128 >> 4), kHi);
            const uint32_t acol = tcol + kColS + part * kColPlo + 8 * ks;
            tc::mma_ts(tcol + kColO, acol, bdesc, kIdescPV, (more || part > 0 || ks > 0) ? 1u : 0u);
          }
        }
      };
      // (j counts the CTA's key tiles from j_lo; query tile t covers
      // [a_t, a_t + n_t) of them, a_t = 0 without a window)
      const int a_t0 = f_t0 - j_lo, a_t1 = f_t1 - j_lo;
      // prologue: the first scores of the query tiles that start at j_lo
      if (ok && !mbar_wait(&k_full[ro], 0)) ok = false;  // ring position ro < STAGES: phase 0
      if (ok) {
        tc::fence_after();
        if (n_t0 > 0 && a_t0 == 0) issue_qk(0, 0);
        if (n_t1 > 0 && a_t1 == 0) issue_qk(1, 0);
        tc::commit(&k_empty[ro]);
      }
      for (int j = 0; ok && j < n_max; ++j) {
        const int u = j + ro;  // ring position
        const int s = u % STAGES;
        const bool next = j + 1 < n_max;
        if (!mbar_wait(&v_full[s], (u / STAGES) & 1)) { ok = false; break; }
        if (next && !mbar_wait(&k_full[(u + 1) % STAGES], ((u + 1) / STAGES) & 1)) { ok = false; break; }
        for (int t = 0; t < QT && ok; ++t) {
          const int nt = t == 0 ? n_t0 : n_t1;
          const int at = t == 0 ? a_t0 : a_t1;
          if (j < at || j >= at + nt) {
            // a query tile whose range starts at the next key tile: its first scores
            if (WIN && nt > 0 && j + 1 == at) issue_qk(t, j + 1);
            continue;
          }
          // U += P_j V_j as soon as this query tile's P_j is ready, then
          // S_{j+1} into the same TMEM columns (issue order = execution order)
          if (!mbar_wait(&p_full[t], (j - at) & 1)) { ok = false; break; }
          tc::fence_after();
          issue_pv(t, j, j > at);
          if (j + 1 < at + nt) issue_qk(t, j + 1);
        }
        if (!ok) break;
        tc::commit(&v_empty[s]);                           // V_j free once these products complete
        if (next) tc::commit(&k_empty[(u + 1) % STAGES]);  // K_{j+1} likewise
      }
      if (!ok) {
        record_error(p.err, kErrTimeout);
        misc[5] = 1;
      }
      // every MMA issued must complete before TMEM is released
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) {
        record_error(p.err, kErrTimeout);
        misc[5] = 1;
      }
    }
  } else {
    // ---------------- rows: online softmax statistics (query tile x) ----------------
    const int n_mine = x == 0 ? n_t0 : n_t1;
    const int my_min = misc[2 + 2 * x];
    const int f_mine = x == 0 ? f_t0 : f_t1;            // first key tile (0 without a window)
    const int win_max = WIN ? misc[7 + 2 * x] : 0;     // keys below it are masked for some row
    // a key tile some row of the query tile does not see in full (the
    // diagonal, a window's leading edge): P goes to the product as P_hi +
    // P_lo (the few-key rows live here); elsewhere as one bf16 P
    auto split_tile = [&](int k0) { return k0 + BN > my_min || (WIN && k0 < win_max); };
    if (n_mine == 0) {
      if (my_row) write_empty_row();
    } else {
      const uint32_t tl = tb + x * kTileCols + ((uint32_t)(32 * (warp & 3)) << 16);  // lane quarter
      float m_ref = kNegInf;  // reference maximum (base-2 units), -inf = no valid key yet
      float l = 0.f;
      bool ok = true;
      // waits are made warp-uniform: the tensor-memory accesses that follow
      // are warp-collective
      auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity));
      };
      for (int j = 0; j < n_mine; ++j) {
        if (!wait_all(&s_full[x], j & 1)) { ok = false; break; }
        tc::fence_after();
        float xs[128];
        {
          // all four 32-column loads in flight, one wait
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tc::ld32(tl + kColS, r0);
          tc::ld32(tl + kColS + 32, r1);
          tc::ld32(tl + kColS + 64, r2);
          tc::ld32(tl + kColS + 96, r3);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            xs[c] = __uint_as_float(r0[c]);
            xs[32 + c] = __uint_as_float(r1[c]);
            xs[64 + c] = __uint_as_float(r2[c]);
            xs[96 + c] = __uint_as_float(r3[c]);
          }
        }
        const int key0 = (f_mine + j) * BN;
        // the mask (select, diagonal tiles only) before any arithmetic
        if (key0 + BN > my_min) {
#pragma unroll
          for (int c = 0; c < 128; ++c) xs[c] = (key0 + c < my_end) ? xs[c] : kNegInf;
        }
        if constexpr (WIN) {
          // sliding window: keys before the row's first visible key
          if (key0 < win_max) {
#pragma unroll
            for (int c = 0; c < 128; ++c) xs[c] = (key0 + c >= my_start) ? xs[c] : kNegInf;
          }
        }
        // block maximum on the raw scores (scale > 0), a tree of short chains
        // (three-input max: 8 chains of 8 steps over 16 values each)
        float mx8[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mx8[c] = xs[c];
#pragma unroll
        for (int c = 8; c < 128; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], xs[c], xs[c + 1]);
        const float mraw = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float mt = (mraw == kNegInf) ? kNegInf : mraw * p.scale_log2;
        float alpha = 1.f;
        bool resc = false;
        if (mt != kNegInf) {
          if (m_ref == kNegInf) {
            m_ref = mt;  // first block with a valid key initialises the state
          } else if (mt > m_ref + kLazyRescale) {
            alpha = fast_exp2(m_ref - mt);
            m_ref = mt;
            l *= alpha;
            resc = true;
          }
        }
        if (__any_sync(0xffffffffu, resc)) {
          // U rows change reference (U += P_{j-1} V_{j-1} has completed: S_j
          // was issued after it)
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t r[32];
            tc::ld32(tl + kColO + 32 * q4, r);
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            tc::st32(tl + kColO + 32 * q4, r);
          }
        }
        // p = 2^(s * scale_log2 - m): masked entries are -inf and give exactly 0;
        // a row with no valid key yet has only masked entries in this tile.
        // Pairs of keys in float2 registers (packed fp32 arithmetic).
        const float m_use = (m_ref == kNegInf) ? 0.f : m_ref;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m_use, -m_use);
        const float2 neg1 = make_float2(-1.f, -1.f);
        float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        if (split_tile(key0)) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {  // 32 keys -> 16 columns of P_hi and of P_lo
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int k2 = 32 * q4 + 2 * c;
              const float2 e = __ffma2_rn(make_float2(xs[k2], xs[k2 + 1]), sc2, nm2);
              const float2 pp = make_float2(fast_exp2(e.x), fast_exp2(e.y));
              ls[c & 3] = __fadd2_rn(ls[c & 3], pp);
              // P = P_hi + P_lo: P_hi = the upper halves (truncation, exact),
              // P_lo = bf16(P - P_hi) (P - P_hi exact in fp32, below 2^-7 P)
              asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(hi[c]) : "r"(__float_as_uint(pp.x)), "r"(__float_as_uint(pp.y)));
              const float2 th = make_float2(__uint_as_float(__float_as_uint(pp.x) & 0xffff0000u),
                                            __uint_as_float(__float_as_uint(pp.y) & 0xffff0000u));
              const float2 rem = __ffma2_rn(th, neg1, pp);
              lo[c] = pack_bf16(rem.x, rem.y);
            }
            tc::st16(tl + kColS + 16 * q4, hi);
            tc::st16(tl + kColPlo + 16 * q4, lo);
          }
        } else {
          // every row sees every key of the tile: P rounded to bf16 (to
          // nearest) is the product's operand, and l sums the rounded values,
          // so u / l stays a convex combination of the values
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {  // 32 keys -> 16 columns of P
            uint32_t pb[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int k2 = 32 * q4 + 2 * c;
              const float2 e = __ffma2_rn(make_float2(xs[k2], xs[k2 + 1]), sc2, nm2);
              pb[c] = pack_bf16(fast_exp2(e.x), fast_exp2(e.y));
              ls[c & 3] = __fadd2_rn(ls[c & 3], make_float2(__uint_as_float(pb[c] << 16),
                                                            __uint_as_float(pb[c] & 0xffff0000u)));
            }
            tc::st16(tl + kColS + 16 * q4, pb);
          }
        }
        {
          const float2 a = __fadd2_rn(ls[0], ls[1]);
          const float2 c2 = __fadd2_rn(ls[2], ls[3]);
          const float2 t2 = __fadd2_rn(a, c2);
          l += t2.x + t2.y;
        }
        if (key0 + BN > cta_end) {
          // last tile of the CTA: zero the V rows past every visible key of
          // both query tiles (both may do it; the values are the same)
          const int u = f_mine - j_lo + j + ro;  // ring position of this key tile
          const int s = u % STAGES;
          if (!wait_all(&v_full[s], (u / STAGES) & 1)) { ok = false; break; }
          unsigned char* vt = sm + kOffV + s * kTileBytes;
          const int z0 = cta_end - key0;
          for (int idx = (int)(threadIdx.x & 127); idx < (BN - z0) * 16; idx += 128) {
            const int r = z0 + (idx >> 4);
            const int c = idx & 15;  // 16-byte chunk over the 128 dims (two boxes)
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kBox + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
      }
      // ---- epilogue: o = u / l, lse = m + ln l ----
      // `drain` completes once every MMA of the CTA has (single phase)
      if (ok && !wait_all(drain, 0)) ok = false;
      if (!ok) {
        if (lane == 0) {
          record_error(p.err, kErrTimeout);
          misc[5] = 1;
        }
      } else {
        tc::fence_after();
        const float inv = (m_ref == kNegInf) ? 0.f : 1.f / l;
        if (p.o_tma && !WIN) {
          // Every MMA has completed (drain), so the K (query tile 0) or V
          // (query tile 1) ring is free.  Each warp stages its 32 rows, 64
          // dims at a time (rows padded to 68 floats: conflict-free both
          // ways), and stores them back 16 lanes to a row (256 contiguous
          // bytes per row per store instruction).  (Measured against the
          // tiled-TMA form below: faster for full causal tiles, slower for
          // the short windowed CTAs, which keep TMA.)
          constexpr int kRow = 68;
          float* stg = reinterpret_cast<float*>(sm + (x == 0 ? kOffK : kOffV) + (warp & 3) * 32 * kRow * 4);
          const int r0 = (2 * pair + x) * BM + 32 * (warp & 3);
          const int rows = min(32, p.Tq - r0);
          float* dst0 = static_cast<float*>(p.out) + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh + (int64_t)r0 * p.o_si;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
#pragma unroll 1
            for (int q2 = 0; q2 < 2; ++q2) {
              uint32_t r[32];
              tc::ld32(tl + kColO + 64 * half + 32 * q2, r);
              tc::wait_ld();
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(stg + lane * kRow + 32 * q2 + c) =
                    make_float4(__uint_as_float(r[c]) * inv, __uint_as_float(r[c + 1]) * inv,
                                __uint_as_float(r[c + 2]) * inv, __uint_as_float(r[c + 3]) * inv);
            }
            __syncwarp();
#pragma unroll 4
            for (int it = 0; it < 16; ++it) {
              const int rr = 2 * it + (lane >> 4);
              if (rr < rows)
                *reinterpret_cast<float4*>(dst0 + rr * p.o_si + 64 * half + 4 * (lane & 15)) =
                    *reinterpret_cast<const float4*>(stg + rr * kRow + 4 * (lane & 15));
            }
            __syncwarp();
          }
        } else if (p.o_tma) {
          // Every MMA has completed (drain), so the K (query tile 0) or V
          // (query tile 1) ring is free.  Each warp stages its 32 rows x 128
          // dims there as four 4 KB boxes of 32 dims in the 128-byte swizzled
          // layout of the output map (16-byte chunk c of row r at c ^ (r mod
          // 8): conflict-free) and one lane stores them with tiled TMA.
          // One 32-dim box at a time (a short loop body for code that runs
          // once per CTA).
          unsigned char* stage = sm + (x == 0 ? kOffK : kOffV) + (warp & 3) * 4 * 4096;
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t r[32];
            tc::ld32(tl + kColO + 32 * q4, r);
            tc::wait_ld();
            float4* box = reinterpret_cast<float4*>(stage + q4 * 4096);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              box[lane * 8 + (c ^ (lane & 7))] =
                  make_float4(__uint_as_float(r[4 * c]) * inv, __uint_as_float(r[4 * c + 1]) * inv,
                              __uint_as_float(r[4 * c + 2]) * inv, __uint_as_float(r[4 * c + 3]) * inv);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // staged rows -> TMA
          __syncwarp();
          const int row_w = (2 * pair + x) * BM + 32 * (warp & 3);
          if (lane == 0 && row_w < p.Tq) {
            // rows past Tq are clipped by the map
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tma_store_4d(&tmo, stage + q4 * 4096, 32 * q4, row_w, h, b);
            bulk_commit();
          }
        } else {
          // the tensor-memory loads are warp-collective: every lane takes
          // part, rows past Tq store nothing
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t r[32];
            tc::ld32(tl + kColO + 32 * q4, r);
            tc::wait_ld();
            if (my_row) {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const float o = __uint_as_float(r[c]) * inv;
                const int64_t oi = out_row + (int64_t)(32 * q4 + c) * p.o_sd;
                if (p.out_bf16)
                  static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
                else
                  static_cast<float*>(p.out)[oi] = o;
              }
            }
          }
        }
        if (my_row) p.lse[lse_idx] = (m_ref == kNegInf) ? kNegInf : (m_ref + __log2f(l)) * kLn2;
        // the staging buffer is released with the CTA: the stores must have
        // read it (no-op for a lane without stores)
        if (WIN && p.o_tma && lane == 0) bulk_wait_read();
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tb, kTmemCols);
}

}  // namespace

int prefill_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill_tc(const FwdParams& p, int n_pairs, const CUtensorMap& tmq, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, const CUtensorMap& tmo, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    for (const void* f : {(const void*)prefill_tc_kernel<false>, (const void*)prefill_tc_kernel<true>}) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  const int64_t heads = (int64_t)p.Hq * p.B;
  if (p.head_group < 1) return cudaErrorInvalidValue;
  const int64_t groups = (heads + p.head_group - 1) / p.head_group;
  const int64_t blocks = groups * p.head_group * n_pairs;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (p.window > 0)
    prefill_tc_kernel<true><<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(p, tmq, tmk, tmv, tmo);
  else
    prefill_tc_kernel<false><<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(p, tmq, tmk, tmv, tmo);
  return cudaGetLastError();
}

}  // namespace blkattn
