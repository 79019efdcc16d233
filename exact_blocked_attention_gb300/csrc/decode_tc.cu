// Decode / verify kernel on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Exact blocked attention of a few query rows per KV head over a long cache
// ("Chapter 33: inference compute optimisation" §33.2, Algorithm 33.1 with
// the statistics (m, l, u) of eq. 33.3 and the merge rule of eqs.
// 33.4-33.5).  The G x T_q query rows that read one KV head form a "unit"
// (at most 48 rows; more rows make several row groups).  The unit's rows are
// the N dimension of the MMA and the keys sit on the 128 TMEM lanes:
//
//   S^T_j  = K_j Q^T       M = 128 keys, N = NR rows, K = 16 x 8
//                          (A = K tile, B = Q rows; both K-major in smem)
//   U^T   += V_j^T P_j^T   M = 128 value dims, N = 2 NR or 64 + NR, K = 16 x 8
//                          (A = the V tile read MN-major, B = P^T in smem)
//
// so a tile of 128 keys costs 16 MMAs whatever the row count.  P is not an
// input: each P^T row is written as bf16 P_hi (columns [0, NR)) and
// P_lo = bf16(P - P_hi) (columns [NR, 2 NR) of the same 64-column atom for up
// to 32 rows, else the same columns of a second atom), P_hi the truncated
// upper half of P; one product gives U_hi and U_lo side by side and
// U = U_hi + U_lo keeps ~2^-17 relative accuracy of P while V stays bf16 and
// is read once.
//
// Work split: the key tiles of all units, in the order (sequence, KV head,
// row group, tile), are cut into P = min(gridDim.x, tiles) equal contiguous
// non-empty ranges, one per CTA (one CTA per SM).  A unit whose tiles lie in
// one CTA is finished in place; otherwise each CTA writes its partial state
// of the unit to workspace slot (CTA index + unit index), counts itself in
// the unit's counter, and the last CTA to arrive folds the unit's partial
// states (no second kernel, no CTA ever waits for another).
// The tile counts come from the device-resident lengths and positions, so
// every CTA streams the same number of tiles whatever the length mix, and no
// SM idles at the end.
//
// Roles (352 threads):
//  * warps 0-7: key threads.  Thread k of lane quarter k / 32 owns key k of
//    the current tile (TMEM lane k); the two warps of a quarter split the NR
//    rows in halves.  A thread reads the scores of its key for its rows,
//    applies the mask by select (cache length, logical position, additive
//    bias with -inf = masked), and writes its part of the P^T row; per unit
//    it then owns value dim k of its rows for the epilogue.
//  * warp 8: producer: K and V tiles of 128 keys x 128 dims by tiled TMA
//    into a ring of 5 slots of 32 KB (4 with 48 rows; K_j and V_j alternate).
//  * warp 10: unit loader: per unit, the query rows (16-byte loads into the
//    128-byte swizzled K-major layout) and the rows' integer facts, into one
//    of two buffers, ahead of the unit's first product.
//  * warp 9: TMEM allocation and the one thread that issues every MMA, in
//    the order S_0, S_1, U += P_0 V_0, S_2, U += P_1 V_1, ...: the scores of
//    tile j + 1 are computed while the key threads work on tile j.  S^T and
//    P^T have two buffers each (by tile parity).  A tcgen05.commit fires
//    once every earlier MMA of the thread has completed, so S_j ready
//    implies the product with P_{j-2} is done and P^T buffer (j mod 2) is
//    free; a rescale of U^T at tile j first waits for the product with
//    P_{j-1} (one more barrier, rarely needed).
//
// Statistics: every key thread keeps its own partial sums l over its keys
// for its rows; the reference maxima m (base-2 units) live in shared memory.
// Per tile the key threads vote (bar.red.or) whether any score exceeds
// its row's m by more than 8.  Only then (always on a unit's first tile)
// are the tile's row maxima reduced across the keys, m raised and l and U^T
// rescaled: with any common reference m >= (max - 8) the state represents
// the same set and every P <= 2^8.  Rows with no visible key keep the empty
// state (out = 0, lse = -inf).  V rows past the unit's last visible key in
// its last tile (cache padding, possibly NaN) are zero-filled before the
// product so that 0 * garbage never reaches U.
//
// Every wait is bounded (%globaltimer); on a timeout the CTA records the
// error word, stops issuing work, lets its own copies and products drain
// and frees its tensor memory.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace blkattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLazyRescale = 8.f;

constexpr int BK = 128;               // keys per tile (TMEM lanes of S^T)
constexpr int D = 128;                // head dim (TMEM lanes of U^T)
constexpr int kBox = BK * 128;        // 128 rows x 64 dims, bf16: 16 KB
constexpr int kSlotBytes = 2 * kBox;  // 128 rows x 128 dims
constexpr int kKeyWarps = 8;   // two warps per TMEM lane quarter, each with half of the rows
constexpr int kKeyThreads = 32 * kKeyWarps;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kLoadWarp = 10;
constexpr int kThreads = 32 * 11;
constexpr int kBarRows = 1;  // named barrier of the key threads
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S^T of tiles with even / odd index: +0 / +64
constexpr uint32_t kColU = 128;  // U^T of units with even / odd index: +0 / +128;
                                 // the P_hi part in columns [0, NR), P_lo from column kLo

// Integer facts of the rows of one unit (written by the producer).
template <int NR>
struct RowFacts {
  int64_t boff[NR];  // bias row offsets (elements)
  int64_t ooff[NR];  // output row offsets
  int64_t loff[NR];  // lse offsets
  uint64_t tree[NR]; // token tree: bit k = the row sees key tree_base + k (all ones without a tree);
                     // with a sliding window instead: the row's first visible key
  int end[NR];       // visible keys are [0, end): min(len, pos + 1), 0 for padding rows
  int unit_end;      // max over the rows
  int min_end;       // min over the real rows
  int tree_base;     // first key of the token tree (len - T_q); INT_MAX without a tree
  int win_max;       // sliding window: the largest first visible key of the rows (0 without)
};

template <int NR>
struct TcLayout {
  // Up to 32 rows, P_hi and P_lo share one 64-column atom (P_lo from column
  // NR, the product's N = 2 NR), which leaves room for a fifth ring slot;
  // 48 rows take two atoms (P_lo from column 64, N = 64 + NR) and four slots.
  static constexpr bool kPacked = NR <= 32;
  static constexpr int kSlots = kPacked ? 5 : 4;
  static constexpr int kLo = kPacked ? NR : 64;          // column of P_lo / U_lo
  static constexpr int kPVN = kPacked ? 2 * NR : 64 + NR;  // N of the PV product
  static constexpr int kPBytes = kPacked ? kBox : 2 * kBox;  // one P^T buffer
  static constexpr int kQBox = NR * 128;  // NR rows x 64 dims
  static constexpr int kQBytes = 2 * kQBox;
  static constexpr int kOffRing = 0;
  static constexpr int kOffQ = kSlots * kSlotBytes;              // two query buffers
  static constexpr int kOffP = kOffQ + 2 * kQBytes;              // two P^T buffers
  static constexpr int kOffRows = kOffP + 2 * kPBytes;           // RowFacts[2]
  static constexpr int kRowsBytes = (int)((sizeof(RowFacts<NR>) + 15) / 16 * 16);
  static constexpr int kOffNTab = kOffRows + 2 * kRowsBytes;     // uint16 tiles per (sequence, row group)
  static constexpr int kOffRed = kOffNTab + kDecodeTcMaxEntries * 2;  // float [4][NR]
  // float [NR] each: m, m_use, thr, alpha of the current unit; m, l, 1 / l
  // of the finished unit whose U readout is pending
  static constexpr int kOffStat = kOffRed + 4 * NR * 4;
  static constexpr int kOffBar = kOffStat + 7 * NR * 4;
  // full[kSlots], empty[kSlots], q_full[2], q_empty[2], s_full[2], p_full[2], u_full[2],
  // pv_done, drain
  static constexpr int kNumBars = 2 * kSlots + 2 + 2 + 2 + 2 + 2 + 1 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 128 + 1024;  // + slack to align to 1024
  static_assert(kOffQ % 1024 == 0 && kQBox % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms");
  static_assert(kOffBar % 8 == 0 && kOffStat % 16 == 0, "alignment");
  static_assert(kBytes <= 232448, "shared memory per block");
};

// The CTA's start in the tile order (written once by warp 0).
struct Start {
  long long t0, t1, W, P, su;
  int b, kvh, rg, j;
};

// Position in the tile order: global tile t of unit (b, kvh, rg), local tile
// j of n, the unit's first global tile su.  Each unit spans n real tiles and
// `extra` weight-only tiles after them (the partition charges a unit for its
// set-up and readout, so CTAs holding many short units get fewer tiles).
struct Cursor {
  int64_t t, su;
  int b, kvh, rg, j, n;
  int extra;
  int s0;               // the unit's first tile (sliding window; 0 otherwise)
  const uint16_t* st;   // per-unit first tiles, or nullptr
  __device__ __forceinline__ int key0() const { return (s0 + j) * BK; }
  // to the first tile of the next unit
  __device__ __forceinline__ void step_unit(const uint16_t* ntab, int RG, int Hkv, int B) {
    su += n + extra;
    t = su;
    j = 0;
    if (++rg == RG) {
      rg = 0;
      if (++kvh == Hkv) {
        kvh = 0;
        ++b;
      }
    }
    n = (b < B) ? (int)ntab[b * RG + rg] : 1;
    s0 = (b < B && st != nullptr) ? (int)st[b * RG + rg] : 0;
  }
  __device__ __forceinline__ void next(const uint16_t* ntab, int RG, int Hkv, int B) {
    if (j + 1 == n) {
      step_unit(ntab, RG, Hkv, B);
    } else {
      ++t;
      ++j;
    }
  }
};

// CTA whose range [c W / P, (c + 1) W / P) holds global tile t.
// (32-bit arithmetic: the host keeps the tile count below 2^24 and
// P <= 255, so (t + 1) P < 2^32; a 64-bit division is a long software
// sequence on the GPU.)
__device__ __forceinline__ int64_t cta_of(int64_t t, int64_t W, int64_t P) {
  const uint32_t w = (uint32_t)W;
  return (int64_t)((((uint32_t)t + 1u) * (uint32_t)P + w - 1u) / w) - 1;
}

// N consecutive TMEM columns of this thread's lane (N = 8, 16 or 24; the
// column offset is a multiple of 8, of 16 for N = 16) -> floats.
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&x)[N]) {
  uint32_t r[N];
  if constexpr (N == 16) {
    tc::ld16(taddr, &r[0]);
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 8) tc::ld8(taddr + c, &r[c]);
  }
  tc::wait_ld();
#pragma unroll
  for (int c = 0; c < N; ++c) x[c] = __uint_as_float(r[c]);
}

template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const float (&x)[N]) {
  uint32_t r[N];
#pragma unroll
  for (int c = 0; c < N; ++c) r[c] = __float_as_uint(x[c]);
  if constexpr (N == 16) {
    tc::st16(taddr, &r[0]);
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 8) tc::st8(taddr + c, &r[c]);
  }
}

// Reduce NH values per lane across the 32 lanes of a warp (NH = 8, 16, 24):
// three reduce-scatter steps (xor 16, 8, 4) halve the values a lane keeps,
// two full steps (xor 2, 1) finish them.  Afterwards lane l holds the
// results for rows base + i, i < NH / 8, base = (l >> 4 & 1) NH / 2 +
// (l >> 3 & 1) NH / 4 + (l >> 2 & 1) NH / 8, in v[0 .. NH / 8).  The
// shuffles of one step are independent (27 in all for NH = 24).
template <int NH, bool kMax>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[NH], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
#pragma unroll
  for (int step = 0; step < 3; ++step) {
    const int off = 16 >> step;
    const int half = NH >> (step + 1);  // values kept after this step
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
#pragma unroll
  for (int off = 2; off >= 1; off >>= 1)
#pragma unroll
    for (int i = 0; i < NH / 8; ++i) v[i] = op(v[i], __shfl_xor_sync(0xffffffffu, v[i], off));
}

template <int NH>
__device__ __forceinline__ int scatter_base(int lane) {
  return ((lane >> 4) & 1) * (NH / 2) + ((lane >> 3) & 1) * (NH / 4) + ((lane >> 2) & 1) * (NH / 8);
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  using L = TcLayout<NR>;
  constexpr uint32_t kIdescQK = tc::idesc_bf16(128, NR, 0, 0);  // K, Q both K-major
  // V^T, P^T both MN-major; N spans the P_hi atom (NR used of 64) and the P_lo atom
  constexpr uint32_t kIdescPV = tc::idesc_bf16(128, L::kPVN, 1, 1);
  constexpr int kSlots = L::kSlots;
  // weight-only tiles per unit in the partition (its set-up and readout)
  constexpr int kUnitExtra = NR >= 48 ? 2 : 0;  // measured best: 48-row units pay a real set-up cost
  constexpr int kPBytes = L::kPBytes;
  constexpr uint32_t kLo = L::kLo;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  RowFacts<NR>* facts0 = reinterpret_cast<RowFacts<NR>*>(sm + L::kOffRows);
  uint16_t* ntab = reinterpret_cast<uint16_t*>(sm + L::kOffNTab);
  // sliding window: the units' first tiles in the upper half of the table
  // (window calls have at most kDecodeTcMaxEntries / 2 units)
  uint16_t* stab = ntab + kDecodeTcMaxEntries / 2;
  float* red = reinterpret_cast<float*>(sm + L::kOffRed);
  float* s_m = reinterpret_cast<float*>(sm + L::kOffStat);  // reference maximum, -inf = none yet
  float* s_muse = s_m + NR;                                  // m, or 0 when none yet
  float* s_thr = s_m + 2 * NR;                               // m + 8, -inf when none yet
  float* s_alpha = s_m + 3 * NR;
  float* s_mfin = s_m + 4 * NR;
  float* s_lfin = s_m + 5 * NR;
  float* s_inv = s_m + 6 * NR;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = full + kSlots;
  uint64_t* q_full = empty + kSlots;  // [2]
  uint64_t* q_empty = q_full + 2;     // [2]
  uint64_t* s_full = q_empty + 2;     // [2] by tile parity
  uint64_t* p_full = s_full + 2;      // [2] by tile parity
  uint64_t* u_full = p_full + 2;      // [2] by unit parity
  uint64_t* pv_done = u_full + 2;     // once per U += P V product
  uint64_t* drain = pv_done + 1;
  // misc: [0] tmem base, [1] error seen by the producer / MMA thread,
  // [2] abort of the key threads, [3] "this CTA folds the unit" (both
  // written before a barrier of the key threads, read after it)
  int* misc = reinterpret_cast<int*>(sm + L::kOffMisc);
  Start* start = reinterpret_cast<Start*>(sm + L::kOffMisc + 64);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int RG = p.row_groups;
  const int R = p.rows_cta;
  const int B = p.B;
  const int Hkv = p.Hkv;

  // ---------------- schedule: tiles per (sequence, row group) ----------------
  {
    int* nb = reinterpret_cast<int*>(sm + L::kOffP);  // per-sequence totals (P^T area, start-up only)
    const int E = B * RG;
    for (int e = threadIdx.x; e < E; e += kThreads) {
      const int b = e / RG;
      const int rg = e - b * RG;
      // the row end min(len, pos + 1) (0 for pos < 0) grows with pos, so the
      // unit's end follows from the largest position of its rows; all loads
      // are independent (one round trip)
      const int len_raw = p.seqlens[b * p.sl_s];
      const int pk0 = rg * R;
      const int pk1 = min(pk0 + R, p.rows_per_head);
      int maxpos = -1, minpos = 0x7fffffff;  // minpos over the rows that see keys
      if (pk1 - pk0 >= p.Tq) {
#pragma unroll 4
        for (int i = 0; i < p.Tq; ++i) {
          const int ps = p.qpos[b * p.qp_sb + i * p.qp_si];
          maxpos = max(maxpos, ps);
          if (ps >= 0) minpos = min(minpos, ps);
        }
      } else {
#pragma unroll 4
        for (int pk = pk0; pk < pk1; ++pk) {
          const int ps = p.qpos[b * p.qp_sb + (pk % p.Tq) * p.qp_si];
          maxpos = max(maxpos, ps);
          if (ps >= 0) minpos = min(minpos, ps);
        }
      }
      const int len = len_raw < 0 ? 0 : (len_raw > p.Tmax ? p.Tmax : len_raw);
      const int uend = maxpos < 0 ? 0 : min(maxpos + 1, len);
      // sliding window: the unit starts at the tile of its earliest visible key
      const int s0 = (p.window > 0 && minpos != 0x7fffffff) ? max(0, minpos - p.window + 1) / BK : 0;
      const int n = (uend + BK - 1) / BK - s0;
      ntab[e] = (uint16_t)(n < 1 ? 1 : n);  // an all-empty unit still takes one (masked) tile
      if (p.window > 0) stab[e] = (uint16_t)s0;
    }
    if (threadIdx.x == 0) {
      misc[1] = 0;
      misc[2] = 0;
      for (int s = 0; s < kSlots; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int x = 0; x < 2; ++x) {
        mbar_init(&q_full[x], 1);
        // query buffer x is free once the unit's last S product completed
        // (MMA commit) and its row facts are no longer read (key threads)
        mbar_init(&q_empty[x], 2);
        mbar_init(&u_full[x], 1);
      }
      for (int x = 0; x < 2; ++x) {
        mbar_init(&s_full[x], 1);
        mbar_init(&p_full[x], kKeyWarps);  // one arrival per key warp
      }
      mbar_init(pv_done, 1);
      mbar_init(drain, 1);
      fence_barrier_init();
    }
    if (threadIdx.x < NR) {
      s_m[threadIdx.x] = kNegInf;
      s_muse[threadIdx.x] = 0.f;
      s_thr[threadIdx.x] = kNegInf;
    }
    if (warp == kMmaWarp) {
      tc::alloc(reinterpret_cast<uint32_t*>(&misc[0]), kTmemCols);
      tc::relinquish();
    }
    __syncthreads();
    for (int b = threadIdx.x; b < B; b += kThreads) {
      int s = 0;
      for (int rg = 0; rg < RG; ++rg) s += ntab[b * RG + rg] + kUnitExtra;
      nb[b] = s;
    }
    __syncthreads();
    if (warp == 0) {
      // tiles of sequence b: Hkv * nb[b]; lane l sums a contiguous run of sequences
      const int per = (B + 31) / 32;
      const int b0 = min(lane * per, B);
      const int b1 = min(b0 + per, B);
      long long s = 0;
      for (int b = b0; b < b1; ++b) s += (long long)nb[b] * Hkv;
      long long incl = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const long long W = __shfl_sync(0xffffffffu, incl, 31);
      // with fewer tiles than CTAs the last CTAs stay idle, so that every
      // working CTA has a tile and the CTAs holding one unit are consecutive
      const long long P = W < (long long)gridDim.x ? W : (long long)gridDim.x;
      const bool works = (long long)blockIdx.x < P;
      // c W / P in 32 bits: W = q P + r, c W / P = c q + c r / P (c r < 2^16)
      const uint32_t q = (uint32_t)W / (uint32_t)(P > 0 ? P : 1), r = (uint32_t)W - q * (uint32_t)P;
      const uint32_t c = blockIdx.x;
      const long long t0 = works ? (long long)(c * q + c * r / (uint32_t)P) : W;
      const long long t1 = works ? (long long)((c + 1) * q + (c + 1) * r / (uint32_t)P) : W;
      const long long excl = incl - s;
      const unsigned own = __ballot_sync(0xffffffffu, t0 < t1 && excl <= t0 && t0 < incl);
      if (lane == 0) {
        start->t0 = t0;
        start->t1 = t1;
        start->W = W;
        start->P = P;
      }
      if (own != 0 && lane == __ffs(own) - 1) {
        long long pre = excl;
        int b = b0;
        while (pre + (long long)nb[b] * Hkv <= t0) {
          pre += (long long)nb[b] * Hkv;
          ++b;
        }
        const long long o = t0 - pre;
        const int kvh = (int)((uint32_t)o / (uint32_t)nb[b]);
        long long o2 = o - (long long)kvh * nb[b];
        long long su = pre + (long long)kvh * nb[b];
        int rg = 0;
        while (o2 >= ntab[b * RG + rg] + kUnitExtra) {
          o2 -= ntab[b * RG + rg] + kUnitExtra;
          su += ntab[b * RG + rg] + kUnitExtra;
          ++rg;
        }
        start->b = b;
        start->kvh = kvh;
        start->rg = rg;
        start->j = (int)o2;
        start->su = su;
      }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }
  const int64_t t0 = start->t0;
  const int64_t t1 = start->t1;
  const int64_t W = start->W;
  const int64_t P_work = start->P;  // CTAs that hold tiles: [0, P_work)
  const uint32_t tb = static_cast<uint32_t>(misc[0]);
  const uint32_t sRing = smem_u32(sm + L::kOffRing);
  const uint32_t sQ = smem_u32(sm + L::kOffQ);
  const uint32_t sP = smem_u32(sm + L::kOffP);
  Cursor cur;
  cur.t = t0;
  cur.su = start->su;
  cur.b = start->b;
  cur.kvh = start->kvh;
  cur.rg = start->rg;
  cur.j = start->j;
  cur.n = (t0 < t1) ? (int)ntab[cur.b * RG + cur.rg] : 1;
  cur.extra = kUnitExtra;
  cur.st = p.window > 0 ? stab : nullptr;
  cur.s0 = (t0 < t1 && cur.st != nullptr) ? (int)stab[cur.b * RG + cur.rg] : 0;
  // a range may start among a unit's weight-only tiles: begin at the next unit
  if (t0 < t1 && cur.j >= cur.n) cur.step_unit(ntab, RG, Hkv, B);

  if (warp == kTmaWarp) {
    // ---------------- producer: K and V tiles ----------------
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
      int64_t issued = 0;
      bool ok = true;
      // g counts this CTA's tiles (positions skip the weight-only tiles)
      for (int64_t g = 0; ok && cur.t < t1; cur.next(ntab, RG, Hkv, B), ++g) {
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const int64_t seq = 2 * g + kv;
          const int s = (int)(seq % kSlots);
          if (seq >= kSlots && !mbar_wait(&empty[s], (uint32_t)(((seq / kSlots) - 1) & 1))) {
            ok = false;
            break;
          }
          unsigned char* dst = sm + L::kOffRing + s * kSlotBytes;
          const void* map = kv ? static_cast<const void*>(&tmv) : static_cast<const void*>(&tmk);
          mbar_arrive_expect_tx(&full[s], kSlotBytes);
          tma_load_4d(dst, map, 0, cur.key0(), cur.kvh, cur.b, &full[s], pol);
          tma_load_4d(dst + kBox, map, 64, cur.key0(), cur.kvh, cur.b, &full[s], pol);
          issued = seq + 1;
        }
        // after the first tile, let the first unit's query rows land before
        // the stream fills the memory queues (they gate the first product)
        if (ok && g == 0 && !mbar_wait(&q_full[0], 0)) ok = false;
      }
      // every issued copy must land before the CTA exits
      for (int64_t seq = issued - kSlots < 0 ? 0 : issued - kSlots; seq < issued; ++seq)
        if (!mbar_wait(&full[seq % kSlots], (uint32_t)((seq / kSlots) & 1))) ok = false;
      if (!ok) {
        record_error(p.err, kErrTimeout);
        misc[1] = 1;
      }
    }
  } else if (warp == kLoadWarp) {
    // ---------------- unit loader: query rows and row facts ----------------
    int uidx = 0;
    bool ok = true;
    for (; t0 < t1 && cur.su < t1; cur.step_unit(ntab, RG, Hkv, B), ++uidx) {
      const int qb = uidx & 1;
      if (uidx >= 2) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&q_empty[qb], (uint32_t)(((uidx >> 1) - 1) & 1));
        if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
      }
      // lane l describes rows l and l + 32 (one division each), then every
      // global load of the unit is issued before any is used (one round
      // trip): cache length, positions, query rows
      unsigned char* qs = sm + L::kOffQ + qb * L::kQBytes;
      const int b = cur.b;
      const int len_raw = p.seqlens[b * p.sl_s];
      bool real[2];
      int hrow[2], irow[2], pos[2] = {-1, -1};
      const __nv_bfloat16* qrow[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int r = lane + 32 * h2;
        const int pk = cur.rg * R + r;
        real[h2] = r < NR && r < R && pk < p.rows_per_head;
        const int g = real[h2] ? pk / p.Tq : 0;
        irow[h2] = real[h2] ? pk - g * p.Tq : 0;
        hrow[h2] = cur.kvh * p.G + g;
        qrow[h2] = static_cast<const __nv_bfloat16*>(p.q) + (int64_t)b * p.q_sb + (int64_t)hrow[h2] * p.q_sh +
                   (int64_t)irow[h2] * p.q_si;
        if (real[h2]) pos[h2] = p.qpos[b * p.qp_sb + irow[h2] * p.qp_si];
        if (real[h2] && p.bias != nullptr) {
          // the bias of the unit's first tile into L2 now (new rows miss)
          const int64_t bo = (int64_t)b * p.bi_sb + (int64_t)hrow[h2] * p.bi_sh + (int64_t)irow[h2] * p.bi_si;
          const int j0 = cur.key0();
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int key = j0 + 32 * q4;
            if (key < p.Tmax) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.bias + bo + (int64_t)key * p.bi_sj));
          }
        }
      }
      // query rows, 128-byte swizzled K-major (rows of 64 dims), by 16-byte
      // asynchronous copies that bypass the registers: all of them are in
      // flight at once whatever the row count (rows past the unit's end are
      // zero-filled); they complete before the rows are announced below
#pragma unroll
      for (int it = 0; it < NR / 2; ++it) {
        // chunk (lane & 15) of row 2 it + (lane >> 4), described by lane (row & 31)
        const int r = 2 * it + (lane >> 4);
        const int c = lane & 15;
        const int set = (2 * it) >> 5;  // rows of this iteration are all < 32 or all >= 32
        const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(qrow[set]), r & 31));
        const bool rr = __shfl_sync(0xffffffffu, real[set], r & 31);
        cp_async_16(smem_u32(qs + (c >> 3) * L::kQBox + r * 128 + (((c & 7) ^ (r & 7)) << 4)),
                    rr ? static_cast<const void*>(reinterpret_cast<const uint4*>(src) + c) : p.q, rr ? 16u : 0u);
      }
      // integer facts of the rows
      const int len = len_raw < 0 ? 0 : (len_raw > p.Tmax ? p.Tmax : len_raw);
      RowFacts<NR>& rf = facts0[qb];
      int umax = 0, umin = 0x7fffffff, wmax = 0;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int r = lane + 32 * h2;
        if (r >= NR) break;
        int e = 0;
        int64_t bo = 0, oo = 0, lo = 0;
        uint64_t tr = ~0ull;
        if (real[h2]) {
          const int h = hrow[h2], i = irow[h2];
          e = pos[h2] < 0 ? 0 : min(pos[h2] + 1, len);
          if (p.tree != nullptr) tr = (uint64_t)p.tree[(int64_t)b * p.tr_sb + (int64_t)i * p.tr_si];
          if (p.window > 0) {  // the row's first visible key (no overflow: pos >= 0 first)
            tr = (uint64_t)(pos[h2] < 0 ? 0 : max(0, pos[h2] - p.window + 1));
            wmax = max(wmax, (int)tr);
          }
          bo = (int64_t)b * p.bi_sb + (int64_t)h * p.bi_sh + (int64_t)i * p.bi_si;
          oo = (int64_t)b * p.o_sb + (int64_t)h * p.o_sh + (int64_t)i * p.o_si;
          lo = (int64_t)b * p.l_sb + (int64_t)h * p.l_sh + (int64_t)i * p.l_si;
          umin = min(umin, e);
        }
        umax = max(umax, e);
        rf.end[r] = e;
        rf.tree[r] = tr;
        rf.boff[r] = bo;
        rf.ooff[r] = oo;
        rf.loff[r] = lo;
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        umax = max(umax, __shfl_xor_sync(0xffffffffu, umax, off));
        umin = min(umin, __shfl_xor_sync(0xffffffffu, umin, off));
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
      }
      if (lane == 0) {
        rf.unit_end = umax;
        rf.min_end = umin;
        rf.tree_base = p.tree != nullptr ? len - p.Tq : 0x7fffffff;
        rf.win_max = wmax;
      }
      cp_async_wait_all();  // this lane's query-row copies have landed
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q rows -> tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[qb]);
    }
    if (!ok && lane == 0) {
      record_error(p.err, kErrTimeout);
      misc[1] = 1;
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue (one thread) ----------------
    // Order S_0, S_1, U += P_0 V_0, S_2, U += P_1 V_1, ...: the products of
    // the next tile's scores run while the key threads work on this tile.
    if (lane == 0) {
      Cursor cq = cur;  // tile of the next S product
      int uq = 0, up = 0;  // unit counters of the S and the U sides
      // Ring positions of the next K (even entries) and V (odd entries)
      // tiles: slot and phase advance by two entries per tile, without
      // divisions on this thread's path.
      struct RingPos {
        uint32_t slot, phase;
        __device__ void adv2() {
          slot += 2;
          if (slot >= (uint32_t)kSlots) {
            slot -= (uint32_t)kSlots;
            phase ^= 1u;
          }
        }
      };
      RingPos kpos{0u, 0u}, vpos{1u, 0u};
      constexpr uint32_t kHi = tc::desc_hi(1024);
      // shared-memory descriptors: only the address word moves per MMA
      const uint32_t qlo0 = tc::desc_lo(sQ, 16);
      auto issue_qk = [&](int64_t gq) -> bool {
        const bool first = cq.t == t0 || cq.j == 0;
        const bool last = cq.t == t1 - 1 || cq.j == cq.n - 1;
        const int qb = uq & 1;
        if (first && !mbar_wait(&q_full[qb], (uint32_t)((uq >> 1) & 1))) return false;
        const uint32_t ks_slot = kpos.slot;
        if (!mbar_wait(&full[ks_slot], kpos.phase)) return false;
        kpos.adv2();
        tc::fence_after();
        // S^T = K_j Q^T into the S buffer of the tile's parity
        const uint32_t klo = tc::desc_lo(sRing + ks_slot * kSlotBytes, 16);
        const uint32_t qlo = qlo0 + (uint32_t)(qb * L::kQBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t adesc = tc::desc_join(klo + (uint32_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4), kHi);
          const uint64_t bdesc = tc::desc_join(qlo + (uint32_t)(((ks >> 2) * L::kQBox + (ks & 3) * 32) >> 4), kHi);
          tc::mma_ss(tb + kColS + 64u * (uint32_t)(gq & 1), adesc, bdesc, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[gq & 1]);
        tc::commit(&empty[ks_slot]);
        if (last) {
          tc::commit(&q_empty[qb]);
          ++uq;
        }
        cq.next(ntab, RG, Hkv, B);
        return true;
      };
      // (test hook: `drain` has no arrival before the thread's own commit
      // below, so this wait runs out)
      bool ok = blockIdx.x != (unsigned)p.test_stall_cta || mbar_wait_ns(drain, 0, 1000000ull);
      ok = ok && (!(cq.t < t1) || issue_qk(0));
      for (int64_t g = 0; ok && cur.t < t1; cur.next(ntab, RG, Hkv, B), ++g) {
        const bool first = cur.t == t0 || cur.j == 0;
        const bool last = cur.t == t1 - 1 || cur.j == cur.n - 1;
        if (cq.t < t1 && !issue_qk(g + 1)) { ok = false; break; }
        // U^T += V_j^T [P_hi | P_lo]^T once the key threads wrote P^T
        const uint32_t vs_slot = vpos.slot;
        if (!mbar_wait(&p_full[g & 1], (uint32_t)((g >> 1) & 1))) { ok = false; break; }
        if (!mbar_wait(&full[vs_slot], vpos.phase)) { ok = false; break; }
        vpos.adv2();
        tc::fence_after();
        const uint32_t vlo = tc::desc_lo(sRing + vs_slot * kSlotBytes, kBox);
        const uint32_t plo = tc::desc_lo(sP + (uint32_t)(g & 1) * kPBytes, kBox);
        const uint32_t ucol = tb + kColU + 128u * (uint32_t)(up & 1);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          // A = V^T: 128 dims (two 64-dim boxes 16 KB apart) x keys [16 ks, 16 ks + 16)
          const uint64_t adesc = tc::desc_join(vlo + (uint32_t)(ks * 2048 >> 4), kHi);
          // B = P^T: keys [16 ks, +16) x [P_hi | P_lo] (one atom, or two 16 KB apart)
          const uint64_t bdesc = tc::desc_join(plo + (uint32_t)(ks * 2048 >> 4), kHi);
          tc::mma_ss(ucol, adesc, bdesc, kIdescPV, (!first || ks > 0) ? 1u : 0u);
        }
        tc::commit(&empty[vs_slot]);
        tc::commit(pv_done);
        if (last) {
          tc::commit(&u_full[up & 1]);
          ++up;
        }
      }
      if (!ok) {
        record_error(p.err, kErrTimeout);
        misc[1] = 1;
      }
      // every MMA issued must complete before TMEM is released
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) {
        record_error(p.err, kErrTimeout);
        misc[1] = 1;
      }
    }
  } else {
    // ---------------- key threads ----------------
    // warp w: TMEM lane quarter (w mod 4), row half (w / 4): thread = key k
    // of the tile (value dim k in the epilogue), rows [c0, c0 + NH)
    constexpr int NH = NR / 2;
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int k = 32 * quarter + lane;
    const int c0 = half * NH;
    const uint32_t tl = tb + ((uint32_t)(32 * quarter) << 16);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    const bool has_bias = p.bias != nullptr;
    float lp[NH];  // this thread's partial sums of P over its keys
#pragma unroll
    for (int r = 0; r < NH; ++r) lp[r] = 0.f;
    int uidx = 0;
    bool ok = true;
    // A finished unit's U is read one tile later, after the next tile's P:
    // by then its last product has completed and the readout does not stall
    // the pipeline.  Its m, l and 1 / l wait in s_mfin / s_lfin / s_inv, its
    // row facts stay in their buffer until the readout releases them.
    bool pend = false;
    int pend_uidx = 0, pend_b = 0, pend_kvh = 0, pend_rg = 0, pend_n = 1;
    int64_t pend_su = 0;
    auto flush = [&]() -> bool {
      const int pb = pend_uidx & 1;
      const RowFacts<NR>& pf = facts0[pb];
      if (!bar_and(kBarRows, kKeyThreads, wait_all(&u_full[pb], (uint32_t)((pend_uidx >> 1) & 1)))) return false;
      tc::fence_after();
      float u[NH];
      {
        float ulo[NH];
        const uint32_t ua = tl + kColU + 128u * (uint32_t)pb + c0;
        ld_cols<NH>(ua, u);
        ld_cols<NH>(ua + kLo, ulo);
#pragma unroll
        for (int r = 0; r < NH; ++r) u[r] += ulo[r];  // U = P_hi V + P_lo V
      }
      const int64_t unit = ((int64_t)pend_b * Hkv + pend_kvh) * RG + pend_rg;
      const int64_t cf = cta_of(pend_su, W, P_work);
      const int64_t cl = cta_of(pend_su + pend_n - 1, W, P_work);
      const int nparts = (int)(cl - cf + 1);
      const int rr = min(R, p.rows_per_head - pend_rg * R);  // real rows of the unit
      if (nparts == 1) {
#pragma unroll
        for (int r = 0; r < NH; ++r) {
          const int row = c0 + r;
          if (row >= rr) break;
          const float o = (s_mfin[row] == kNegInf) ? 0.f : u[r] * s_inv[row];
          const int64_t oi = pf.ooff[row] + (int64_t)k * p.o_sd;
          if (p.out_bf16)
            static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
          else
            static_cast<float*>(p.out)[oi] = o;
        }
        if (half == 0 && k < rr) {
          const float m = s_mfin[k];
          p.lse[pf.loff[k]] = (m == kNegInf) ? kNegInf : (m + __log2f(s_lfin[k])) * kLn2;
        }
      } else {
        // (kept in L2 until the fold reads it: the key stream passing through
        // meanwhile is marked evict-first)
        const uint64_t keep = policy_evict_last();
        // this CTA's partial state of the unit, then the last of the unit's
        // CTAs to get here folds all of them (eqs. 33.4-33.5, in CTA order)
        const int64_t slot = (int64_t)blockIdx.x + unit;
#pragma unroll
        for (int r = 0; r < NH; ++r) {
          const int row = c0 + r;
          if (row >= rr) break;
          st_global_hint(p.ws_u + ((slot * R + row) * D) + k, u[r], keep);
        }
        if (half == 0 && k < rr) {
          st_global_hint(p.ws_m + slot * R + k, s_mfin[k], keep);
          st_global_hint(p.ws_l + slot * R + k, s_lfin[k], keep);
        }
        __threadfence();  // the partial state is visible before the count says so
        bar_sync(kBarRows, kKeyThreads);
        if (threadIdx.x == 0)
          misc[3] = (atomicAdd(&p.unit_cnt[unit], 1u) == (unsigned)(nparts - 1)) ? 1 : 0;
        bar_sync(kBarRows, kKeyThreads);
        if (misc[3] != 0) {
          __threadfence();
          if (threadIdx.x == 0) p.unit_cnt[unit] = 0u;  // ready for the next launch
          const int64_t fs = cf + unit;  // the unit's first slot; its parts are consecutive
          // items (row, 4 value dims) over the key threads, two items at a
          // time, the parts in batches of 4: all loads of a step in flight
          const int n_items = rr * (D / 4);
          for (int it0 = threadIdx.x; it0 < n_items; it0 += 2 * kKeyThreads) {
            int row[2], d4[2];
            bool live[2];
            float M[2] = {kNegInf, kNegInf}, Ls[2] = {0.f, 0.f};
            float4 Us[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll
            for (int x2 = 0; x2 < 2; ++x2) {
              const int item = it0 + x2 * kKeyThreads;
              live[x2] = item < n_items;
              row[x2] = live[x2] ? item / (D / 4) : 0;
              d4[x2] = live[x2] ? item - row[x2] * (D / 4) : 0;
            }
            for (int s0 = 0; s0 < nparts; s0 += 4) {
              float ms[2][4], ls[2][4];
              float4 us[2][4];
#pragma unroll
              for (int x2 = 0; x2 < 2; ++x2)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  ms[x2][e] = kNegInf;
                  if (live[x2] && s0 + e < nparts) {
                    const int64_t idx = (fs + s0 + e) * R + row[x2];
                    ms[x2][e] = __ldcg(p.ws_m + idx);
                    ls[x2][e] = __ldcg(p.ws_l + idx);
                    us[x2][e] = __ldcg(reinterpret_cast<const float4*>(p.ws_u + idx * D) + d4[x2]);
                  }
                }
#pragma unroll
              for (int x2 = 0; x2 < 2; ++x2)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  if (ms[x2][e] == kNegInf) continue;  // an empty part contributes nothing
                  float ca, cb;                        // scale of the running sum, of part e
                  if (ms[x2][e] > M[x2]) {
                    ca = (M[x2] == kNegInf) ? 0.f : fast_exp2(M[x2] - ms[x2][e]);
                    cb = 1.f;
                    M[x2] = ms[x2][e];
                  } else {
                    ca = 1.f;
                    cb = fast_exp2(ms[x2][e] - M[x2]);
                  }
                  Ls[x2] = fmaf(Ls[x2], ca, cb * ls[x2][e]);
                  Us[x2].x = fmaf(Us[x2].x, ca, cb * us[x2][e].x);
                  Us[x2].y = fmaf(Us[x2].y, ca, cb * us[x2][e].y);
                  Us[x2].z = fmaf(Us[x2].z, ca, cb * us[x2][e].z);
                  Us[x2].w = fmaf(Us[x2].w, ca, cb * us[x2][e].w);
                }
            }
#pragma unroll
            for (int x2 = 0; x2 < 2; ++x2) {
              if (!live[x2]) continue;
              const float inv = (M[x2] == kNegInf) ? 0.f : 1.f / Ls[x2];
              const float o4[4] = {Us[x2].x * inv, Us[x2].y * inv, Us[x2].z * inv, Us[x2].w * inv};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int64_t oi = pf.ooff[row[x2]] + (int64_t)(4 * d4[x2] + e) * p.o_sd;
                if (p.out_bf16)
                  static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o4[e]);
                else
                  static_cast<float*>(p.out)[oi] = o4[e];
              }
              if (d4[x2] == 0)
                p.lse[pf.loff[row[x2]]] = (M[x2] == kNegInf) ? kNegInf : (M[x2] + __log2f(Ls[x2])) * kLn2;
            }
          }
        }
      }
      bar_sync(kBarRows, kKeyThreads);  // the finished unit's statistics and row facts are read
      if (threadIdx.x == 0) mbar_arrive(&q_empty[pb]);
      return true;
    };
    for (int64_t g = 0; cur.t < t1; cur.next(ntab, RG, Hkv, B), ++g) {
      const bool first = cur.t == t0 || cur.j == 0;
      const bool last = cur.t == t1 - 1 || cur.j == cur.n - 1;
      const int ub = uidx & 1;
      const RowFacts<NR>& rf = facts0[ub];
      if (first) {
        // the row facts come with the query rows
        const bool w = bar_and(kBarRows, kKeyThreads, wait_all(&q_full[ub], (uint32_t)((uidx >> 1) & 1)));
        if (!w) { ok = false; break; }
      }
      const int key0 = cur.key0();
      const int key = key0 + k;
      float x[NH];
      if (has_bias) {
        // this tile's bias (rows of one sequence share lines: L1 hits); a
        // per-row prefetch of the next tile measured slower (memory-pipe
        // instructions, not bytes, are the cost here)
        const bool kin = key < p.Tmax;
#pragma unroll
        for (int r = 0; r < NH; ++r)
          x[r] = kin ? __ldg(p.bias + rf.boff[c0 + r] + (int64_t)key * p.bi_sj) : 0.f;
      }
      const bool sok = wait_all(&s_full[g & 1], (uint32_t)((g >> 1) & 1));
      bool trig = !sok;
      if (sok) {
        tc::fence_after();
        float sc[NH];
        ld_cols<NH>(tl + kColS + 64u * (uint32_t)(g & 1) + c0, sc);
        const bool tail = key0 + BK > rf.min_end;
        // pairs of rows in packed fp32 (f32x2) arithmetic
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        if (has_bias) {
          const float2 l2e = make_float2(kLog2e, kLog2e);
#pragma unroll
          for (int r = 0; r < NH; r += 2) {
            const float2 v = __ffma2_rn(make_float2(sc[r], sc[r + 1]), sc2,
                                        __fmul2_rn(make_float2(x[r], x[r + 1]), l2e));
            x[r] = v.x;
            x[r + 1] = v.y;
          }
        } else {
#pragma unroll
          for (int r = 0; r < NH; r += 2) {
            const float2 v = __fmul2_rn(make_float2(sc[r], sc[r + 1]), sc2);
            x[r] = v.x;
            x[r + 1] = v.y;
          }
        }
        if (tail) {
#pragma unroll
          for (int r = 0; r < NH; ++r)
            if (key >= rf.end[c0 + r]) x[r] = kNegInf;
        }
        if (key0 < rf.win_max) {
          // sliding window: keys before a row's first visible key
#pragma unroll
          for (int r = 0; r < NH; ++r)
            if (key < (int)rf.tree[c0 + r]) x[r] = kNegInf;
        }
        if (key0 + BK > rf.tree_base) {
          // token tree: inside it a row sees only the nodes of its mask
          const int node = key - rf.tree_base;
          if (node >= 0 && node < 64) {
#pragma unroll
            for (int r = 0; r < NH; ++r)
              if (!((rf.tree[c0 + r] >> node) & 1ull)) x[r] = kNegInf;
          }
        }
#pragma unroll
        for (int r4 = 0; r4 < NH / 4; ++r4) {
          const float4 t4 = reinterpret_cast<const float4*>(s_thr + c0)[r4];
          trig |= (x[4 * r4] > t4.x) | (x[4 * r4 + 1] > t4.y) | (x[4 * r4 + 2] > t4.z) | (x[4 * r4 + 3] > t4.w);
        }
      } else if (lane == 0) {
        misc[2] = 1;
      }
      bool resc = false;
      if (bar_or(kBarRows, kKeyThreads, trig)) {
        if (misc[2] != 0) { ok = false; break; }  // read after the barrier: same answer everywhere
        // ---- raise the reference maxima: tile maxima over the 128 keys ----
        {
          float v[NH];
#pragma unroll
          for (int r = 0; r < NH; ++r) v[r] = x[r];
          warp_reduce_scatter<NH, true>(v, lane);
          if ((lane & 3) == 0) {
            const int base = scatter_base<NH>(lane);
#pragma unroll
            for (int i = 0; i < NH / 8; ++i) red[quarter * NR + c0 + base + i] = v[i];
          }
        }
        bar_sync(kBarRows, kKeyThreads);
        if (half == 0 && k < NR) {
          const float tmax = fmaxf(fmaxf(red[k], red[NR + k]), fmaxf(red[2 * NR + k], red[3 * NR + k]));
          const float mo = s_m[k];
          float a = 1.f;
          if (tmax > s_thr[k]) {
            a = (mo == kNegInf) ? 1.f : fast_exp2(mo - tmax);  // a row with no key yet has l = u = 0
            s_m[k] = tmax;
            s_muse[k] = tmax;
            s_thr[k] = tmax + kLazyRescale;
          }
          s_alpha[k] = a;
        }
        bar_sync(kBarRows, kKeyThreads);
#pragma unroll
        for (int r4 = 0; r4 < NH / 4; ++r4) {
          const float4 a4 = reinterpret_cast<const float4*>(s_alpha + c0)[r4];
          lp[4 * r4] *= a4.x;
          lp[4 * r4 + 1] *= a4.y;
          lp[4 * r4 + 2] *= a4.z;
          lp[4 * r4 + 3] *= a4.w;
        }
        if (!first) {
          // U^T lane k = value dim k, this half's columns of both parts; the
          // product with P_{j-1} must have completed (U += P_j V_j waits for
          // this tile's P)
          const bool pv = bar_and(kBarRows, kKeyThreads, wait_all(pv_done, (uint32_t)((g - 1) & 1)));
          if (!pv) { ok = false; break; }
          tc::fence_after();
          const uint32_t ua = tl + kColU + 128u * (uint32_t)ub + c0;
#pragma unroll 1
          for (int part = 0; part < 2; ++part) {
            float u[NH];
            ld_cols<NH>(ua + kLo * part, u);
#pragma unroll
            for (int r = 0; r < NH; ++r) u[r] *= s_alpha[c0 + r];
            st_cols<NH>(ua + kLo * part, u);
          }
          resc = true;
        }
      }
      // ---- P^T row of key k, this half's rows: 2^(x - m) as bf16 P_hi + P_lo ----
      {
        unsigned char* ph = sm + L::kOffP + (int)(g & 1) * kPBytes + k * 128;
#pragma unroll
        for (int c8 = 0; c8 < NH / 8; ++c8) {
          const float4 m0 = reinterpret_cast<const float4*>(s_muse + c0)[2 * c8];
          const float4 m1 = reinterpret_cast<const float4*>(s_muse + c0)[2 * c8 + 1];
          const float mu[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int r = 8 * c8 + 2 * e2;
            const float2 e = __ffma2_rn(make_float2(mu[2 * e2], mu[2 * e2 + 1]), make_float2(-1.f, -1.f),
                                        make_float2(x[r], x[r + 1]));
            const float2 pp = make_float2(fast_exp2(e.x), fast_exp2(e.y));  // masked: 2^-inf = 0
            const float2 l2 = __fadd2_rn(make_float2(lp[r], lp[r + 1]), pp);
            lp[r] = l2.x;
            lp[r + 1] = l2.y;
            asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(hi[e2]) : "r"(__float_as_uint(pp.x)), "r"(__float_as_uint(pp.y)));
            const float2 rem = __ffma2_rn(make_float2(__uint_as_float(__float_as_uint(pp.x) & 0xffff0000u),
                                                      __uint_as_float(__float_as_uint(pp.y) & 0xffff0000u)),
                                          make_float2(-1.f, -1.f), pp);
            lo[e2] = pack_bf16(rem.x, rem.y);
          }
          const int c = c0 / 8 + c8;  // 16-byte chunk of the row's P_hi
          const int off = ((c ^ (k & 7)) << 4);
          const int off_lo = L::kPacked ? (((c + NR / 8) ^ (k & 7)) << 4) : kBox + off;
          *reinterpret_cast<uint4*>(ph + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(ph + off_lo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      if (cur.j == cur.n - 1 && key0 + BK > rf.unit_end) {
        // the unit's last tile: zero the V rows past every visible key (each
        // half of the warps one 64-dim box)
        const int64_t sv = 2 * g + 1;
        const bool vok = bar_and(kBarRows, kKeyThreads, wait_all(&full[sv % kSlots], (uint32_t)((sv / kSlots) & 1)));
        if (!vok) { ok = false; break; }
        if (key >= rf.unit_end) {
          unsigned char* vr = sm + L::kOffRing + (int)(sv % kSlots) * kSlotBytes + half * kBox + k * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vr + ((c ^ (k & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P^T, V rows -> tensor core
      if (resc) tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[g & 1]);

      // the U readout of the previous unit (its last product has long
      // completed by now)
      if (pend) {
        if (!flush()) { ok = false; break; }
        pend = false;
      }
      if (last) {
        // ---- close the unit (or this CTA's part of it): l over the keys ----
        warp_reduce_scatter<NH, false>(lp, lane);
        if ((lane & 3) == 0) {
          const int base = scatter_base<NH>(lane);
#pragma unroll
          for (int i = 0; i < NH / 8; ++i) red[quarter * NR + c0 + base + i] = lp[i];
        }
#pragma unroll
        for (int r = 0; r < NH; ++r) lp[r] = 0.f;
        bar_sync(kBarRows, kKeyThreads);
        if (half == 0 && k < NR) {
          const float l = (red[k] + red[NR + k]) + (red[2 * NR + k] + red[3 * NR + k]);
          const float m = s_m[k];
          s_mfin[k] = m;
          s_lfin[k] = l;
          s_inv[k] = (m == kNegInf) ? 0.f : 1.f / l;
          // fresh statistics for the next unit
          s_m[k] = kNegInf;
          s_muse[k] = 0.f;
          s_thr[k] = kNegInf;
        }
        bar_sync(kBarRows, kKeyThreads);
        pend = true;
        pend_uidx = uidx;
        pend_su = cur.su;
        pend_b = cur.b;
        pend_kvh = cur.kvh;
        pend_rg = cur.rg;
        pend_n = cur.n;
        ++uidx;
      }
    }
    if (ok && pend && !flush()) ok = false;
    if (!ok && lane == 0) record_error(p.err, kErrTimeout);
  }

  // the merge grid may start launching (it waits for this grid's completion
  // before reading anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tb, kTmemCols);
}

template <int NR>
cudaError_t launch_nr(const FwdParams& p, int ctas, const CUtensorMap& tmk, const CUtensorMap& tmv,
                      cudaStream_t stream) {
  using L = TcLayout<NR>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_tc_kernel<NR>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  decode_tc_kernel<NR><<<ctas, kThreads, L::kBytes, stream>>>(p, tmk, tmv);
  return cudaGetLastError();
}

}  // namespace

size_t decode_tc_smem_bytes(int nr) {
  if (nr <= 16) return TcLayout<16>::kBytes;
  if (nr <= 32) return TcLayout<32>::kBytes;
  return TcLayout<48>::kBytes;
}

cudaError_t launch_decode_tc(const FwdParams& p, int ctas, const CUtensorMap& tmk, const CUtensorMap& tmv,
                             cudaStream_t stream) {
  if (p.rows_cta < 1 || p.rows_cta > 48 || ctas < 1 ||
      p.B * p.row_groups > (p.window > 0 ? kDecodeTcMaxEntries / 2 : kDecodeTcMaxEntries))
    return cudaErrorInvalidValue;
  if (p.rows_cta <= 16) return launch_nr<16>(p, ctas, tmk, tmv, stream);
  if (p.rows_cta <= 32) return launch_nr<32>(p, ctas, tmk, tmv, stream);
  return launch_nr<48>(p, ctas, tmk, tmv, stream);
}

}  // namespace blkattn
