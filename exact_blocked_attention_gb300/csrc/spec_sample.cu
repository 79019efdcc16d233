// One speculative-decoding verification step per sequence: in-order
// acceptance of the draft's candidates and the draw of the token that follows
// them ("Chapter 33: inference compute optimisation" §33.5, eqs. 33.10–33.13;
// §33.6 for the order).
//
//   candidate x_i is kept iff u_i * q_i(x_i) < p_i(x_i)      (eq. 33.10, fp64:
//                                      exact for fp32 operands)
//   at the first rejection, draw from [p_i - q_i]_+ / Z     (eq. 33.12)
//   if all k are kept, draw from p_{k+1}
//
// The draw is an inverse CDF in fixed point: the mass of token x is the
// exact difference p(x) - q(x) for a residual (eq. 33.12 does not round it)
// or p(x) for a target, clamped to [0, 2]; its weight is F(m) = floor(m *
// 2^40).  The difference is kept as an unevaluated pair hi + lo with Knuth's
// TwoSum (TAOCP vol. 2, §4.2.2: hi = fl(p - q) and lo = (p - q) - hi, both
// exact fp32 values), F(hi) is formed as two exact 20-bit halves with fp32
// floors, and lo moves the weight only when hi * 2^40 is an integer (then
// by floor(lo * 2^40); otherwise |lo| 2^40 is below the distance from
// hi * 2^40 to either neighbouring integer).  No fp64 and no 64-bit
// conversion: both run at a small fraction of the fp32 rate here.  When
// every mass of a warp's share of a slot lies in [0, 1] (as for any real
// distribution) a shorter exact form without the pair and the clamps gives
// the same weights; the warp checks that and takes the full form otherwise.
// Integer
// prefix sums (order-independent, so every reduction shape gives the same
// token), threshold floor(s * Z / 2^32) for
// the row's 32-bit uniform s, and the token is the smallest index whose
// prefix sum exceeds it.  A rejection that meets a zero residual keeps the
// candidate (rejection has probability zero there); a candidate outside the
// vocabulary or with q = 0 cannot have been proposed and is rejected (with no
// residual mass at its position, the token is drawn from p_i itself).  A
// distribution without mass at 2^-40 resolution gives token 0.
//
// A cluster of two CTAs per sequence; each CTA sums the weights of one half
// of the row drawn from.  In a CTA, a producer warp streams its half through
// a ring of three 64 KB shared-memory slots (8192 entries of p and of q per
// slot) with 1-D bulk asynchronous copies, when the rows are 16-byte aligned
// (plain loads otherwise), and 16 consumer warps sum 512 entries of every
// slot each, keeping the sum of each (chunk of slots, warp) on chip.  Warp 0
// tests the candidates 32 at a time first (the lowest rejected lane wins).
// The two CTAs exchange their totals through distributed shared memory; the
// CTA whose half holds the threshold finds the chunk and the warp's 512
// entries from its own sums and scans those entries once more (from L2) with
// the whole CTA.  The row pair (p, q) of the chosen position is the only
// vocabulary-sized traffic.
#include <cooperative_groups.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace blkattn {
namespace {

constexpr int kWarps = 16;                  // consumer warps
constexpr int kProducer = kWarps;           // the copy-issuing warp
constexpr int kThreads = 32 * (kWarps + 1);
constexpr int kCluster = 2;                 // CTAs per sequence
constexpr int kSlot = 8192;                 // entries per ring slot (p and q)
constexpr int kStages = 3;                  // ring slots
constexpr int kPerWarp = kSlot / kWarps;    // entries of a slot per consumer warp (16 per lane)
constexpr int kMaxChunks = 64;              // recorded chunk sums per CTA
constexpr int kRingBytes = kStages * kSlot * 4 * 2;
constexpr int kSmemBytes = kRingBytes + kMaxChunks * kWarps * 8 + 64;
constexpr float kTwo20 = 1048576.0f;         // 2^20
constexpr float kTwo40 = 1099511627776.0f;   // 2^40
constexpr float kTwoM20 = 1.0f / 1048576.0f;  // 2^-20
constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23: x + kMagic holds integer |x| < 2^22 in its low bits
constexpr int kMagicBits = 0x4B400000;

// Weight F(m) = floor(m 2^40) of one entry, m = clamp(p - q, 0, 2) with the
// exact difference (has_q) or m = clamp(p, 0, 2), added to the lane's 32-bit
// counters as F = sh 2^20 + sl:
//   hi = fl(p - q), lo = (p - q) - hi         (TwoSum: exact for finite p, q)
//   c = clamp(hi, 0, 2), t = c 2^20 (exact), h = floor(t) <= 2^21,
//   r = (t - h) 2^20 (exact), l = floor(r) < 2^20, and F = h 2^20 + l + e with
//   e = floor(lo 2^40) when 0 < hi <= 2 and r == l (c 2^40 is an integer,
//   so F = c 2^40 + floor(lo 2^40)); e <= 0 when hi == 2 (m above 2 clamps);
//   e = 0 otherwise: hi <= 0 means m <= 0 (|lo| < |hi|), hi > 2 means m > 2,
//   and for a non-integer c 2^40, |lo| 2^40 <= ulp(c 2^40) / 2 keeps it
//   between the same integers.  |e| <= 2^17 (|lo| <= ulp(hi) / 2 <= 2^-23).
// Each floor is one addition of 1.5 * 2^23 rounded down (exact for |x| <
// 2^22: the sum lies in [2^23, 2^24), where fp32 steps by 1), whose low bits
// hold the integer: no round-to-integer instruction and no conversion.
// NaN masses count as 0 (fmaxf skips NaN), +inf as 2.
template <bool HQ>
__device__ __forceinline__ void add_entry(float pv, float qv, int& sh, int& sl) {
  constexpr bool has_q = HQ;
  float hi = pv;
  int e = 0;
  if constexpr (HQ) {
    hi = __fsub_rn(pv, qv);
    const float bb = __fsub_rn(hi, pv);  // the part of hi that came from -q
    const float lo = __fadd_rn(__fsub_rn(pv, __fsub_rn(hi, bb)), __fsub_rn(-qv, bb));
    e = __float_as_int(__fadd_rd(__fmul_rn(lo, kTwo40), kMagic)) - kMagicBits;  // floor(lo 2^40), used below only
    if (hi >= 2.f) e = min(e, 0);
  }
  const float c = fminf(fmaxf(hi, 0.f), 2.f);
  const float t = __fmul_rn(c, kTwo20);
  const float mh = __fadd_rd(t, kMagic);                                        // floor(t) in the low bits
  const float r = __fmul_rn(__fsub_rn(t, __fsub_rn(mh, kMagic)), kTwo20);       // frac(t) 2^20
  const float ml = __fadd_rd(r, kMagic);                                        // floor(r) in the low bits
  if (!(has_q && hi > 0.f && hi <= 2.f && r == __fsub_rn(ml, kMagic))) e = 0;
  sh += __float_as_int(mh) - kMagicBits;
  sl += __float_as_int(ml) - kMagicBits + e;
}
// The same weight for masses already in [0, 1], where no clamp acts, in
// seven fp32 operations and no select.  With qs = min(q, p) (m = 0 when
// q >= p) and v = p - qs >= 0:
//   y  = rd(v)                       floor(y 2^20) = floor(v 2^20): that floor
//                                    times 2^-20 is an fp32 value <= v
//   mh = rd(y 2^20 + 1.5 2^23)       one fused rounding: 1.5 2^23 + h, h = floor(v 2^20)
//   D  = p - h 2^-20                 exact: a multiple of ulp(p) in [0, p]
//   t  = rd(D - qs)                  D - qs = v - h 2^-20 lies in [0, 2^-20)
//   ml = rd(t 2^40 + 1.5 2^23)       1.5 2^23 + l, l = floor((v - h 2^-20) 2^40)
// and F = h 2^20 + l.  (rd: rounding toward -inf; the floor of a value whose
// floor is an fp32 number equals the floor of its round-down.)  in_range
// collects the bit patterns: all of them <= 0x3F800000 (1.0f) means every
// mass was a non-negative number <= 1 (-0, NaN, inf and negatives fail).
template <bool HQ>
__device__ __forceinline__ void add_entry_unit(float pv, float qv, int& sh, int& sl, unsigned& bits) {
  bits = max(bits, __float_as_uint(pv));
  float qs = 0.f, y = pv;
  if constexpr (HQ) {
    bits = max(bits, __float_as_uint(qv));
    qs = fminf(qv, pv);
    y = __fadd_rd(pv, -qs);
  }
  const float mh = __fmaf_rd(y, kTwo20, kMagic);
  const float d = __fmaf_rn(-__fsub_rn(mh, kMagic), kTwoM20, pv);
  const float t = HQ ? __fadd_rd(d, -qs) : d;
  const float ml = __fmaf_rd(t, kTwo40, kMagic);
  sh += __float_as_int(mh) - kMagicBits;
  sl += __float_as_int(ml) - kMagicBits;
}
constexpr unsigned kOneBits = 0x3F800000u;

// (sl may be negative: l + e < 0 when l = 0 and lo < 0)
__device__ __forceinline__ uint64_t combine(int sh, int sl) {
  return (uint64_t)((int64_t)sh * (1 << 20) + (int64_t)sl);
}

// weight of entry x of the residual of (p, q) (q == nullptr: of p itself)
__device__ __forceinline__ uint64_t weight(const float* p, const float* q, int64_t x) {
  int sh = 0, sl = 0;
  if (q != nullptr)
    add_entry<true>(__ldg(p + x), __ldg(q + x), sh, sl);
  else
    add_entry<false>(__ldg(p + x), 0.f, sh, sl);
  return combine(sh, sl);
}

// The weights of one consumer warp's entries of a ring slot, added to the
// lane's counters: 16 entries per lane from shared memory (all 512 copied),
// or entry by entry (the ragged end, and rows not 16-byte aligned: plain
// loads from global memory where the copy did not reach).
template <bool HQ>
__device__ __forceinline__ void slot_sum(const float* sp, const float* sq, const float* gp, const float* gq,
                                         int nw, int copied_here, int lane, int& sh, int& sl) {
  if (copied_here >= kPerWarp) {
    int fh = 0, fl = 0;
    unsigned bits = 0;
#pragma unroll
    for (int v4 = 0; v4 < kPerWarp / 128; ++v4) {
      const float4 a = reinterpret_cast<const float4*>(sp)[v4 * 32 + lane];
      const float4 c = HQ ? reinterpret_cast<const float4*>(sq)[v4 * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      add_entry_unit<HQ>(a.x, c.x, fh, fl, bits);
      add_entry_unit<HQ>(a.y, c.y, fh, fl, bits);
      add_entry_unit<HQ>(a.z, c.z, fh, fl, bits);
      add_entry_unit<HQ>(a.w, c.w, fh, fl, bits);
    }
    if (__any_sync(0xffffffffu, bits > kOneBits)) {
      // a mass outside [0, 1] in the warp's 512 entries: all of them again
      // with the clamps
      fh = fl = 0;
#pragma unroll 1
      for (int v4 = 0; v4 < kPerWarp / 128; ++v4) {
        const float4 a = reinterpret_cast<const float4*>(sp)[v4 * 32 + lane];
        const float4 c = HQ ? reinterpret_cast<const float4*>(sq)[v4 * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        add_entry<HQ>(a.x, c.x, fh, fl);
        add_entry<HQ>(a.y, c.y, fh, fl);
        add_entry<HQ>(a.z, c.z, fh, fl);
        add_entry<HQ>(a.w, c.w, fh, fl);
      }
    }
    sh += fh;
    sl += fl;
  } else {
    for (int e = lane; e < nw; e += 32) {
      const float pv = e < copied_here ? sp[e] : __ldg(gp + e);
      const float qv = !HQ ? 0.f : (e < copied_here ? sq[e] : __ldg(gq + e));
      add_entry<HQ>(pv, qv, sh, sl);
    }
  }
}

// Boundary of the two CTAs' halves of a row of V entries: a multiple of 4,
// so a 16-byte aligned row stays aligned at the second half.
__device__ __forceinline__ int64_t half_cut(int64_t V, unsigned r) {
  return r == 0 ? 0 : (r >= kCluster ? V : ((V / 2) & ~(int64_t)3));
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    spec_sample_kernel(const float* __restrict__ p, int64_t p_sb, int64_t p_si, const float* __restrict__ q,
                       int64_t q_sb, int64_t q_si, const int32_t* __restrict__ draft, int64_t d_sb, int64_t d_si,
                       const float* __restrict__ u_acc, int64_t u_sb, int64_t u_si,
                       const int32_t* __restrict__ u_smp, int64_t s_sb, int k, int64_t V,
                       int32_t* __restrict__ n_out, int64_t n_sb, int32_t* __restrict__ tok_out, int64_t t_sb,
                       int* __restrict__ err) {
  namespace cg = cooperative_groups;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* ring = reinterpret_cast<float*>(smem_raw);  // slot s: p at [2 s kSlot], q at [(2 s + 1) kSlot]
  uint64_t* csum = reinterpret_cast<uint64_t*>(smem_raw + kRingBytes);  // [chunk][warp]
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ uint64_t part[kWarps];   // each consumer warp's total over this CTA's half
  // the two halves' totals of a row sum, by the parity of the sum's round:
  // each CTA writes its total into both CTAs' copy, so one cluster barrier
  // makes both visible (a copy is written again two rounds later, after the
  // next round's barrier, which both CTAs reach only after reading it)
  __shared__ uint64_t halves[2][kCluster];
  __shared__ uint64_t wtot[2][kWarps + 1];  // warp totals of the final scan (every warp takes part)
  __shared__ uint64_t pick_c;  // the draw's prefix before the warp range it lies in
  __shared__ int pick_w;
  // [0] first position not kept, [1] its candidate is possible, [2] the
  // row's 32 random bits (loaded with the candidates, not at the draw)
  __shared__ int state[3];
  cg::cluster_group cl = cg::this_cluster();
  const unsigned rank = cl.block_rank();
  const int b = blockIdx.x / kCluster;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kWarps);  // one arrival per consumer warp
    }
    fence_barrier_init();
  }
  __syncthreads();
  // this CTA has started; the matching wait precedes the first write into
  // the peer's shared memory
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // this CTA's half of the row: slots of kSlot entries, chunks of m slots
  const int64_t c_lo = half_cut(V, rank), c_hi = half_cut(V, rank + 1);
  // (32-bit slot counts: a half has at most 2^18 slots, and the rows a call
  // streams, at most k + 2 of them, fit in device memory)
  const int n_slots = (int)((c_hi - c_lo + kSlot - 1) / kSlot);
  const int m = max(1, (n_slots + kMaxChunks - 1) / kMaxChunks);
  uint32_t ring_pos = 0;  // slots streamed so far (ring slot and phase)
  int round = 0;          // row sums done
  uint64_t h_first = 0;   // the first half's total in the last row sum
  bool ok = true;

  // Z of one row: each CTA sums its half through the ring, the pair
  // exchanges the two totals
  auto row_sum = [&](const float* pr_, const float* qr_, bool vec_) -> uint64_t {
    const bool hq = qr_ != nullptr;
    if (warp == kProducer) {
      if (lane == 0 && vec_) {
        const uint64_t pol = policy_evict_first();  // the rows are read once
        for (int u = 0; u < n_slots; ++u) {
          const uint32_t g = ring_pos + (uint32_t)u;
          const int st = (int)(g % kStages);
          if (g >= kStages && !mbar_wait(&empty[st], ((g / kStages) - 1) & 1)) { ok = false; break; }
          const int64_t x0 = c_lo + (int64_t)u * kSlot;
          const uint32_t bytes = (uint32_t)((min((int64_t)kSlot, c_hi - x0) & ~(int64_t)3) * 4);
          mbar_arrive_expect_tx(&full[st], hq ? 2 * bytes : bytes);
          if (bytes > 0) {
            bulk_g2s(ring + 2 * st * kSlot, pr_ + x0, bytes, &full[st], pol);
            if (hq) bulk_g2s(ring + (2 * st + 1) * kSlot, qr_ + x0, bytes, &full[st], pol);
          }
        }
      }
    } else {
      uint64_t tot = 0;
      int sh = 0, sl = 0;
      int ch = 0, in_ch = 0;  // chunk of the slot, slots of the chunk done
      for (int u = 0; u < n_slots; ++u) {
        const uint32_t g = ring_pos + (uint32_t)u;
        const int st = (int)(g % kStages);
        const int64_t x0 = c_lo + (int64_t)u * kSlot;
        const int64_t xw = x0 + warp * kPerWarp;  // this warp's 512 entries
        const int64_t nw = min((int64_t)kPerWarp, c_hi - xw);  // (<= 0: none)
        if (vec_) {
          if (!__all_sync(0xffffffffu, ok && mbar_wait(&full[st], (g / kStages) & 1))) ok = false;
          // slot entries [0, copied) came by copy; a ragged end of <= 3 by plain loads
          const int copied = (int)(min((int64_t)kSlot, c_hi - x0) & ~(int64_t)3);
          const int here = (int)max((int64_t)0, min((int64_t)kPerWarp, (int64_t)copied - warp * kPerWarp));
          const float* sp = ring + 2 * st * kSlot + warp * kPerWarp;
          const float* sq = ring + (2 * st + 1) * kSlot + warp * kPerWarp;
          if (ok && nw > 0) {
            if (hq)
              slot_sum<true>(sp, sq, pr_ + xw, qr_ + xw, (int)nw, here, lane, sh, sl);
            else
              slot_sum<false>(sp, sq, pr_ + xw, nullptr, (int)nw, here, lane, sh, sl);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the slot
        } else if (nw > 0) {
          if (hq)
            slot_sum<true>(nullptr, nullptr, pr_ + xw, qr_ + xw, (int)nw, 0, lane, sh, sl);
          else
            slot_sum<false>(nullptr, nullptr, pr_ + xw, nullptr, (int)nw, 0, lane, sh, sl);
        }
        // fold the lane counters (16 entries per slot: every 32 slots at
        // least) and record the warp's running total at each chunk's end
        const bool chunk_end = ++in_ch == m || u + 1 == n_slots;
        if (chunk_end || ((u + 1) & 31) == 0) {
          uint64_t cs = combine(sh, sl);
          sh = sl = 0;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
          tot += cs;
          if (chunk_end && lane == 0) csum[ch * kWarps + warp] = tot;
        }
        if (chunk_end) {
          ++ch;
          in_ch = 0;
        }
      }
      if (lane == 0) part[warp] = tot;
    }
    if (warp == kProducer && lane == 0 && vec_) {
      // the copies this thread issued have landed before anything moves on
      const uint32_t end = ring_pos + (uint32_t)n_slots;
      for (uint32_t g = n_slots > kStages ? end - kStages : ring_pos; g < end; ++g)
        if (!mbar_wait(&full[g % kStages], (g / kStages) & 1)) ok = false;
    }
    if (vec_) ring_pos += (uint32_t)n_slots;  // (the barriers' phases advance only on this path)
    __syncthreads();
    uint64_t* hv = halves[round & 1];
    if (round == 0) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // the peer has started
    if (threadIdx.x == 0) {
      uint64_t h = 0;
      for (int w = 0; w < kWarps; ++w) h += part[w];
      hv[rank] = h;
      *cl.map_shared_rank(&hv[rank], rank ^ 1u) = h;
    }
    cl.sync();  // both totals are in both CTAs
    ++round;
    h_first = hv[0];
    return hv[0] + hv[1];
  };

  int i = 0;
  uint32_t s = 0;
  const float* pr = nullptr;
  const float* qr = nullptr;
  bool vec = false;
  uint64_t Z = 0;
  while (true) {
    // ---- in-order acceptance, up to the first rejection: warp 0 tests 32
    // candidates at once (their loads in parallel), the lowest failing lane wins
    if (warp == 0) {
      const int sv = lane == 0 ? u_smp[(int64_t)b * s_sb] : 0;
      int j = k, valid = 0;
      for (int j0 = i; j0 < k; j0 += 32) {
        const int jj = j0 + lane;
        bool keep = true, okc = false;
        if (jj < k) {
          const int x = draft[(int64_t)b * d_sb + (int64_t)jj * d_si];
          keep = false;
          if (x >= 0 && (int64_t)x < V) {  // otherwise it cannot have been proposed
            const double px = (double)p[(int64_t)b * p_sb + (int64_t)jj * p_si + x];
            const double qx = (double)q[(int64_t)b * q_sb + (int64_t)jj * q_si + x];
            const double u = (double)u_acc[(int64_t)b * u_sb + (int64_t)jj * u_si];
            okc = qx > 0.0;
            keep = okc && u * qx < px;
          }
        }
        const unsigned stop = __ballot_sync(0xffffffffu, !keep);
        if (stop != 0u) {
          const int l = __ffs(stop) - 1;
          j = j0 + l;
          valid = __shfl_sync(0xffffffffu, (int)okc, l);
          break;
        }
      }
      if (lane == 0) {
        state[0] = j;
        state[1] = valid;
        state[2] = sv;
      }
    }
    __syncthreads();
    i = state[0];
    const bool valid = state[1] != 0;
    s = (uint32_t)state[2];
    // the distribution to draw from: the residual at the rejected position,
    // or the target one past the candidates
    pr = p + (int64_t)b * p_sb + (int64_t)i * p_si;
    qr = i < k ? q + (int64_t)b * q_sb + (int64_t)i * q_si : nullptr;
    vec = ((reinterpret_cast<uintptr_t>(pr) | reinterpret_cast<uintptr_t>(qr)) & 15) == 0;
    Z = row_sum(pr, qr, vec);
    if (Z != 0 || i >= k) break;
    if (!valid) {
      // an impossible candidate and no residual mass: draw from p_i itself
      qr = nullptr;
      vec = (reinterpret_cast<uintptr_t>(pr) & 15) == 0;
      Z = row_sum(pr, qr, vec);
      break;
    }
    // a rejection with no residual mass: keep the candidate, go on
    ++i;
    __syncthreads();  // every thread has read state[]
  }
  if (!ok && lane == 0) record_error(err, kErrTimeout);
  if (Z == 0) {  // the distribution drawn from has no mass above 2^-40: token 0 by definition
    if (rank == 0 && threadIdx.x == 0) {
      n_out[(int64_t)b * n_sb] = i;
      tok_out[(int64_t)b * t_sb] = 0;
    }
    return;
  }
  const uint64_t T = __umul64hi((uint64_t)s << 32, Z);  // floor(s Z / 2^32) < Z

  // ---- the half holding T; its CTA finishes the draw from its own sums ----
  const unsigned owner = T < h_first ? 0u : 1u;
  if (rank != owner) return;
  uint64_t c = owner == 0 ? 0 : h_first;
  // the chunk holding T: the half's running total at a chunk's end is the
  // sum of the warps' running totals there, and these grow along the
  // vocabulary, so the chunk is the number of chunk ends at or below T (one
  // thread per chunk end; the last chunk holds T if no earlier one does)
  const int n_ch = (n_slots + m - 1) / m;
  auto chunk_end = [&](int x) -> uint64_t {  // (x < 0: before the first chunk)
    uint64_t t = 0;
    if (x >= 0) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += csum[x * kWarps + w];
    }
    return t;
  };
  const int ch = __syncthreads_count((int)threadIdx.x < n_ch - 1 && c + chunk_end((int)threadIdx.x) <= T);
  int64_t L0 = c_lo + (int64_t)ch * m * kSlot;
  int64_t L1 = min(c_hi, L0 + (int64_t)m * kSlot);
  if (m > 1) {
    c += chunk_end(ch - 1);
  } else {
    // one-slot chunks: the warp whose 512 entries hold T.  Warp 0, lane w:
    // warp w's running totals before and at the chunk's end; their sum over
    // the lanes is the chunk's base, their differences the warps' amounts,
    // whose inclusive prefix passes T - base first at the warp sought
    if (warp == 0) {
      uint64_t before = 0, amount = 0;
      if (lane < kWarps) {
        before = ch > 0 ? csum[(ch - 1) * kWarps + lane] : 0;
        amount = csum[ch * kWarps + lane] - before;
      }
      uint64_t base = before;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) base += __shfl_xor_sync(0xffffffffu, base, off);
      base += c;
#pragma unroll
      for (int off = 1; off < kWarps; off <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, amount, off);
        if (lane >= off) amount += y;
      }
      const int w = __popc(__ballot_sync(0xffffffffu, lane < kWarps - 1 && base + amount <= T));
      const uint64_t below = __shfl_sync(0xffffffffu, amount, w > 0 ? w - 1 : 0);
      if (lane == 0) {
        pick_w = w;
        pick_c = base + (w > 0 ? below : 0);
      }
    }
    __syncthreads();
    c = pick_c;
    L0 = min(c_hi, L0 + (int64_t)pick_w * kPerWarp);
    L1 = min(c_hi, L0 + kPerWarp);
  }
  // ---- one scan of [L0, L1), kThreads entries a round: an inclusive prefix
  // over each warp's lanes, then over the warps' totals.  T lies in the round
  // whose total passes it, in the one warp whose range holds it, at the lowest
  // lane whose prefix passes it; that lane writes the result ----
  for (int64_t x0 = L0, r = 0; x0 < L1; x0 += kThreads, ++r) {
    const int64_t x = x0 + threadIdx.x;
    uint64_t v = x < L1 ? weight(pr, qr, x) : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += y;
    }
    // (two buffers: a round's totals are rewritten two rounds later, after
    // the next round's barrier, which follows every read of them)
    uint64_t* wt = wtot[r & 1];
    if (lane == 31) wt[warp] = v;
    __syncthreads();
    uint64_t before = c, total = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWarps + 1; ++w2) {
      before += w2 < warp ? wt[w2] : 0;
      total += wt[w2];
    }
    const unsigned past = __ballot_sync(0xffffffffu, before + v > T);
    if (before <= T && T < before + wt[warp] && lane == __ffs(past) - 1) {
      n_out[(int64_t)b * n_sb] = i;
      tok_out[(int64_t)b * t_sb] = (int32_t)x;  // T < Z: some round holds it
    }
    if (c + total > T) break;
    c += total;
  }
}

bool dims(const blkattn_tensor* t, int n) {
  if (t == nullptr || t->ndim != n) return false;
  for (int i = 0; i < n; ++i)
    if (t->sizes[i] < 0 || t->strides[i] < 0) return false;
  return true;
}

}  // namespace
}  // namespace blkattn

extern "C" int blkattn_spec_sample(const blkattn_tensor* p, const blkattn_tensor* q, const blkattn_tensor* draft,
                                   const blkattn_tensor* u_accept, const blkattn_tensor* u_sample,
                                   const blkattn_tensor* n_accepted, const blkattn_tensor* token,
                                   blkattn_stream_t stream) {
  using blkattn::dims;
  if (!dims(p, 3) || !dims(q, 3) || !dims(draft, 2) || !dims(u_accept, 2) || !dims(u_sample, 1) ||
      !dims(n_accepted, 1) || !dims(token, 1))
    return BLKATTN_ERR_INVALID_ARG;
  if (p->dtype != BLKATTN_F32 || q->dtype != BLKATTN_F32 || draft->dtype != BLKATTN_I32 ||
      u_accept->dtype != BLKATTN_F32 || u_sample->dtype != BLKATTN_I32 || n_accepted->dtype != BLKATTN_I32 ||
      token->dtype != BLKATTN_I32)
    return BLKATTN_ERR_INVALID_ARG;
  const int64_t B = p->sizes[0], k = p->sizes[1] - 1, V = p->sizes[2];
  if (k < 0 || V < 1 || q->sizes[0] != B || q->sizes[1] != k || q->sizes[2] != V || draft->sizes[0] != B ||
      draft->sizes[1] != k || u_accept->sizes[0] != B || u_accept->sizes[1] != k || u_sample->sizes[0] != B ||
      n_accepted->sizes[0] != B || token->sizes[0] != B)
    return BLKATTN_ERR_INVALID_ARG;
  // vocabulary contiguous (an empty q, or a vocabulary of one, has no such stride)
  if ((V > 1 && p->strides[2] != 1) || (k > 0 && V > 1 && q->strides[2] != 1)) return BLKATTN_ERR_INVALID_ARG;
  // one device, the current one
  for (const blkattn_tensor* t : {q, draft, u_accept, u_sample, n_accepted, token})
    if (t->device != p->device) return BLKATTN_ERR_INVALID_ARG;
  if (p->device < 0) return BLKATTN_ERR_INVALID_ARG;
  if (B == 0) return BLKATTN_OK;
  if (B > 0x3fffffff || k > 0x7fffffff || V > 0x7fffffff) return BLKATTN_ERR_UNSUPPORTED;  // grid: two CTAs a row
  for (const blkattn_tensor* t : {p, q, draft, u_accept, u_sample, n_accepted, token})
    if (t->data == nullptr && !(t == q && k == 0) && !(t == draft && k == 0) && !(t == u_accept && k == 0))
      return BLKATTN_ERR_INVALID_ARG;
  {
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return blkattn::report_cuda_failure(e);
    if (dev != p->device) return BLKATTN_ERR_INVALID_ARG;
  }
  int* err = nullptr;
  if (int st = blkattn::device_error_word(&err); st != BLKATTN_OK) return st;
  static bool attr_set = false;  // (the ring takes more than the default 48 KB of shared memory)
  if (!attr_set) {
    if (cudaError_t e = cudaFuncSetAttribute(blkattn::spec_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             blkattn::kSmemBytes);
        e != cudaSuccess)
      return blkattn::report_cuda_failure(e);
    attr_set = true;
  }
  blkattn::spec_sample_kernel<<<(unsigned)(B * blkattn::kCluster), blkattn::kThreads, blkattn::kSmemBytes,
                                 reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const float*>(p->data), p->strides[0], p->strides[1], static_cast<const float*>(q->data),
      q->strides[0], q->strides[1], static_cast<const int32_t*>(draft->data), draft->strides[0], draft->strides[1],
      static_cast<const float*>(u_accept->data), u_accept->strides[0], u_accept->strides[1],
      static_cast<const int32_t*>(u_sample->data), u_sample->strides[0], (int)k, V,
      static_cast<int32_t*>(n_accepted->data), n_accepted->strides[0], static_cast<int32_t*>(token->data),
      token->strides[0], err);
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return blkattn::report_cuda_failure(e);
  return BLKATTN_OK;
}
