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
// conversion: both run at a small fraction of the fp32 rate here.  Integer
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
#pragma unroll
    for (int v4 = 0; v4 < kPerWarp / 128; ++v4) {
      const float4 a = reinterpret_cast<const float4*>(sp)[v4 * 32 + lane];
      const float4 c = HQ ? reinterpret_cast<const float4*>(sq)[v4 * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      add_entry<HQ>(a.x, c.x, sh, sl);
      add_entry<HQ>(a.y, c.y, sh, sl);
      add_entry<HQ>(a.z, c.z, sh, sl);
      add_entry<HQ>(a.w, c.w, sh, sl);
    }
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
  __shared__ uint64_t halves[kCluster];
  __shared__ uint64_t wtot[kWarps + 1];  // warp totals of the final scan (every warp takes part)
  __shared__ int state[2];            // [0] first position not kept, [1] its candidate is possible
  cg::cluster_group cl = cg::this_cluster();
  const unsigned rank = cl.block_rank();
  const int b = blockIdx.x / kCluster;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t s = (uint32_t)u_smp[(int64_t)b * s_sb];
  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kWarps);  // one arrival per consumer warp
    }
    fence_barrier_init();
  }
  __syncthreads();

  // this CTA's half of the row: slots of kSlot entries, chunks of m slots
  const int64_t c_lo = half_cut(V, rank), c_hi = half_cut(V, rank + 1);
  const int64_t n_slots = (c_hi - c_lo + kSlot - 1) / kSlot;
  const int64_t m = (n_slots + kMaxChunks - 1) / kMaxChunks < 1 ? 1 : (n_slots + kMaxChunks - 1) / kMaxChunks;
  int64_t ring_pos = 0;  // slots streamed so far (ring slot and phase)
  bool ok = true;

  // Z of one row: each CTA sums its half through the ring, the pair
  // exchanges the two totals
  auto row_sum = [&](const float* pr_, const float* qr_, bool vec_) -> uint64_t {
    const bool hq = qr_ != nullptr;
    if (warp == kProducer) {
      if (lane == 0 && vec_) {
        const uint64_t pol = policy_evict_first();  // the rows are read once
        for (int64_t u = 0; u < n_slots; ++u) {
          const int64_t g = ring_pos + u;
          const int st = (int)(g % kStages);
          if (g >= kStages && !mbar_wait(&empty[st], (uint32_t)(((g / kStages) - 1) & 1))) { ok = false; break; }
          const int64_t x0 = c_lo + u * kSlot;
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
      for (int64_t u = 0; u < n_slots; ++u) {
        const int64_t g = ring_pos + u;
        const int st = (int)(g % kStages);
        const int64_t x0 = c_lo + u * kSlot;
        const int64_t xw = x0 + warp * kPerWarp;  // this warp's 512 entries
        const int64_t nw = min((int64_t)kPerWarp, c_hi - xw);  // (<= 0: none)
        if (vec_) {
          if (!__all_sync(0xffffffffu, ok && mbar_wait(&full[st], (uint32_t)((g / kStages) & 1)))) ok = false;
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
        const bool chunk_end = (u + 1) % m == 0 || u + 1 == n_slots;
        if (chunk_end || ((u + 1) & 31) == 0) {
          uint64_t cs = combine(sh, sl);
          sh = sl = 0;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
          tot += cs;
          if (chunk_end && lane == 0) csum[(u / m) * kWarps + warp] = tot;
        }
      }
      if (lane == 0) part[warp] = tot;
    }
    if (warp == kProducer && lane == 0 && vec_) {
      // the copies this thread issued have landed before anything moves on
      for (int64_t g = max(ring_pos, ring_pos + n_slots - kStages); g < ring_pos + n_slots; ++g)
        if (!mbar_wait(&full[g % kStages], (uint32_t)((g / kStages) & 1))) ok = false;
    }
    if (vec_) ring_pos += n_slots;  // (the barriers' phases advance only on this path)
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t h = 0;
      for (int w = 0; w < kWarps; ++w) h += part[w];
      halves[rank] = h;
    }
    cl.sync();  // both halves' totals are written
    if (threadIdx.x == 0) halves[rank ^ 1u] = cl.map_shared_rank(halves, rank ^ 1u)[rank ^ 1u];
    cl.sync();  // the remote read is done before either CTA rewrites halves[] or exits
    return halves[0] + halves[1];
  };

  int i = 0;
  const float* pr = nullptr;
  const float* qr = nullptr;
  bool vec = false;
  uint64_t Z = 0;
  while (true) {
    // ---- in-order acceptance, up to the first rejection: warp 0 tests 32
    // candidates at once (their loads in parallel), the lowest failing lane wins
    if (warp == 0) {
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
      }
    }
    __syncthreads();
    i = state[0];
    const bool valid = state[1] != 0;
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
  const unsigned owner = T < halves[0] ? 0u : 1u;
  if (rank != owner) return;
  uint64_t c = owner == 0 ? 0 : halves[0];
  // the chunk, then (one-slot chunks) the warp's 512 entries holding T; the
  // chunk sums are differences of the warps' running totals
  const int64_t n_ch = (n_slots + m - 1) / m;
  int64_t ch = 0;
  uint64_t prev[kWarps];
#pragma unroll
  for (int w = 0; w < kWarps; ++w) prev[w] = 0;
  for (; ch < n_ch - 1; ++ch) {
    uint64_t cs = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) cs += csum[ch * kWarps + w] - prev[w];
    if (c + cs > T) break;
    c += cs;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) prev[w] = csum[ch * kWarps + w];
  }
  int64_t L0 = c_lo + ch * m * kSlot;
  int64_t L1 = min(c_hi, L0 + m * kSlot);
  if (m == 1) {
    int w = 0;
    for (; w < kWarps - 1; ++w) {
      const uint64_t ws = csum[ch * kWarps + w] - prev[w];
      if (c + ws > T) break;
      c += ws;
    }
    L0 = min(c_hi, L0 + (int64_t)w * kPerWarp);
    L1 = min(c_hi, L0 + kPerWarp);
  }
  // ---- one scan of [L0, L1) over the whole CTA, kThreads entries at a time
  // (prefix sums grow along the vocabulary, so the entries past T are a
  // suffix: the first of them is the count of those before it) ----
  int64_t found = -1;
  for (int64_t x0 = L0; x0 < L1; x0 += kThreads) {
    const int64_t x = x0 + threadIdx.x;
    uint64_t v = x < L1 ? weight(pr, qr, x) : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {  // inclusive prefix sum over the lanes
      const uint64_t y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += y;
    }
    if (lane == 31) wtot[warp] = v;
    __syncthreads();
    uint64_t before = c, chunk = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWarps + 1; ++w2) {
      before += w2 < warp ? wtot[w2] : 0;
      chunk += wtot[w2];
    }
    const int nvalid = (int)min((int64_t)kThreads, L1 - x0);
    // (the barrier also ends every thread's reads of wtot)
    const int ahead = __syncthreads_count(x < L1 && before + v <= T);
    if (ahead < nvalid) {
      found = x0 + ahead;
      break;
    }
    c += chunk;
  }
  if (threadIdx.x == 0) {
    n_out[(int64_t)b * n_sb] = i;
    tok_out[(int64_t)b * t_sb] = (int32_t)found;  // found >= 0: T < Z
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
