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
// A cluster of two CTAs per sequence, 16 warps each.  The vocabulary is cut
// into 32 contiguous slices (one per warp of the pair, 16-byte loads of 4
// entries per lane, eight loads in
// flight, when the rows are 16-byte aligned); the candidates are tested 32 at
// a time by one warp (the lowest rejected lane wins); the two CTAs exchange
// their slice sums through distributed shared memory, and the first one
// cuts the slice holding the threshold into 16, that piece once more, and
// scans the final piece with one warp's inclusive prefix sums.  Every pass reads its rows with plain
// coalesced loads: the row pair (p, q) of the chosen position is the only
// vocabulary-sized traffic (twice for the slice re-reads, from L2).
#include <cooperative_groups.h>

#include <cstdint>

#include "kernels.h"

namespace blkattn {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kCluster = 2;                 // CTAs per sequence
constexpr int kParts = kCluster * kWarps;   // first-level slices
constexpr float kTwo20 = 1048576.0f;         // 2^20
constexpr float kTwo40 = 1099511627776.0f;   // 2^40
constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23: x + kMagic holds integer |x| < 2^22 in its low bits
constexpr int kMagicBits = 0x4B400000;

// Weight F(m) = floor(m 2^40) of one entry, m = clamp(p - q, 0, 2) with the
// exact difference (has_q) or m = clamp(p, 0, 2), added to the lane's 32-bit
// counters as F = sh 2^20 + sl:
//   hi = fl(p - q), lo = (p - q) - hi         (TwoSum: exact for finite p, q)
//   h = floor(c 2^20) <= 2^21, r = c 2^40 - h 2^20 (exact), l = floor(r) < 2^20
//   for c = clamp(hi, 0, 2), and F = h 2^20 + l + e with
//   e = floor(lo 2^40) when 0 < hi <= 2 and r == l (c 2^40 is an integer,
//   so F = c 2^40 + floor(lo 2^40)); e <= 0 when hi == 2 (m above 2 clamps);
//   e = 0 otherwise: hi <= 0 means m <= 0 (|lo| < |hi|), hi > 2 means m > 2,
//   and for a non-integer c 2^40, |lo| 2^40 <= ulp(c 2^40) / 2 keeps it
//   between the same integers.  |e| <= 2^17 (|lo| <= ulp(hi) / 2 <= 2^-23).
// NaN masses count as 0 (fmaxf skips NaN), +inf as 2.
__device__ __forceinline__ void add_entry(float pv, float qv, bool has_q, int& sh, int& sl) {
  float hi = pv, e = 0.f;
  if (has_q) {
    hi = __fsub_rn(pv, qv);
    const float bb = __fsub_rn(hi, pv);  // the part of hi that came from -q
    const float lo = __fadd_rn(__fsub_rn(pv, __fsub_rn(hi, bb)), __fsub_rn(-qv, bb));
    e = floorf(lo * kTwo40);
    if (hi >= 2.f) e = fminf(e, 0.f);
    if (!(hi > 0.f && hi <= 2.f)) e = 0.f;
  }
  const float c = fminf(fmaxf(hi, 0.f), 2.f);
  const float h = floorf(c * kTwo20);
  const float r = fmaf(h, -kTwo20, c * kTwo40);
  const float l = floorf(r);
  if (r != l) e = 0.f;
  sh += __float_as_int(h + kMagic) - kMagicBits;
  sl += __float_as_int((l + e) + kMagic) - kMagicBits;  // l + e exact: |l + e| < 2^21
}
// (sl may be negative: l + e < 0 when l = 0 and lo < 0)
__device__ __forceinline__ uint64_t combine(int sh, int sl) {
  return (uint64_t)((int64_t)sh * (1 << 20) + (int64_t)sl);
}

// weight of entry x of the residual of (p, q) (q == nullptr: of p itself)
__device__ __forceinline__ uint64_t weight(const float* p, const float* q, int64_t x) {
  int sh = 0, sl = 0;
  add_entry(__ldg(p + x), q != nullptr ? __ldg(q + x) : 0.f, q != nullptr, sh, sl);
  return combine(sh, sl);
}

// Boundary w of a cut of [L0, L0 + n) into `parts` parts, on multiples of 4
// (L0 is one): the vector loads of a part never straddle two parts.
__device__ __forceinline__ int64_t cut(int64_t L0, int64_t n, int w, int parts = kWarps) {
  return w >= parts ? L0 + n : L0 + ((n * w / parts) & ~(int64_t)3);
}

// sum of the weights of [lo, hi) by one warp.  A lane's 32-bit counters
// take at most 2^9 entries between folds into its 64-bit sum (2^9 (2^21 +
// 2^20 + 2^17) < 2^31).
__device__ __forceinline__ uint64_t warp_sum(const float* p, const float* q, int64_t lo, int64_t hi, int lane,
                                             bool vec) {
  uint64_t s = 0;
  int64_t x = lo;
  const bool hq = q != nullptr;
  if (vec) {  // 16-byte loads: 128 entries per warp step (lo is a multiple of 4)
    const int64_t hv = lo + ((hi - lo) & ~(int64_t)127);
    for (int64_t xb = lo; xb < hv; xb += 128 * 64) {  // 64 steps = 256 entries per lane per fold
      const int64_t xe = min(hv, xb + 128 * 64);
      int sh = 0, sl = 0;
#pragma unroll 8
      for (int64_t x0 = xb + 4 * lane; x0 < xe; x0 += 128) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p + x0));
        const float4 c = hq ? __ldg(reinterpret_cast<const float4*>(q + x0)) : make_float4(0.f, 0.f, 0.f, 0.f);
        add_entry(a.x, c.x, hq, sh, sl);
        add_entry(a.y, c.y, hq, sh, sl);
        add_entry(a.z, c.z, hq, sh, sl);
        add_entry(a.w, c.w, hq, sh, sl);
      }
      s += combine(sh, sl);
    }
    x = hv;
  }
  {
    int sh = 0, sl = 0, n = 0;
    for (int64_t y = x + lane; y < hi; y += 32) {
      add_entry(__ldg(p + y), hq ? __ldg(q + y) : 0.f, hq, sh, sl);
      if (++n == 256) {
        s += combine(sh, sl);
        sh = sl = n = 0;
      }
    }
    s += combine(sh, sl);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    spec_sample_kernel(const float* __restrict__ p, int64_t p_sb, int64_t p_si, const float* __restrict__ q,
                       int64_t q_sb, int64_t q_si, const int32_t* __restrict__ draft, int64_t d_sb, int64_t d_si,
                       const float* __restrict__ u_acc, int64_t u_sb, int64_t u_si,
                       const int32_t* __restrict__ u_smp, int64_t s_sb, int k, int64_t V,
                       int32_t* __restrict__ n_out, int64_t n_sb, int32_t* __restrict__ tok_out, int64_t t_sb) {
  namespace cg = cooperative_groups;
  __shared__ uint64_t part[kWarps];     // this CTA's slice (or piece) sums
  __shared__ uint64_t allpart[kParts];  // the first-level slice sums of the pair
  __shared__ int64_t bounds[2];  // the current search range [lo, hi)
  __shared__ uint64_t base;      // prefix sum before lo
  __shared__ int state[2];       // [0] first position not kept, [1] its candidate is possible
  cg::cluster_group cl = cg::this_cluster();
  const unsigned rank = cl.block_rank();
  const int b = blockIdx.x / kCluster;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t s = (uint32_t)u_smp[(int64_t)b * s_sb];

  // Z of a whole row: each CTA sums its 16 slices, the pair exchanges them
  auto row_sum = [&](const float* pr_, const float* qr_, bool vec_) -> uint64_t {
    const int sl = (int)rank * kWarps + warp;
    const uint64_t ws = warp_sum(pr_, qr_, cut(0, V, sl, kParts), cut(0, V, sl + 1, kParts), lane, vec_);
    if (lane == 0) part[warp] = ws;
    cl.sync();  // both CTAs' slice sums are written
    if (threadIdx.x < kParts)
      allpart[threadIdx.x] = cl.map_shared_rank(part, threadIdx.x / kWarps)[threadIdx.x % kWarps];
    cl.sync();  // the remote reads are done before either CTA rewrites part[] or exits
    uint64_t z = 0;
#pragma unroll
    for (int w = 0; w < kParts; ++w) z += allpart[w];
    return z;
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
        bool keep = true, ok = false;
        if (jj < k) {
          const int x = draft[(int64_t)b * d_sb + (int64_t)jj * d_si];
          keep = false;
          if (x >= 0 && (int64_t)x < V) {  // otherwise it cannot have been proposed
            const double px = (double)p[(int64_t)b * p_sb + (int64_t)jj * p_si + x];
            const double qx = (double)q[(int64_t)b * q_sb + (int64_t)jj * q_si + x];
            const double u = (double)u_acc[(int64_t)b * u_sb + (int64_t)jj * u_si];
            ok = qx > 0.0;
            keep = ok && u * qx < px;
          }
        }
        const unsigned stop = __ballot_sync(0xffffffffu, !keep);
        if (stop != 0u) {
          const int l = __ffs(stop) - 1;
          j = j0 + l;
          valid = __shfl_sync(0xffffffffu, (int)ok, l);
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
    // ---- Z: the 32 slice sums of the pair ----
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
    __syncthreads();  // every thread has read state[] and part[]
  }
  if (rank != 0) return;  // the first CTA of the pair finishes the draw
  if (Z == 0) {  // the distribution drawn from has no mass above 2^-40: token 0 by definition
    if (threadIdx.x == 0) {
      n_out[(int64_t)b * n_sb] = i;
      tok_out[(int64_t)b * t_sb] = 0;
    }
    return;
  }
  const uint64_t T = __umul64hi((uint64_t)s << 32, Z);  // floor(s Z / 2^32) < Z

  // ---- level 1: the slice holding T ----
  if (threadIdx.x == 0) {
    uint64_t c = 0;
    int w = 0;
    for (; w < kParts - 1; ++w) {
      if (c + allpart[w] > T) break;
      c += allpart[w];
    }
    bounds[0] = cut(0, V, w, kParts);
    bounds[1] = cut(0, V, w + 1, kParts);
    base = c;
  }
  __syncthreads();
  // ---- level 2: cut that slice into 16 pieces ----
  {
    // (and level 3: cut the chosen piece into 16 once more)
    for (int level = 0; level < 2; ++level) {
      const int64_t L0 = bounds[0], L1 = bounds[1], n = L1 - L0;
      const int64_t lo = cut(L0, n, warp), hi = cut(L0, n, warp + 1);
      const uint64_t ws = warp_sum(pr, qr, lo, hi, lane, vec);
      __syncthreads();  // everyone has read bounds
      if (lane == 0) part[warp] = ws;
      __syncthreads();
      if (threadIdx.x == 0) {
        uint64_t c = base;
        int w = 0;
        for (; w < kWarps - 1; ++w) {
          if (c + part[w] > T) break;
          c += part[w];
        }
        bounds[0] = cut(L0, n, w);
        bounds[1] = cut(L0, n, w + 1);
        base = c;
      }
      __syncthreads();
    }
  }
  // ---- last level: one warp scans the piece, 32 entries at a time ----
  if (warp == 0) {
    uint64_t c = base;
    int64_t found = -1;
    for (int64_t x0 = bounds[0]; x0 < bounds[1] && found < 0; x0 += 32) {
      const int64_t x = x0 + lane;
      uint64_t v = x < bounds[1] ? weight(pr, qr, x) : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {  // inclusive prefix sum over the lanes
        const uint64_t y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, x < bounds[1] && c + v > T);
      if (hit != 0u) found = x0 + (__ffs(hit) - 1);
      c += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
      n_out[(int64_t)b * n_sb] = i;
      tok_out[(int64_t)b * t_sb] = (int32_t)found;  // found >= 0: T < Z
    }
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
  blkattn::spec_sample_kernel<<<(unsigned)(B * blkattn::kCluster), blkattn::kThreads, 0,
                                 reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const float*>(p->data), p->strides[0], p->strides[1], static_cast<const float*>(q->data),
      q->strides[0], q->strides[1], static_cast<const int32_t*>(draft->data), draft->strides[0], draft->strides[1],
      static_cast<const float*>(u_accept->data), u_accept->strides[0], u_accept->strides[1],
      static_cast<const int32_t*>(u_sample->data), u_sample->strides[0], (int)k, V,
      static_cast<int32_t*>(n_accepted->data), n_accepted->strides[0], static_cast<int32_t*>(token->data),
      token->strides[0]);
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return blkattn::report_cuda_failure(e);
  return BLKATTN_OK;
}
