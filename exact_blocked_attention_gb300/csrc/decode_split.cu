// Split-KV decode / verify kernel (CUDA-core arithmetic).
//
// Exact blocked attention of "Chapter 33: inference compute optimisation"
// §33.2: each CTA owns the query rows of ONE KV head that share it (the G
// grouped query heads x T_q rows, packed so K/V are read once per KV head) and
// one split (a contiguous key range) of the cache.  It streams the split's K/V
// rows into a shared-memory ring with bulk asynchronous copies (a dedicated
// producer warp, mbarrier-synchronised, no multicast) and runs Algorithm 33.1
// on it: per 16-key sub-block a consumer warp forms the scores, applies the
// visibility rule by SELECT (never by adding a mask to garbage rows), takes
// the block statistics of eq. 33.3 and folds them into its running
// (m, l, u) with eqs. 33.4–33.5, using an explicit "no valid key yet" flag
// (m == -inf is only tested, never subtracted).  The consumer warps' states
// are then merged with the same rule.  A split whose rows see keys in only
// this split writes the final o = u / l and lse directly; otherwise it writes
// its partial state for the split-merge kernel.
//
// Scores are carried in base-2 units (z * log2 e) so that exponentials are
// single ex2 instructions; lse is converted back to natural-log units.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace blkattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

template <typename T>
struct EltTraits;
template <>
struct EltTraits<__nv_bfloat16> {
  static constexpr int kBytes = 2;
};
template <>
struct EltTraits<float> {
  static constexpr int kBytes = 4;
};

// 16 bytes of K (8 bf16 or 4 f32) -> floats
template <typename T>
__device__ __forceinline__ void unpack16(const uint4 w, float* f);
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 w, float* f) {
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
  f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
  f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 w, float* f) {
  f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
  f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
}

// DPL consecutive elements of a V row -> floats
template <typename T, int DPL>
__device__ __forceinline__ void load_v(const unsigned char* src, float* f) {
  if constexpr (EltTraits<T>::kBytes == 2) {
    if constexpr (DPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
      f[0] = bf16lo(w); f[1] = bf16hi(w);
    }
  } else {
    if constexpr (DPL == 4) {
      const float4 w = *reinterpret_cast<const float4*>(src);
      f[0] = w.x; f[1] = w.y; f[2] = w.z; f[3] = w.w;
    } else {
      const float2 w = *reinterpret_cast<const float2*>(src);
      f[0] = w.x; f[1] = w.y;
    }
  }
}

template <typename T>
__device__ __forceinline__ float load_elt(const void* base, int64_t idx) {
  if constexpr (EltTraits<T>::kBytes == 2)
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
  else
    return static_cast<const float*>(base)[idx];
}

template <typename T, int D, int R, int NW, int STAGES>
struct DecodeLayout {
  static constexpr int kRowBytes = D * EltTraits<T>::kBytes;
  static constexpr int kRowPad = kRowBytes + 16;  // 16 B skew: conflict-free key-per-lane reads
  static constexpr int kTile = 16 * NW;           // keys per stage
  static constexpr int kStageBytes = 2 * kTile * kRowPad;
  static constexpr int kQRow = D + 4;             // floats; 16 B gap between the two halves
  static constexpr int kKvBytes = STAGES * kStageBytes;
  static constexpr int kQOff = kKvBytes;
  static constexpr int kPOff = kQOff + R * kQRow * 4;
  static constexpr int kBarOff = (kPOff + NW * 16 * R * 4 + 15) / 16 * 16;
  static constexpr int kMiscOff = kBarOff + 2 * STAGES * 8;
  static constexpr int kBytes = kMiscOff + 16;
  // cross-warp reduction area (reuses the K/V ring once every copy has landed)
  static constexpr int kRedBytes = NW * R * (D + 2) * 4;
  static_assert(kRedBytes <= kKvBytes, "reduction area must fit in the ring");
};

template <typename T, int D, int R, int NW, int STAGES>
__global__ void __launch_bounds__((NW + 1) * 32)
    decode_split_kernel(const FwdParams p) {
  using L = DecodeLayout<T, D, R, NW, STAGES>;
  constexpr int kRowBytes = L::kRowBytes;
  constexpr int kRowPad = L::kRowPad;
  constexpr int kTile = L::kTile;
  constexpr int CH = kRowBytes / 16;        // 16-byte chunks per row
  constexpr int EPC = 16 / EltTraits<T>::kBytes;
  constexpr int HALF = D / 2;
  constexpr int DPL = D / 32;               // value dims per lane in the PV product

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  float* q_s = reinterpret_cast<float*>(smem + L::kQOff);
  float* p_s = reinterpret_cast<float*>(smem + L::kPOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  int* issued_s = reinterpret_cast<int*>(smem + L::kMiscOff);
  int* timeout_s = issued_s + 1;

  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int b = blockIdx.z / p.row_groups;
  const int rg = blockIdx.z % p.row_groups;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- visibility bookkeeping (integers, identical in every thread) ----
  int len = p.seqlens[b * p.sl_s];
  len = len < 0 ? 0 : (len > p.Tmax ? p.Tmax : len);
  int row_end[R];  // keys [0, row_end) pass the length and position tests
  int row_h[R], row_i[R];
  int cta_end = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int pk = rg * R + r;
    row_end[r] = 0;
    row_h[r] = 0;
    row_i[r] = 0;
    if (pk < p.rows_per_head) {
      const int g = pk / p.Tq;
      const int i = pk - g * p.Tq;
      row_h[r] = hk * p.G + g;
      row_i[r] = i;
      const int pos = p.qpos[b * p.qp_sb + i * p.qp_si];
      const int e = pos < 0 ? 0 : (pos >= len ? len : pos + 1);
      row_end[r] = e;
      cta_end = e > cta_end ? e : cta_end;
    }
  }
  const int k0 = split * p.chunk;
  // Split 0 always runs: it writes the rows that no split sees.
  if (split > 0 && k0 >= cta_end) return;
  const int k1 = min(k0 + p.chunk, cta_end);
  const int n_tiles = k1 > k0 ? (k1 - k0 + kTile - 1) / kTile : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    *issued_s = 0;
    *timeout_s = 0;
    fence_barrier_init();
  }
  // query rows -> shared memory as f32 (exact widening), zero for absent rows
  for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
    const int r = idx / D;
    const int d = idx - r * D;
    float val = 0.f;
    const int pk = rg * R + r;
    if (pk < p.rows_per_head) {
      const int g = pk / p.Tq;
      const int i = pk - g * p.Tq;
      val = load_elt<T>(p.q, (int64_t)b * p.q_sb + (int64_t)(hk * p.G + g) * p.q_sh +
                                 (int64_t)i * p.q_si + (int64_t)d * p.q_sd);
    }
    q_s[r * L::kQRow + (d < HALF ? d : d + 4)] = val;
  }
  __syncthreads();

  // per-warp running state (base-2 units)
  float m_run[R];
  float l_lane[R];  // this lane's share of l (lanes 0..15 count)
  float u[R][DPL];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m_run[r] = kNegInf;
    l_lane[r] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) u[r][e] = 0.f;
  }

  if (warp == NW) {
    // ---------------- producer warp: bulk copies of K and V rows ----------------
    const uint64_t pol = policy_evict_first();
    const char* kbase = p.k + (int64_t)b * p.k_sb + (int64_t)hk * p.k_sh;
    const char* vbase = p.v + (int64_t)b * p.v_sb + (int64_t)hk * p.v_sh;
    int t = 0;
    for (; t < n_tiles; ++t) {
      const int st = t % STAGES;
      if (t >= STAGES) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[st], ((t / STAGES) - 1) & 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) { record_error(p.err, kErrTimeout); *timeout_s = 1; }
          break;
        }
      }
      const int key0 = k0 + t * kTile;
      const int nrows = min(kTile, k1 - key0);
      unsigned char* kdst = ring + st * L::kStageBytes;
      unsigned char* vdst = kdst + kTile * kRowPad;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * nrows * kRowBytes));
      __syncwarp();
      for (int r = lane; r < nrows; r += 32) {
        bulk_g2s(kdst + r * kRowPad, kbase + (int64_t)(key0 + r) * p.k_st, kRowBytes, &full[st], pol);
        bulk_g2s(vdst + r * kRowPad, vbase + (int64_t)(key0 + r) * p.v_st, kRowBytes, &full[st], pol);
      }
    }
    if (lane == 0) *issued_s = t;
  } else {
    // ---------------- consumer warps ----------------
    const int kk = lane & 15;    // key slot within the warp's 16 keys
    const int half = lane >> 4;  // which half of the head dimension this lane sums
    int row_hi[R];               // split-local end of the visible range per row
#pragma unroll
    for (int r = 0; r < R; ++r) row_hi[r] = min(row_end[r], k0 + p.chunk);
    // token tree: keys from tbase on are seen only where the row's mask says
    const int tbase = p.tree != nullptr ? len - p.Tq : 0x7fffffff;
    uint64_t row_tree[R];
    int row_lo[R];  // sliding window: each row's first visible key
#pragma unroll
    for (int r = 0; r < R; ++r) {
      row_tree[r] = p.tree != nullptr ? (uint64_t)p.tree[(int64_t)b * p.tr_sb + (int64_t)row_i[r] * p.tr_si] : ~0ull;
      row_lo[r] = 0;
      if (p.window > 0) {  // (pos >= 0 first: the difference cannot overflow)
        const int ps = p.qpos[b * p.qp_sb + row_i[r] * p.qp_si];
        row_lo[r] = ps < 0 ? 0 : max(0, ps - p.window + 1);
      }
    }

    for (int t = 0; t < n_tiles; ++t) {
      const int st = t % STAGES;
      const bool ok = mbar_wait(&full[st], (t / STAGES) & 1);
      if (!ok) {
        if (lane == 0) { record_error(p.err, kErrTimeout); *timeout_s = 1; }
        break;
      }
      const int tile_k0 = k0 + t * kTile;
      const int key = tile_k0 + warp * 16 + kk;
      const unsigned char* kst = ring + st * L::kStageBytes;
      const unsigned char* vst = kst + kTile * kRowPad;

      // scores: lane pair (kk, kk+16) splits one key's dot product in halves
      float acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = 0.f;
      const unsigned char* krow = kst + (warp * 16 + kk) * kRowPad + half * (kRowBytes / 2);
      const float* qh = q_s + half * (HALF + 4);
#pragma unroll
      for (int c = 0; c < CH / 2; ++c) {
        float kf[EPC];
        unpack16<T>(*reinterpret_cast<const uint4*>(krow + c * 16), kf);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float* qc = qh + r * L::kQRow + c * EPC;
#pragma unroll
          for (int e4 = 0; e4 < EPC; e4 += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(qc + e4);
            acc[r] = fmaf(qv.x, kf[e4 + 0], acc[r]);
            acc[r] = fmaf(qv.y, kf[e4 + 1], acc[r]);
            acc[r] = fmaf(qv.z, kf[e4 + 2], acc[r]);
            acc[r] = fmaf(qv.w, kf[e4 + 3], acc[r]);
          }
        }
      }
      float s[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], 16);
        bool vis = key < row_hi[r] && key >= row_lo[r];
        if (key >= tbase) {
          const int node = key - tbase;
          vis = vis && node < 64 && ((row_tree[r] >> (node & 63)) & 1ull);
        }
        float bias = 0.f;
        if (p.bias != nullptr && vis) {
          bias = p.bias[(int64_t)b * p.bi_sb + (int64_t)row_h[r] * p.bi_sh +
                        (int64_t)row_i[r] * p.bi_si + (int64_t)key * p.bi_sj];
          vis = bias != kNegInf;
        }
        s[r] = vis ? fmaf(acc[r], p.scale_log2, bias * kLog2e) : kNegInf;
      }

      // block statistics and the online merge (eqs. 33.3-33.5, valid flags)
      float pr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float mt = s[r];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        pr[r] = 0.f;
        if (mt != kNegInf) {  // this block has a valid key for row r
          const float m_new = fmaxf(m_run[r], mt);
          const float alpha = (m_run[r] == kNegInf) ? 0.f : fast_exp2(m_run[r] - m_new);
          pr[r] = (s[r] == kNegInf) ? 0.f : fast_exp2(s[r] - m_new);
          m_run[r] = m_new;
          l_lane[r] = fmaf(l_lane[r], alpha, pr[r]);
#pragma unroll
          for (int e = 0; e < DPL; ++e) u[r][e] *= alpha;
        }
      }
      float* pw = p_s + warp * 16 * R;
      if (lane < 16) {
#pragma unroll
        for (int r = 0; r < R; ++r) pw[kk * R + r] = pr[r];
      }
      __syncwarp();
      // PV over this warp's keys that were loaded (never the rows past k1)
      int nk = k1 - (tile_k0 + warp * 16);
      nk = nk < 0 ? 0 : (nk > 16 ? 16 : nk);
      const unsigned char* vrow = vst + (warp * 16) * kRowPad + lane * DPL * EltTraits<T>::kBytes;
#pragma unroll 4
      for (int j = 0; j < nk; ++j) {
        float vf[DPL];
        load_v<T, DPL>(vrow + j * kRowPad, vf);
        float pj[R];
        if constexpr (R % 4 == 0) {
#pragma unroll
          for (int r4 = 0; r4 < R; r4 += 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(pw + j * R + r4);
            pj[r4] = t4.x; pj[r4 + 1] = t4.y; pj[r4 + 2] = t4.z; pj[r4 + 3] = t4.w;
          }
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) pj[r] = pw[j * R + r];
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < DPL; ++e) u[r][e] = fmaf(pj[r], vf[e], u[r][e]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // this warp's l: sum of the 16 key slots
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float l = (lane < 16) ? l_lane[r] : 0.f;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      l_lane[r] = l;
    }
  }

  // the split-merge grid may start launching now (it waits for this grid's
  // completion before reading anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- drain: every issued copy must have landed before the ring is reused ----
  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = *issued_s;
    for (int t = issued - STAGES < 0 ? 0 : issued - STAGES; t < issued; ++t)
      if (!mbar_wait(&full[t % STAGES], (t / STAGES) & 1)) {
        record_error(p.err, kErrTimeout);
        *timeout_s = 1;
      }
  }
  __syncthreads();
  if (*timeout_s) return;

  // ---- merge the consumer warps' states (eqs. 33.4-33.5) ----
  float* red_m = reinterpret_cast<float*>(ring);  // [NW][R]
  float* red_l = red_m + NW * R;                   // [NW][R]
  float* red_u = red_l + NW * R;                   // [NW][R][D]
  if (warp < NW) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (lane == 0) {
        red_m[warp * R + r] = m_run[r];
        red_l[warp * R + r] = l_lane[r];
      }
#pragma unroll
      for (int e = 0; e < DPL; ++e) red_u[(warp * R + r) * D + lane * DPL + e] = u[r][e];
    }
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
    const int r = idx / D;
    const int d = idx - r * D;
    const int pk = rg * R + r;
    if (pk >= p.rows_per_head) continue;
    // recomputed here (runtime r) so the per-row arrays stay in registers
    const int g = pk / p.Tq;
    const int ri = pk - g * p.Tq;
    const int rh = hk * p.G + g;
    const int rpos = p.qpos[b * p.qp_sb + ri * p.qp_si];
    const int rend = rpos < 0 ? 0 : (rpos >= len ? len : rpos + 1);
    // no key of this row lies in this split: only split 0 has to write it
    if (k0 >= rend && split != 0) continue;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * R + r]);
    float Ls = 0.f, Us = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = red_m[w * R + r];
        if (mw == kNegInf) continue;  // empty warp state: contributes nothing
        const float c = fast_exp2(mw - M);
        Ls = fmaf(c, red_l[w * R + r], Ls);
        Us = fmaf(c, red_u[(w * R + r) * D + d], Us);
      }
    }
    const int64_t row = ((int64_t)b * p.Hq + rh) * p.Tq + ri;
    const int n_active = (rend + p.chunk - 1) / p.chunk;
    if (n_active <= 1) {
      // the whole visible range of this row is in split 0: final result
      const float o = (M == kNegInf) ? 0.f : Us / Ls;
      const int64_t oi = (int64_t)b * p.o_sb + (int64_t)rh * p.o_sh +
                         (int64_t)ri * p.o_si + (int64_t)d * p.o_sd;
      if (p.out_bf16)
        static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
      else
        static_cast<float*>(p.out)[oi] = o;
      if (d == 0)
        p.lse[(int64_t)b * p.l_sb + (int64_t)rh * p.l_sh + (int64_t)ri * p.l_si] =
            (M == kNegInf) ? kNegInf : (M + __log2f(Ls)) * kLn2;
    } else {
      const int64_t wi = row * p.n_splits + split;
      p.ws_u[wi * D + d] = Us;
      if (d == 0) {
        p.ws_m[wi] = M;
        p.ws_l[wi] = Ls;
      }
    }
  }
}

template <typename T, int D, int R, int NW, int STAGES>
cudaError_t launch_one(const FwdParams& p, const DecodeConfig& cfg, cudaStream_t stream) {
  using L = DecodeLayout<T, D, R, NW, STAGES>;
  auto kern = decode_split_kernel<T, D, R, NW, STAGES>;
  static bool attr_set = false;  // per instantiation (one device per process is assumed per call)
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(cfg.n_splits, p.Hkv, p.B * cfg.row_groups);
  kern<<<grid, (NW + 1) * 32, L::kBytes, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int D, int NW, int STAGES>
cudaError_t dispatch_rows(const FwdParams& p, const DecodeConfig& cfg, cudaStream_t s) {
  switch (cfg.rows_per_cta) {
    case 1: return launch_one<T, D, 1, NW, STAGES>(p, cfg, s);
    case 2: return launch_one<T, D, 2, NW, STAGES>(p, cfg, s);
    case 4: return launch_one<T, D, 4, NW, STAGES>(p, cfg, s);
    case 8: return launch_one<T, D, 8, NW, STAGES>(p, cfg, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// The decode kernel runs 4 consumer warps (64-key stages); 3 stages for
// 16-bit rows of 128 (two CTAs fit an SM), 2 stages for 512-byte f32 rows.
size_t decode_smem_bytes(Elt elt, int d, const DecodeConfig& cfg) {
  const int rb = d * (elt == Elt::BF16 ? 2 : 4);
  const int tile = 16 * cfg.warps;
  size_t bytes = (size_t)cfg.stages * 2 * tile * (rb + 16);
  bytes += (size_t)cfg.rows_per_cta * (d + 4) * 4 + (size_t)cfg.warps * 16 * cfg.rows_per_cta * 4;
  return bytes + 2 * cfg.stages * 8 + 32;
}

cudaError_t launch_decode_split(const FwdParams& p, Elt elt, int d, const DecodeConfig& cfg,
                                cudaStream_t stream) {
  if (cfg.warps != 4) return cudaErrorInvalidValue;
  if (elt == Elt::BF16) {
    if (cfg.stages != 3) return cudaErrorInvalidValue;
    if (d == 128) return dispatch_rows<__nv_bfloat16, 128, 4, 3>(p, cfg, stream);
    if (d == 64) return dispatch_rows<__nv_bfloat16, 64, 4, 3>(p, cfg, stream);
  } else {
    if (cfg.stages != 2) return cudaErrorInvalidValue;
    if (d == 128) return dispatch_rows<float, 128, 4, 2>(p, cfg, stream);
    if (d == 64) return dispatch_rows<float, 64, 4, 2>(p, cfg, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace blkattn
