// Causal prefill kernel on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Exact blocked attention ("Chapter 33: inference compute optimisation"
// §33.2, Algorithm 33.1; §33.3 for the on-chip tiling and the skipping of
// fully invisible blocks): one CTA owns 128 consecutive query rows of one
// head and walks the key tiles of 64 keys that hold any key visible to them,
// keeping per row the statistics (m, l, u) of eq. 33.3 with u in tensor
// memory.  Key tiles beyond the CTA's last visible key are never loaded.
//
//   S_j  = Q K_j^T         tcgen05.mma M=128 N=64  K=16 x 8   (smem x smem -> TMEM)
//   U   += P_j V_j         tcgen05.mma M=128 N=128 K=16 x 4 x 2 (P from TMEM, V smem)
//
// Roles (192 threads): warps 0-3 = one thread per query row (TMEM lane):
// scores, mask by select, online statistics, P; warp 4 = TMA producer (Q
// once, K/V tiles into a 2-stage ring); warp 5 = TMEM allocation and the
// single thread that issues every MMA.  Two S buffers let S_{j+1} be formed
// while the rows work on S_j; P_j is written back over S_j's columns as
// bf16 P_hi and P_lo (P = P_hi + P_lo to ~16 bits, so the PV product keeps
// ~2^-17 relative accuracy although P is not an input).
//
// Online rescaling is lazy: a row keeps its reference maximum m until a tile
// raises the row maximum by more than 8 (base-2 units); only then is its U
// row rescaled in TMEM (after the previous PV product has completed).  With
// any reference m >= (true max - 8) the state (m, l, u) still represents the
// same set (eqs. 33.4-33.5 hold for any common reference), and P <= 2^8.
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

constexpr int BM = 128;  // query rows per CTA (TMEM lanes)
constexpr int BN = 64;   // keys per tile
constexpr int D = 128;   // head dim
constexpr int STAGES = 2;
constexpr int kQBox = BM * 128;    // one 64-dim (128-byte) box of Q: 16 KB
constexpr int kKVBox = BN * 128;   // one 64-dim box of a K or V tile: 8 KB
constexpr int kQBytes = 2 * kQBox;
constexpr int kKVTile = 2 * kKVBox;
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + STAGES * kKVTile;
constexpr int kOffBar = kOffV + STAGES * kKVTile;
// q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full[2], o_done, drain
constexpr int kNumBars = 1 + 3 * STAGES + 6;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align to 1024
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;    // S buffers at [0, 64) and [64, 128); P_b over S_b
constexpr uint32_t kColO = 128;  // U (the unnormalised output) at [128, 256)
constexpr int kThreads = 192;
constexpr uint32_t kIdescQK = tc::idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16(BM, D, 0, 1);   // P (TMEM), V MN-major

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__global__ void __launch_bounds__(kThreads, 2)
    prefill_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + STAGES;
  uint64_t* kv_empty = v_full + STAGES;
  uint64_t* s_full = kv_empty + STAGES;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  int* misc = reinterpret_cast<int*>(sm + kOffMisc);  // tmem base, cta_end, cta_min, timeout

  const int qt = gridDim.x - 1 - blockIdx.x;  // the longest (latest) query tiles first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int hk = h / p.G;
  const int i0 = qt * BM;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- visibility of this CTA's rows (integers) ----
  int len = p.seqlens[b * p.sl_s];
  len = len < 0 ? 0 : (len > p.Tmax ? p.Tmax : len);
  if (threadIdx.x == 0) {
    misc[1] = 0;
    misc[2] = 0x7fffffff;
    misc[3] = 0;
  }
  __syncthreads();
  int my_end = 0;
  bool my_row = false;
  if (warp < 4) {
    const int i = i0 + (int)threadIdx.x;
    if (i < p.Tq) {
      const int pos = p.qpos[b * p.qp_sb + i * p.qp_si];
      my_end = pos < 0 ? 0 : (pos >= len ? len : pos + 1);
      my_row = true;
      atomicMax(&misc[1], my_end);
      atomicMin(&misc[2], my_end);
    }
  }
  __syncthreads();
  const int cta_end = misc[1];
  const int cta_min = misc[2];
  const int n_tiles = (cta_end + BN - 1) / BN;
  const int64_t out_row = (int64_t)b * p.o_sb + (int64_t)h * p.o_sh + (int64_t)(i0 + (int)threadIdx.x) * p.o_si;
  const int64_t lse_idx = (int64_t)b * p.l_sb + (int64_t)h * p.l_sh + (int64_t)(i0 + (int)threadIdx.x) * p.l_si;
  if (n_tiles == 0) {  // no row of this tile sees any key: the defined output
    if (my_row) {
      for (int d = 0; d < D; ++d) {
        if (p.out_bf16)
          static_cast<__nv_bfloat16*>(p.out)[out_row + (int64_t)d * p.o_sd] = __float2bfloat16_rn(0.f);
        else
          static_cast<float*>(p.out)[out_row + (int64_t)d * p.o_sd] = 0.f;
      }
      p.lse[lse_idx] = kNegInf;
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);  // one arrival per row warp
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tc::alloc(reinterpret_cast<uint32_t*>(&misc[0]), kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = static_cast<uint32_t>(misc[0]);
  const uint32_t sQ = smem_u32(sm + kOffQ);
  const uint32_t sK = smem_u32(sm + kOffK);
  const uint32_t sV = smem_u32(sm + kOffV);

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();  // K/V tiles are re-read by the other query tiles
      mbar_arrive_expect_tx(q_full, kQBytes);
      tma_load_4d(sm + kOffQ, &tmq, 0, i0, h, b, q_full, pol_q);
      tma_load_4d(sm + kOffQ + kQBox, &tmq, 64, i0, h, b, q_full, pol_q);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % STAGES;
        if (j >= STAGES && !mbar_wait(&kv_empty[s], ((j / STAGES) - 1) & 1)) {
          record_error(p.err, kErrTimeout);
          misc[3] = 1;
          break;
        }
        const int key0 = j * BN;
        unsigned char* kd = sm + kOffK + s * kKVTile;
        unsigned char* vd = sm + kOffV + s * kKVTile;
        mbar_arrive_expect_tx(&k_full[s], kKVTile);
        tma_load_4d(kd, &tmk, 0, key0, hk, b, &k_full[s], pol_kv);
        tma_load_4d(kd + kKVBox, &tmk, 64, key0, hk, b, &k_full[s], pol_kv);
        mbar_arrive_expect_tx(&v_full[s], kKVTile);
        tma_load_4d(vd, &tmv, 0, key0, hk, b, &v_full[s], pol_kv);
        tma_load_4d(vd + kKVBox, &tmv, 64, key0, hk, b, &v_full[s], pol_kv);
        issued = j + 1;
      }
      // every issued copy must land before the CTA can exit
      if (!mbar_wait(q_full, 0)) misc[3] = 1;
      for (int j = issued - STAGES < 0 ? 0 : issued - STAGES; j < issued; ++j) {
        const int s = j % STAGES;
        if (!mbar_wait(&k_full[s], (j / STAGES) & 1) || !mbar_wait(&v_full[s], (j / STAGES) & 1)) {
          record_error(p.err, kErrTimeout);
          misc[3] = 1;
        }
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0);
      auto issue_pv = [&](int jj) -> bool {
        const int bb = jj & 1;
        const int ss = jj % STAGES;
        if (!mbar_wait(&v_full[ss], (jj / STAGES) & 1)) return false;
        if (!mbar_wait(&p_full[bb], (jj >> 1) & 1)) return false;
        tc::fence_after();
        const uint32_t vbase = sV + ss * kKVTile;
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // P_hi, then P_lo
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            // B = V rows [16ks, 16ks+16) (keys, K) x 128 dims (N, two 64-dim boxes 8 KB apart)
            const uint64_t bdesc = tc::smem_desc(vbase + ks * 16 * 128, kKVBox, 1024);
            const uint32_t acol = tb + kColS + 64 * bb + 32 * part + 8 * ks;
            tc::mma_ts(tb + kColO, acol, bdesc, kIdescPV, (jj > 0 || part > 0 || ks > 0) ? 1u : 0u);
          }
        }
        tc::commit(o_done);
        tc::commit(&kv_empty[ss]);
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int bb = j & 1;
        const int s = j % STAGES;
        if (!mbar_wait(&k_full[s], (j / STAGES) & 1)) { ok = false; break; }
        tc::fence_after();
        const uint32_t kbase = sK + s * kKVTile;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t adesc = tc::smem_desc(sQ + (ks >> 2) * kQBox + (ks & 3) * 32, 16, 1024);
          const uint64_t bdesc = tc::smem_desc(kbase + (ks >> 2) * kKVBox + (ks & 3) * 32, 16, 1024);
          tc::mma_ss(tb + kColS + 64 * bb, adesc, bdesc, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[bb]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && !issue_pv(n_tiles - 1)) ok = false;
      if (!ok) {
        record_error(p.err, kErrTimeout);
        misc[3] = 1;
      }
      // every MMA issued must complete before TMEM is released
      tc::commit(drain);
      if (!mbar_wait(drain, 0)) {
        record_error(p.err, kErrTimeout);
        misc[3] = 1;
      }
    }
  } else {
    // ---------------- rows: online softmax statistics ----------------
    const uint32_t tl = tb + ((uint32_t)(32 * warp) << 16);  // this warp's TMEM lane quarter
    float m_ref = kNegInf;  // reference maximum (base-2 units), -inf = no valid key yet
    float l = 0.f;
    bool ok = true;
    // waits are made warp-uniform: the tensor-memory accesses that follow
    // are warp-collective
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    for (int j = 0; j < n_tiles; ++j) {
      const int bb = j & 1;
      if (!wait_all(&s_full[bb], (j >> 1) & 1)) { ok = false; break; }
      tc::fence_after();
      uint32_t sa[32], sb2[32];
      tc::ld32(tl + kColS + 64 * bb, sa);
      tc::ld32(tl + kColS + 64 * bb + 32, sb2);
      tc::wait_ld();
      const int key0 = j * BN;
      const bool need_mask = key0 + BN > cta_min;
      float x[64];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = __uint_as_float(sa[c]) * p.scale_log2;
        x[32 + c] = __uint_as_float(sb2[c]) * p.scale_log2;
      }
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = (key0 + c < my_end) ? x[c] : kNegInf;
      }
      float mt = x[0];
#pragma unroll
      for (int c = 1; c < 64; ++c) mt = fmaxf(mt, x[c]);
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
        // U rows change reference: wait for the previous PV product, rescale.
        // (S_j being ready implies PV_{j-2} completed, so o_done is at phase
        // j-1 or j and the parity wait is unambiguous.)
        if (!wait_all(o_done, (j - 1) & 1)) { ok = false; break; }
        tc::fence_after();
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t r[32];
          tc::ld32(tl + kColO + 32 * q4, r);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
          tc::st32(tl + kColO + 32 * q4, r);
        }
        tc::wait_st();
      }
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = (x[2 * c] == kNegInf) ? 0.f : fast_exp2(x[2 * c] - m_ref);
        const float p1 = (x[2 * c + 1] == kNegInf) ? 0.f : fast_exp2(x[2 * c + 1] - m_ref);
        l += p0 + p1;
        split_bf16(p0, p1, hi[c], lo[c]);
      }
      tc::st32(tl + kColS + 64 * bb, hi);
      tc::st32(tl + kColS + 64 * bb + 32, lo);
      if (key0 + BN > cta_end) {
        // last tile: zero the V rows past the CTA's last visible key
        const int s = j % STAGES;
        if (!wait_all(&v_full[s], (j / STAGES) & 1)) { ok = false; break; }
        unsigned char* vt = sm + kOffV + s * kKVTile;
        const int z0 = cta_end - key0;
        for (int idx = threadIdx.x; idx < (BN - z0) * 16; idx += 128) {
          const int r = z0 + (idx >> 4);
          const int c = idx & 15;  // 16-byte chunk over the 128 dims (two boxes)
          *reinterpret_cast<uint4*>(vt + (c >> 3) * kKVBox + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[bb]);
    }
    // ---- epilogue: o = u / l, lse = m + ln l ----
    // `drain` completes once every MMA of the CTA has (single phase)
    if (ok && !wait_all(drain, 0)) ok = false;
    if (!ok) {
      if (lane == 0) {
        record_error(p.err, kErrTimeout);
        misc[3] = 1;
      }
    } else {
      tc::fence_after();
      const float inv = (m_ref == kNegInf) ? 0.f : 1.f / l;
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
      if (my_row) p.lse[lse_idx] = (m_ref == kNegInf) ? kNegInf : (m_ref + __log2f(l)) * kLn2;
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 5) tc::dealloc(tb, kTmemCols);
}

}  // namespace

int prefill_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill_tc(const FwdParams& p, int n_qtiles, const CUtensorMap& tmq, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(n_qtiles, p.Hq, p.B);
  prefill_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p, tmq, tmk, tmv);
  return cudaGetLastError();
}

}  // namespace blkattn
