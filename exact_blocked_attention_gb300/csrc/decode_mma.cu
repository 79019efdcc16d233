// Split-KV decode / verify kernel on warp-level tensor cores (bf16 inputs).
//
// Same algorithm and work split as the CUDA-core kernel (decode_split.cu):
// one CTA = the packed query rows of one KV head x one key split, K/V tiles
// streamed into a shared-memory ring by tiled TMA (64 keys x 64 dims per box,
// 128-byte swizzle, no multicast) from a producer warp, Algorithm 33.1 of "Chapter 33: inference compute
// optimisation" §33.2 run per 16-key sub-block by each consumer warp with the
// (m, l, u) statistics of eq. 33.3 and the merge rule of eqs. 33.4–33.5.
//
// The two contractions run on mma.sync m16n8k16 (bf16 x bf16 -> fp32):
//   S = Q K^T   A = 16 query rows (packed G x T_q rows, zero-padded), B = K
//   U += P V    A = P from the score fragments, B = V (ldmatrix.trans)
// Q and K are bf16 inputs, so every product is exact and sums are fp32, as on
// CUDA cores.  P is not an input: to keep it exact to ~16 significant bits it
// is split as P = P_hi + P_lo, both bf16, and U += P_hi V + P_lo V.  The mask
// is applied by select on the fp32 scores; V rows of the last tile past the
// split's last visible key (cache padding, possibly NaN) are zero-filled in
// shared memory so that 0 * garbage never reaches the accumulator.
//
// Warp layout: MT m-tiles of 16 rows x NWK key slices of 16 keys per stage;
// consumer warp w owns m-tile (w % MT) and key slice (w / MT).  The NWK
// states of one m-tile are merged with eqs. 33.4–33.5 at the end of the split.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace blkattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

template <int D, int MT, int NWK, int STAGES>
struct MmaLayout {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kBoxes = D / 64;            // 64-dim (128-byte) swizzled boxes per row
  static constexpr int kKpw = 16;                  // keys per warp per stage
  static constexpr int kTile = kKpw * NWK;         // keys per stage (= TMA box rows)
  static constexpr int kBoxBytes = kTile * 128;
  static constexpr int kTensorBytes = kBoxes * kBoxBytes;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTensorBytes;
  static constexpr int kRing = STAGES * kStageBytes;       // 1024-aligned start
  static constexpr int kRows = 16 * MT;
  static constexpr int kNW = MT * NWK;
  static constexpr int kRedPitch = D + 4;  // floats per reduced row (bank skew)
  // cross-slice reduction area, reusing the ring once every copy has landed
  static constexpr int kRedBytes = NWK * kRows * (kRedPitch + 2) * 4;
  static constexpr int kRingAlloc = kRing > kRedBytes ? kRing : kRedBytes;
  static constexpr int kQPad = kRowBytes + 16;     // padded Q rows (ldmatrix, no conflicts)
  static constexpr int kQOff = kRingAlloc;
  static constexpr int kRowInfoOff = kQOff + kRows * kQPad;  // int[3][kRows]
  static constexpr int kBarOff = (kRowInfoOff + 3 * kRows * 4 + 15) / 16 * 16;
  static constexpr int kMiscOff = kBarOff + 2 * STAGES * 8;
  static constexpr int kBytes = kMiscOff + 16 + 1024;  // + slack to align the ring to 1024
  static_assert(kTile == 64, "TMA box is 64 rows");
};

// Byte offset of 16-byte chunk `c` (0 .. D/8-1) of row `r` in a swizzled tile:
// boxes of 64 dims, rows of 128 bytes, chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((c >> 3) * (64 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Register cap so that two CTAs (2 x 5 warps) share an SM at MT = 1: the
// register file is split per sub-partition, 3 warps x 168 x 32 fit one.
template <int MT, int NWK>
constexpr int mma_max_regs() {
  return (MT * NWK + 1) <= 5 ? 168 : ((MT * NWK + 1) <= 9 ? 168 : 128);
}

template <int D, int MT, int NWK, int STAGES>
__global__ void __maxnreg__((mma_max_regs<MT, NWK>()))
    decode_mma_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  using L = MmaLayout<D, MT, NWK, STAGES>;
  constexpr int NW = L::kNW;
  constexpr int kRowBytes = L::kRowBytes;
  constexpr int kQPad = L::kQPad;
  constexpr int kTile = L::kTile;
  constexpr int kRows = L::kRows;
  constexpr int KS = D / 16;  // k16 steps over the head dim
  constexpr int NT = D / 8;   // n8 tiles over the value dim

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle repeats every 1024 bytes: align the ring to it
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char* ring = smem;
  unsigned char* q_s = smem + L::kQOff;
  int* row_end_s = reinterpret_cast<int*>(smem + L::kRowInfoOff);
  int* row_h_s = row_end_s + kRows;
  int* row_i_s = row_h_s + kRows;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  int* misc = reinterpret_cast<int*>(smem + L::kMiscOff);  // [0] issued, [1] timeout, [2] cta_end

  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int b = blockIdx.z / p.row_groups;
  const int rg = blockIdx.z % p.row_groups;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- per-row visibility bookkeeping (integers) ----
  int len = p.seqlens[b * p.sl_s];
  len = len < 0 ? 0 : (len > p.Tmax ? p.Tmax : len);
  if (threadIdx.x == 0) misc[2] = 0;
  __syncthreads();
  if (threadIdx.x < kRows) {
    const int r = threadIdx.x;
    const int pk = rg * kRows + r;
    int e = 0, h = 0, i = 0;
    if (pk < p.rows_per_head) {
      const int g = pk / p.Tq;
      i = pk - g * p.Tq;
      h = hk * p.G + g;
      const int pos = p.qpos[b * p.qp_sb + i * p.qp_si];
      e = pos < 0 ? 0 : (pos >= len ? len : pos + 1);
    }
    row_end_s[r] = e;
    row_h_s[r] = h;
    row_i_s[r] = i;
    atomicMax(&misc[2], e);
  }
  __syncthreads();
  const int cta_end = misc[2];
  const int k0 = split * p.chunk;
  if (split > 0 && k0 >= cta_end) return;  // uniform: split 0 always runs
  const int k1 = min(k0 + p.chunk, cta_end);
  const int n_tiles = k1 > k0 ? (k1 - k0 + kTile - 1) / kTile : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    misc[0] = 0;
    misc[1] = 0;
    fence_barrier_init();
  }
  // query rows -> shared memory (bf16, padded pitch), zero for absent rows
  for (int idx = threadIdx.x; idx < kRows * (D / 2); idx += blockDim.x) {
    const int r = idx / (D / 2);
    const int d2 = idx - r * (D / 2);
    uint32_t w = 0;
    const int pk = rg * kRows + r;
    if (pk < p.rows_per_head) {
      const int g = pk / p.Tq;
      const int i = pk - g * p.Tq;
      const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) + (int64_t)b * p.q_sb +
                                  (int64_t)(hk * p.G + g) * p.q_sh + (int64_t)i * p.q_si;
      const unsigned short lo = __bfloat16_as_ushort(qrow[(int64_t)(2 * d2) * p.q_sd]);
      const unsigned short hi = __bfloat16_as_ushort(qrow[(int64_t)(2 * d2 + 1) * p.q_sd]);
      w = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint32_t*>(q_s + r * kQPad + d2 * 4) = w;
  }
  __syncthreads();

  const int mt = warp % MT;
  const int ks = warp / MT;
  const int g = lane >> 2;
  const int t = lane & 3;
  float o[NT][4];
  float m_run[2] = {kNegInf, kNegInf};
  float l_part[2] = {0.f, 0.f};

  if (warp == NW) {
    // ---------------- producer warp ----------------
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    int tt = 0;
    for (; tt < n_tiles; ++tt) {
      const int st = tt % STAGES;
      if (tt >= STAGES) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[st], ((tt / STAGES) - 1) & 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) { record_error(p.err, kErrTimeout); misc[1] = 1; }
          break;
        }
      }
      const int key0 = k0 + tt * kTile;
      unsigned char* kdst = ring + st * L::kStageBytes;
      unsigned char* vdst = kdst + L::kTensorBytes;
      if (lane == 0) {
        // full boxes always: rows past T_max are zero-filled and still counted
        mbar_arrive_expect_tx(&full[st], (uint32_t)L::kStageBytes);
#pragma unroll
        for (int bx = 0; bx < L::kBoxes; ++bx) {
          tma_load_4d(kdst + bx * L::kBoxBytes, &tmk, bx * 64, key0, hk, b, &full[st], pol);
          tma_load_4d(vdst + bx * L::kBoxBytes, &tmv, bx * 64, key0, hk, b, &full[st], pol);
        }
      }
      __syncwarp();
    }
    if (lane == 0) misc[0] = tt;
  } else {
    // ---------------- consumer warps ----------------
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    // Q fragments of this warp's m-tile, kept in registers
    uint32_t qa[KS][4];
    {
      const int m = lane >> 3, rr = lane & 7;
      const uint32_t base = smem_u32(q_s) + (16 * mt + rr + ((m & 1) ? 8 : 0)) * kQPad;
#pragma unroll
      for (int k = 0; k < KS; ++k)
        ldsm_x4(base + (2 * k + (m >> 1)) * 16, qa[k][0], qa[k][1], qa[k][2], qa[k][3]);
    }
    const int r0 = 16 * mt + g;
    const int r1 = r0 + 8;
    const int hi0 = min(row_end_s[r0], k0 + p.chunk);
    const int hi1 = min(row_end_s[r1], k0 + p.chunk);
    // token tree: keys from tbase on are seen only where the row's mask says
    const int tbase = p.tree != nullptr ? len - p.Tq : 0x7fffffff;
    const uint64_t tr0 = p.tree != nullptr ? (uint64_t)p.tree[(int64_t)b * p.tr_sb + (int64_t)row_i_s[r0] * p.tr_si] : ~0ull;
    const uint64_t tr1 = p.tree != nullptr ? (uint64_t)p.tree[(int64_t)b * p.tr_sb + (int64_t)row_i_s[r1] * p.tr_si] : ~0ull;
    // sliding window: each row's first visible key (pos >= 0 first, so the
    // difference cannot overflow)
    int ws0 = 0, ws1 = 0;
    if (p.window > 0) {
      const int q0 = p.qpos[b * p.qp_sb + row_i_s[r0] * p.qp_si];
      const int q1 = p.qpos[b * p.qp_sb + row_i_s[r1] * p.qp_si];
      ws0 = q0 < 0 ? 0 : max(0, q0 - p.window + 1);
      ws1 = q1 < 0 ? 0 : max(0, q1 - p.window + 1);
    }
    const float* bias0 = nullptr;
    const float* bias1 = nullptr;
    if (p.bias != nullptr) {
      bias0 = p.bias + (int64_t)b * p.bi_sb + (int64_t)row_h_s[r0] * p.bi_sh + (int64_t)row_i_s[r0] * p.bi_si;
      bias1 = p.bias + (int64_t)b * p.bi_sb + (int64_t)row_h_s[r1] * p.bi_sh + (int64_t)row_i_s[r1] * p.bi_si;
    }
    // ldmatrix lane addressing (rows of a 16-key slice; row mod 8 == lr)
    const int lm = lane >> 3, lr = lane & 7;
    const int k_row = ks * 16 + lr + ((lm >= 2) ? 8 : 0);  // K: (keys 0-7 | 8-15) x (lo | hi 8 dims)
    const int k_chk = lm & 1;
    const int v_row = ks * 16 + lr + ((lm & 1) ? 8 : 0);   // V^T: (keys 0-7 | 8-15) x (dv lo | hi 8)
    const int v_chk = lm >> 1;

    for (int tt = 0; tt < n_tiles; ++tt) {
      const int st = tt % STAGES;
      if (!mbar_wait(&full[st], (tt / STAGES) & 1)) {
        if (lane == 0) { record_error(p.err, kErrTimeout); misc[1] = 1; }
        break;
      }
      const int tile_k0 = k0 + tt * kTile;
      unsigned char* kst = ring + st * L::kStageBytes;
      unsigned char* vst = kst + L::kTensorBytes;
      const int key_base = tile_k0 + ks * 16;
      // zero the V rows of this slice past the split's last visible key
      // (last tile only: cache padding or zero fill past T_max)
      const int n_valid = k1 - key_base;
      if (n_valid < 16) {
        const int z0 = n_valid < 0 ? 0 : n_valid;
        for (int idx = lane; idx < (16 - z0) * (kRowBytes / 16); idx += 32) {
          const int rr = ks * 16 + z0 + idx / (kRowBytes / 16);
          const int cc = idx % (kRowBytes / 16);
          *reinterpret_cast<uint4*>(vst + swz(rr, cc)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }

      // ---- S = Q K^T over this warp's 16 keys ----
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t kaddr = smem_u32(kst);
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kaddr + swz(k_row, 2 * k + k_chk), b0, b1, b2, b3);
        mma_bf16(s[0], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b0, b1);
        mma_bf16(s[1], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b2, b3);
      }
      // ---- scores in base-2 units, visibility by select ----
      float x[2][4];  // [row 0/1][n-tile*2 + col]
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key_base + nt * 8 + 2 * t + e;
          bool v0 = key < hi0 && key >= ws0, v1 = key < hi1 && key >= ws1;
          if (key >= tbase) {
            const int node = key - tbase;
            v0 = v0 && node < 64 && ((tr0 >> (node & 63)) & 1ull);
            v1 = v1 && node < 64 && ((tr1 >> (node & 63)) & 1ull);
          }
          float bb0 = 0.f, bb1 = 0.f;
          if (bias0 != nullptr) {
            if (v0) { bb0 = bias0[(int64_t)key * p.bi_sj]; v0 = bb0 != kNegInf; }
            if (v1) { bb1 = bias1[(int64_t)key * p.bi_sj]; v1 = bb1 != kNegInf; }
          }
          x[0][nt * 2 + e] = v0 ? fmaf(s[nt][e], p.scale_log2, bb0 * kLog2e) : kNegInf;
          x[1][nt * 2 + e] = v1 ? fmaf(s[nt][2 + e], p.scale_log2, bb1 * kLog2e) : kNegInf;
        }
      // ---- block statistics + online merge (valid flags) ----
      float alpha[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float mx = fmaxf(fmaxf(x[rr][0], x[rr][1]), fmaxf(x[rr][2], x[rr][3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        alpha[rr] = 1.f;
        if (mx != kNegInf) {
          const float m_new = fmaxf(m_run[rr], mx);
          alpha[rr] = (m_run[rr] == kNegInf) ? 0.f : fast_exp2(m_run[rr] - m_new);
          float ls = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float pj = (x[rr][j] == kNegInf) ? 0.f : fast_exp2(x[rr][j] - m_new);
            x[rr][j] = pj;
            ls += pj;
          }
          l_part[rr] = fmaf(l_part[rr], alpha[rr], ls);
          m_run[rr] = m_new;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) x[rr][j] = 0.f;
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[nt][0] *= alpha[0];
        o[nt][1] *= alpha[0];
        o[nt][2] *= alpha[1];
        o[nt][3] *= alpha[1];
      }
      // ---- P fragments (A operand), split hi + lo ----
      uint32_t ph[4], pl[4];
      split_bf16(x[0][0], x[0][1], ph[0], pl[0]);  // row g,   keys 2t..2t+1
      split_bf16(x[1][0], x[1][1], ph[1], pl[1]);  // row g+8
      split_bf16(x[0][2], x[0][3], ph[2], pl[2]);  // row g,   keys 8+2t..
      split_bf16(x[1][2], x[1][3], ph[3], pl[3]);  // row g+8
      // ---- U += P V ----
      const uint32_t vaddr = smem_u32(vst);
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vaddr + swz(v_row, 2 * np + v_chk), v0, v1, v2, v3);
        mma_bf16(o[2 * np], ph[0], ph[1], ph[2], ph[3], v0, v1);
        mma_bf16(o[2 * np], pl[0], pl[1], pl[2], pl[3], v0, v1);
        mma_bf16(o[2 * np + 1], ph[0], ph[1], ph[2], ph[3], v2, v3);
        mma_bf16(o[2 * np + 1], pl[0], pl[1], pl[2], pl[3], v2, v3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // l: sum over the 4 lanes of a quad (they hold different keys of the row)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 1);
      l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 2);
    }
  }

  // the split-merge grid may start launching now (it waits for this grid's
  // completion before reading anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- drain every issued copy before the ring is reused ----
  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = misc[0];
    for (int tt = issued - STAGES < 0 ? 0 : issued - STAGES; tt < issued; ++tt)
      if (!mbar_wait(&full[tt % STAGES], (tt / STAGES) & 1)) {
        record_error(p.err, kErrTimeout);
        misc[1] = 1;
      }
  }
  __syncthreads();
  if (misc[1]) return;

  // ---- merge the key slices of each m-tile (eqs. 33.4-33.5) ----
  float* red_m = reinterpret_cast<float*>(ring);  // [NWK][kRows]
  float* red_l = red_m + NWK * kRows;              // [NWK][kRows]
  float* red_o = red_l + NWK * kRows;              // [NWK][kRows][kRedPitch]
  constexpr int P_ = L::kRedPitch;
  if (warp < NW) {
    const int r0 = 16 * mt + g;
    if (t == 0) {
      red_m[ks * kRows + r0] = m_run[0];
      red_m[ks * kRows + r0 + 8] = m_run[1];
      red_l[ks * kRows + r0] = l_part[0];
      red_l[ks * kRows + r0 + 8] = l_part[1];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      *reinterpret_cast<float2*>(&red_o[(ks * kRows + r0) * P_ + nt * 8 + 2 * t]) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(&red_o[(ks * kRows + r0 + 8) * P_ + nt * 8 + 2 * t]) = make_float2(o[nt][2], o[nt][3]);
    }
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < kRows * D; idx += blockDim.x) {
    const int r = idx / D;
    const int d = idx - r * D;
    const int pk = rg * kRows + r;
    if (pk >= p.rows_per_head) continue;
    const int rend = row_end_s[r];
    if (k0 >= rend && split != 0) continue;  // nothing of this row here; split 0 writes it
    const int rh = row_h_s[r];
    const int ri = row_i_s[r];
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NWK; ++w) M = fmaxf(M, red_m[w * kRows + r]);
    float Ls = 0.f, Us = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NWK; ++w) {
        const float mw = red_m[w * kRows + r];
        if (mw == kNegInf) continue;  // empty slice state
        const float c = fast_exp2(mw - M);
        Ls = fmaf(c, red_l[w * kRows + r], Ls);
        Us = fmaf(c, red_o[(w * kRows + r) * P_ + d], Us);
      }
    }
    const int n_active = (rend + p.chunk - 1) / p.chunk;
    if (n_active <= 1) {
      const float ov = (M == kNegInf) ? 0.f : Us / Ls;
      const int64_t oi = (int64_t)b * p.o_sb + (int64_t)rh * p.o_sh + (int64_t)ri * p.o_si + (int64_t)d * p.o_sd;
      if (p.out_bf16)
        static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(ov);
      else
        static_cast<float*>(p.out)[oi] = ov;
      if (d == 0)
        p.lse[(int64_t)b * p.l_sb + (int64_t)rh * p.l_sh + (int64_t)ri * p.l_si] =
            (M == kNegInf) ? kNegInf : (M + __log2f(Ls)) * kLn2;
    } else {
      const int64_t row = ((int64_t)b * p.Hq + rh) * p.Tq + ri;
      const int64_t wi = row * p.n_splits + split;
      p.ws_u[wi * D + d] = Us;
      if (d == 0) {
        p.ws_m[wi] = M;
        p.ws_l[wi] = Ls;
      }
    }
  }
}

template <int D, int MT>
cudaError_t launch_mt(const FwdParams& p, const DecodeConfig& cfg, const CUtensorMap& tmk,
                      const CUtensorMap& tmv, cudaStream_t stream) {
  constexpr int NWK = 4, STAGES = 3;
  using L = MmaLayout<D, MT, NWK, STAGES>;
  auto kern = decode_mma_kernel<D, MT, NWK, STAGES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared storage as shared memory: two ~100 KB CTAs per SM
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(cfg.n_splits, p.Hkv, p.B * cfg.row_groups);
  kern<<<grid, (L::kNW + 1) * 32, L::kBytes, stream>>>(p, tmk, tmv);
  return cudaGetLastError();
}

}  // namespace

size_t decode_mma_smem_bytes(int d, int mt) {
  if (d == 128) {
    if (mt == 1) return MmaLayout<128, 1, 4, 3>::kBytes;
    if (mt == 2) return MmaLayout<128, 2, 4, 3>::kBytes;
    return MmaLayout<128, 3, 4, 3>::kBytes;
  }
  if (mt == 1) return MmaLayout<64, 1, 4, 3>::kBytes;
  if (mt == 2) return MmaLayout<64, 2, 4, 3>::kBytes;
  return MmaLayout<64, 3, 4, 3>::kBytes;
}

cudaError_t launch_decode_mma(const FwdParams& p, int d, const DecodeConfig& cfg,
                              const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
  const int mt = cfg.rows_per_cta / 16;
  if (cfg.rows_per_cta % 16 != 0 || mt < 1 || mt > 3) return cudaErrorInvalidValue;
  if (d == 128) {
    if (mt == 1) return launch_mt<128, 1>(p, cfg, tmk, tmv, stream);
    if (mt == 2) return launch_mt<128, 2>(p, cfg, tmk, tmv, stream);
    return launch_mt<128, 3>(p, cfg, tmk, tmv, stream);
  }
  if (d == 64) {
    if (mt == 1) return launch_mt<64, 1>(p, cfg, tmk, tmv, stream);
    if (mt == 2) return launch_mt<64, 2>(p, cfg, tmk, tmv, stream);
    return launch_mt<64, 3>(p, cfg, tmk, tmv, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace blkattn
