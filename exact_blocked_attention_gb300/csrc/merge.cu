// Merge kernels: eqs. 33.4–33.5 of "Chapter 33: inference compute
// optimisation" §33.2, in fp32, with the valid-flag rule for empty states.
//
//  * split_merge_kernel: one CTA per query row folds the per-split partial
//    states of the split-KV kernels (fixed order per warp, fixed warp order:
//    deterministic, no atomics), then finishes with o = u / l and
//    lse = m + ln l.  Rows whose visible keys lie in a single split were
//    finished by the split kernel and are skipped here; the row's split count
//    is recomputed on the device from the same integers (cache length,
//    logical position, chunk), so no value crosses to the host.
//  * state_merge_kernel: the public two-state merge (blkattn_merge).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace blkattn {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kWarpsPerBlock = 8;

constexpr int kMergeWarps = 4;

// One CTA per query row; its warps share the row's splits.  Pass 1 takes the
// maximum m over the non-empty splits, pass 2 sums e^{m_s - m} l_s and
// e^{m_s - m} u_s (independent terms, so the loads of many splits are in
// flight at once), then the warps' partial sums are added.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) split_merge_kernel(const FwdParams p) {
  constexpr int DPL = D / 32;
  // launched as a programmatic dependent of the split kernel: wait for its
  // writes (a no-op when launched normally)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  const int i = (int)(row % p.Tq);
  const int h = (int)((row / p.Tq) % p.Hq);
  const int b = (int)(row / ((int64_t)p.Tq * p.Hq));
  int len = p.seqlens[b * p.sl_s];
  len = len < 0 ? 0 : (len > p.Tmax ? p.Tmax : len);
  const int pos = p.qpos[b * p.qp_sb + i * p.qp_si];
  const int end = pos < 0 ? 0 : (pos >= len ? len : pos + 1);
  const int n_active = (end + p.chunk - 1) / p.chunk;
  if (n_active <= 1) return;  // finished by the split kernel
  __shared__ float red_m[kMergeWarps];
  __shared__ float red_l[kMergeWarps];
  __shared__ float red_u[kMergeWarps][D];
  const float* wm = p.ws_m + row * p.n_splits;
  const float* wl = p.ws_l + row * p.n_splits;
  const float* wu = p.ws_u + row * p.n_splits * D;

  float M = kNegInf;
  for (int s = threadIdx.x; s < n_active; s += kMergeWarps * 32) M = fmaxf(M, wm[s]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red_m[warp] = M;
  __syncthreads();
  M = red_m[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) M = fmaxf(M, red_m[w]);

  float Ls = 0.f;
  float U[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) U[e] = 0.f;
  if (M != kNegInf) {
#pragma unroll 4
    for (int s = warp; s < n_active; s += kMergeWarps) {
      const float ms = wm[s];
      if (ms == kNegInf) continue;  // an empty state contributes nothing
      const float c = fast_exp2(ms - M);
      Ls = fmaf(c, wl[s], Ls);
      const float* us = wu + (int64_t)s * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 u4 = *reinterpret_cast<const float4*>(us);
        U[0] = fmaf(c, u4.x, U[0]); U[1] = fmaf(c, u4.y, U[1]);
        U[2] = fmaf(c, u4.z, U[2]); U[3] = fmaf(c, u4.w, U[3]);
      } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) U[e] = fmaf(c, us[e], U[e]);
      }
    }
  }
  if (lane == 0) red_l[warp] = Ls;
#pragma unroll
  for (int e = 0; e < DPL; ++e) red_u[warp][lane * DPL + e] = U[e];
  __syncthreads();

  const int64_t ob = (int64_t)b * p.o_sb + (int64_t)h * p.o_sh + (int64_t)i * p.o_si;
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) L += red_l[w];
  for (int d = threadIdx.x; d < D; d += kMergeWarps * 32) {
    float u = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) u += red_u[w][d];
    const float o = (M == kNegInf) ? 0.f : u / L;
    const int64_t oi = ob + (int64_t)d * p.o_sd;
    if (p.out_bf16)
      static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
    else
      static_cast<float*>(p.out)[oi] = o;
  }
  if (threadIdx.x == 0)
    p.lse[(int64_t)b * p.l_sb + (int64_t)h * p.l_sh + (int64_t)i * p.l_si] =
        (M == kNegInf) ? kNegInf : (M + __log2f(L)) * kLn2;
}

// Public merge of two states per row (natural-log m).  One warp per row.
__global__ void __launch_bounds__(kWarpsPerBlock * 32) state_merge_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
  if (row >= p.rows) return;
  const float ma = p.am[row];
  const float mb = p.bm[row];
  const bool va = ma != kNegInf;  // valid flags
  const bool vb = mb != kNegInf;
  const float la = va ? (p.al ? p.al[row] : 1.f) : 0.f;
  const float lb = vb ? (p.bl ? p.bl[row] : 1.f) : 0.f;
  float m = kNegInf, ca = 0.f, cb = 0.f;
  if (va && vb) {
    m = fmaxf(ma, mb);
    ca = fast_exp2((ma - m) * kLog2e);
    cb = fast_exp2((mb - m) * kLog2e);
  } else if (va) {
    m = ma;
    ca = 1.f;
  } else if (vb) {
    m = mb;
    cb = 1.f;
  }
  const float l = ca * la + cb * lb;
  const bool normalise = p.ol == nullptr;
  // every lane reads its columns before any lane writes (out may alias a or b)
  for (int d0 = 0; d0 < p.d; d0 += 32) {
    const int d = d0 + lane;
    if (d < p.d) {
      float uo = 0.f;
      if (va) uo = ca * p.au[row * p.a_us + d];
      if (vb) uo = fmaf(cb, p.bu[row * p.b_us + d], uo);
      if (normalise) uo = (m == kNegInf) ? 0.f : uo / l;
      p.ou[row * p.o_us + d] = uo;
    }
  }
  __syncwarp();
  if (lane == 0) {
    if (normalise) {
      p.om[row] = (m == kNegInf) ? kNegInf : m + __logf(l);
    } else {
      p.om[row] = m;
      p.ol[row] = l;
    }
  }
}

}  // namespace

cudaError_t launch_split_merge(const FwdParams& p, int d, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Tq;
  if (rows == 0) return cudaSuccess;
  if (rows > 0x7fffffff) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // programmatic dependent launch: the merge grid may be scheduled while the
  // split kernel drains; griddepcontrol.wait orders its reads after it
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (d == 128) return cudaLaunchKernelEx(&cfg, split_merge_kernel<128>, p);
  if (d == 64) return cudaLaunchKernelEx(&cfg, split_merge_kernel<64>, p);
  return cudaErrorInvalidValue;
}

cudaError_t launch_state_merge(const MergeParams& p, cudaStream_t stream) {
  const int64_t blocks = (p.rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  state_merge_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace blkattn
