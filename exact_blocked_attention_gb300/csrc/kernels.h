// Parameter blocks and launcher declarations shared by the host API and the
// kernel translation units.  Internal to libblkattn (not part of the C ABI).
#pragma once
#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "blkattn.h"

namespace blkattn {

enum class Elt : int { BF16 = 1, F32 = 2 };

// One blkattn_fwd call, after validation.  K/V strides are in BYTES, all the
// others in elements.
struct FwdParams {
  // query rows
  const void* q;
  int64_t q_sb, q_sh, q_si, q_sd;
  // cache (device pointers, 16-byte aligned rows)
  const char* k;
  const char* v;
  int64_t k_sb, k_sh, k_st;
  int64_t v_sb, v_sh, v_st;
  // lengths and logical positions (device int32)
  const int32_t* seqlens;
  int64_t sl_s;
  const int32_t* qpos;
  int64_t qp_sb, qp_si;
  // optional additive bias (device f32), 0-strides broadcast
  const float* bias;
  int64_t bi_sb, bi_sh, bi_si, bi_sj;
  // optional token tree (device int64 [B, T_q], T_q <= 64): bit k of
  // tree[b, i] lets row i see key len_b - T_q + k; keys before len_b - T_q
  // are not affected
  const int64_t* tree;
  int64_t tr_sb, tr_si;
  // optional sliding window: > 0 keeps only keys j > pos - window
  int window;
  float scale_log2;  // scale * log2(e): scores are kept in base-2 units
  // results
  void* out;
  int out_bf16;
  int64_t o_sb, o_sh, o_si, o_sd;
  float* lse;
  int64_t l_sb, l_sh, l_si;
  // sizes
  int B, Hq, Hkv, G, Tq, Tmax;
  int rows_per_head;  // G * Tq query rows read one KV head
  int row_groups;     // CTAs along those rows
  int chunk;          // keys per split
  int n_splits;
  // per-split partial states (only when n_splits > 1): index row*n_splits+s,
  // row = (b*Hq + h)*Tq + i; m and l in base-2 units, u [.., d]
  float* ws_m;
  float* ws_l;
  float* ws_u;
  int* err;  // device error word
  int head_group;  // prefill: (sequence, head) pairs dispatched together (L2 reuse of K/V)
  // tcgen05 decode kernel: query rows per unit (one row group of one KV head);
  // the partial state of unit row r from CTA c sits in slot c + unit, at
  // index slot * rows_cta + r; unit_cnt counts the CTAs of each unit that
  // wrote theirs (zero before the launch, left zero after it)
  int rows_cta;
  unsigned* unit_cnt;
  // prefill: 1 when the output tensor map (fp32, boxes {32, 32}, 128-byte
  // swizzle) is valid and the kernel stores whole output tiles with TMA
  int o_tma;
  // test hook of the tcgen05 decode kernel (-1: none): the MMA-issuing thread
  // of this CTA waits on a barrier nothing completes, gives up after 1 ms
  // and issues no product, so the CTA's other roles run out their bounded
  // waits (blkattn_debug_stall_next_decode)
  int test_stall_cta;
};

// Split-KV kernel configuration chosen by the planner.
enum class Kernel : int { CudaCore = 0, TensorCore = 1, Prefill = 2, DecodeTc = 3 };
struct DecodeConfig {
  Kernel kernel;
  int rows_per_cta;  // CUDA-core: 1, 2, 4 or 8; tensor-core: 16, 32 or 48
  int warps;         // consumer warps; keys per stage = 16 * warps
  int stages;
  int chunk;
  int n_splits;
  int row_groups;
};

cudaError_t launch_decode_split(const FwdParams& p, Elt elt, int d, const DecodeConfig& cfg,
                                cudaStream_t stream);
cudaError_t launch_split_merge(const FwdParams& p, int d, cudaStream_t stream);

struct MergeParams {
  const float* am; const float* al; const float* au; int64_t a_us;
  const float* bm; const float* bl; const float* bu; int64_t b_us;
  float* om; float* ol; float* ou; int64_t o_us;
  int64_t rows;
  int d;
};
cudaError_t launch_state_merge(const MergeParams& p, cudaStream_t stream);

size_t decode_smem_bytes(Elt elt, int d, const DecodeConfig& cfg);

// Tensor-core (mma.sync, bf16) split-KV kernel: 16 * mt query rows per CTA.
// K and V tiles arrive by tiled TMA through these maps: 4-D {d, T_max, H_kv,
// B}, box {64, 64, 1, 1}, bf16, 128-byte swizzle.
cudaError_t launch_decode_mma(const FwdParams& p, int d, const DecodeConfig& cfg,
                              const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, cudaStream_t stream);
size_t decode_mma_smem_bytes(int d, int mt);

// Causal prefill on tcgen05 (bf16, d = 128, no bias): one CTA per 256 query
// rows of one head (two 128-row query tiles); maps: Q and K/V boxes {64, 128},
// all 128-byte swizzle; tmo (read only when p.o_tma) the fp32 output with
// boxes {32, 32}, 128-byte swizzle.
cudaError_t launch_prefill_tc(const FwdParams& p, int n_pairs, const CUtensorMap& tmq, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, const CUtensorMap& tmo, cudaStream_t stream);
int prefill_tc_smem_bytes();

// Decode / verify on tcgen05 (bf16, d = 128, 16-byte aligned query rows, at
// most 48 query rows per unit): `ctas` persistent CTAs share the key tiles of
// all units equally; maps as for the prefill kernel (K/V boxes {64, 128}).
// The (sequence, row group) table lives in shared memory: B * row_groups
// must not exceed kDecodeTcMaxEntries.
constexpr int kDecodeTcMaxEntries = 1024;
// blkattn_fwd_static_scratch keeps the tcgen05 decode kernel's per-unit
// counters in the last kStaticCounterBytes of its array (one 32-bit counter
// per unit), outside every plan's workspace.
constexpr size_t kStaticCounterBytes = 256 * 1024;
void clear_static_counters();
cudaError_t launch_decode_tc(const FwdParams& p, int ctas, const CUtensorMap& tmk, const CUtensorMap& tmv,
                             cudaStream_t stream);
size_t decode_tc_smem_bytes(int rows_cta);

// ---- backward pass (eqs. 33.6-33.8), tcgen05, bf16, d = 128 ----
struct BwdParams {
  const void* out;  // forward output o [B, H_q, T_q, d] (bf16 or fp32), read for D = g_o . o
  int out_bf16;
  int out_vec;  // fp32 rows with unit dim stride, 16-byte aligned (vector loads)
  int64_t o_sb, o_sh, o_si, o_sd;
  const float* lse;  // forward lse [B, H_q, T_q] (natural log, -inf = empty row)
  int64_t l_sb, l_sh, l_si;
  const void* dout;  // upstream gradient g_o, bf16 [B, H_q, T_q, d] (unit dim stride)
  int64_t g_sb, g_sh, g_si;
  const int* seqlens;
  int64_t sl_s;
  const int* qpos;
  int64_t qp_sb, qp_si;
  const float* bias;  // nullptr or [B, H_q, T_q, T_max] view
  int64_t bi_sb, bi_sh, bi_si, bi_sj;
  float* dq;  // fp32 [B, H_q, T_q, d], unit dim stride, 16-byte aligned rows
  int64_t dq_sb, dq_sh, dq_si;
  float* dk;  // fp32 [B, H_kv, T_max, d], likewise
  int64_t dk_sb, dk_sh, dk_sj;
  float* dv;
  int64_t dv_sb, dv_sh, dv_sj;
  float* ws_D;    // [B * H_q * T_q] row sums g_o . o
  float* ws_L;    // [B * H_q * T_q] lse in base-2 units (+inf for an empty row)
  int* ws_end;    // [B * n_qt] largest row end min(pos + 1, len) of each 128-row query tile
  int* ws_start;  // [B * n_qt] smallest first visible key of the tile's rows that see a key (INT_MAX: none)
  int window;     // sliding window (0: none): a row sees keys pos - window < j <= pos
  int B, Hq, Hkv, G, Tq, Tmax, n_qt, n_kt;
  int hg_q;   // dQ: (sequence, head) pairs dispatched together (their K/V fit in L2)
  int hg_kv;  // dK/dV: (sequence, KV head) pairs dispatched together (their Q, g_o fit in L2)
  float scale, scale_log2;
  int* err;
};
// Row facts, then dQ (one CTA per 128-row query tile), then dK/dV (one CTA
// per 128-key tile); maps: Q, g_o, K, V, boxes {64, 128}, 128-byte swizzle.
cudaError_t launch_backward(const BwdParams& p, const CUtensorMap& tmq, const CUtensorMap& tmg,
                            const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream);
int backward_smem_bytes();

// Validation only (no CUDA call), and blkattn_fwd with caller-given scratch
// for the per-split states (no allocation; BLKATTN_ERR_SCRATCH_LIMIT when the
// plan needs more than scratch_bytes).  Both live in api.cu.
int validate_fwd_args(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                      const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                      const blkattn_tensor* mask_bias, const blkattn_tensor* out,
                      const blkattn_tensor* lse);
int fwd_with_scratch(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                     const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                     const blkattn_tensor* tree, const blkattn_tensor* mask_bias, float scale,
                     const blkattn_tensor* out, const blkattn_tensor* lse, blkattn_stream_t stream,
                     void* scratch, size_t scratch_bytes);
// Records a CUDA failure for blkattn_last_cuda_error; returns BLKATTN_ERR_CUDA.
int report_cuda_failure(cudaError_t e);
// The current device's error word (kernels record a bounded wait that ran
// out there; blkattn_check_device_error reads and clears it).
int device_error_word(int** out);
// blkattn_fwd / _tree / _window (tree may be NULL, window 0 = none) on the
// library's workspace.
int fwd_impl(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
             const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos, const blkattn_tensor* tree,
             int64_t window, const blkattn_tensor* mask_bias, float scale, const blkattn_tensor* out,
             const blkattn_tensor* lse, blkattn_stream_t stream);

}  // namespace blkattn
