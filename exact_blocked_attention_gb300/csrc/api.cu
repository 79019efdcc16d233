// Host side of libblkattn: the C ABI of include/blkattn.h.
//
// Every argument is validated before any CUDA call, so invalid requests fail
// the same way with or without a GPU.  The split plan is pure integer host
// arithmetic on sizes the host already knows (T_max, heads, rows, SM count);
// cache lengths and logical positions are only ever read on the device, so a
// call never synchronises with the GPU ("Chapter 33: inference compute
// optimisation" §33.4: host reads of device values cut a capturable region).
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "blkattn.h"
#include "kernels.h"

namespace {

using blkattn::DecodeConfig;
using blkattn::Elt;
using blkattn::FwdParams;

__device__ int g_error_word;  // set by kernels whose bounded waits ran out

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int* err = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  // per-unit counters of the tcgen05 decode kernel: zeroed when allocated,
  // left zero by every launch
  unsigned* cnt = nullptr;
  size_t cnt_n = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
cudaEvent_t g_split_event = nullptr;  // measurement hook (blkattn_debug_set_split_event)
int g_stall_next = -1;                // test hook (blkattn_debug_stall_next_decode)

// The CUDA error behind the last BLKATTN_ERR_CUDA (blkattn_last_cuda_error).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
int cuda_fail(cudaError_t e) {
  g_last_cuda_error = e;
  return BLKATTN_ERR_CUDA;
}

// ------------------------------------------------------------ validation
bool is_float_dtype(int32_t t) { return t == BLKATTN_BF16 || t == BLKATTN_F32; }
int elt_bytes(int32_t t) { return t == BLKATTN_BF16 ? 2 : 4; }

bool dims_ok(const blkattn_tensor* t, int ndim) {
  if (t == nullptr || t->ndim != ndim) return false;
  for (int i = 0; i < ndim; ++i)
    if (t->sizes[i] < 0 || t->strides[i] < 0) return false;
  return true;
}

// Every tensor given (NULL entries skipped) names the same device ordinal
// as `first`, and that ordinal is a device (not host memory).
bool same_device(const blkattn_tensor* first, std::initializer_list<const blkattn_tensor*> ts) {
  if (first->device < 0) return false;
  for (const blkattn_tensor* t : ts)
    if (t != nullptr && t->device != first->device) return false;
  return true;
}

// The call's device must be the current one (the library never switches it).
int check_current_device(int32_t device) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_fail(e);
  return dev == device ? BLKATTN_OK : BLKATTN_ERR_INVALID_ARG;
}


// Integer plan shared by blkattn_fwd and blkattn_debug_plan.
struct Plan {
  DecodeConfig cfg;
  int tile;
  int64_t ctas;
  int64_t ws_bytes;
  int64_t units = 0;  // tcgen05 decode kernel: per-unit counters needed
};

int resident_ctas_per_sm(size_t smem_bytes) {
  const size_t per_sm = 228 * 1024;
  const size_t per_cta = smem_bytes + 1024;  // 1 KB the runtime reserves per CTA
  int n = (int)(per_sm / per_cta);
  return n < 1 ? 1 : n;
}

// prefill_ok: the request qualifies for the tcgen05 prefill kernel (bf16,
// d = 128, no bias, 16-byte aligned query rows) if it also has T_q >= 64.
// q_vec_ok: the query rows are contiguous and 16-byte aligned (the tcgen05
// decode kernel loads them with 16-byte vector loads).
// windowed: a sliding-window call (the tcgen05 decode kernel then keeps its
// per-unit start tiles in half of its unit table).
Plan make_plan(int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tmax, int d, Elt elt,
               int sms, bool prefill_ok, bool q_vec_ok, bool windowed = false) {
  Plan pl;
  const int64_t rows = (Hq / Hkv) * Tq;  // query rows that read one KV head
  const char* force = std::getenv("BLKATTN_KERNEL");  // comparison runs only
  const bool force_mma = force && std::strcmp(force, "mma") == 0;
  const bool force_cudacore = force && std::strcmp(force, "cudacore") == 0;
  if (prefill_ok && elt == Elt::BF16 && d == 128 && Tq >= 64 && (Tq + 255) / 256 <= 65535) {
    // many query rows per head: two 128-row query tiles per CTA on tcgen05,
    // no splits
    pl.cfg.kernel = blkattn::Kernel::Prefill;
    pl.cfg.rows_per_cta = 256;
    pl.cfg.row_groups = (int)((Tq + 255) / 256);
    pl.cfg.warps = 4;
    pl.cfg.stages = 2;
    pl.tile = 128;
    pl.cfg.chunk = (int)((Tmax + 127) / 128 * 128);
    pl.cfg.n_splits = 1;
    pl.ctas = (int64_t)pl.cfg.row_groups * Hq * B;
    pl.ws_bytes = 0;
    return pl;
  }
  {
    // few rows per KV head: tcgen05 with the keys on the TMEM lanes, one
    // persistent CTA per SM sharing the key tiles of all units equally
    const int64_t rg = (rows + 47) / 48;
    const int64_t R = (rows + rg - 1) / rg;
    // (the kernel's schedule uses 32-bit arithmetic: fewer than 2^24 key
    // tiles in all, at most 255 CTAs)
    const int64_t max_tiles = B * Hkv * rg * ((Tmax + 127) / 128 + 2);  // + the per-unit weight
    if (q_vec_ok && elt == Elt::BF16 && d == 128 && !force_mma && !force_cudacore && rows >= 1 &&
        B * rg <= (windowed ? blkattn::kDecodeTcMaxEntries / 2 : blkattn::kDecodeTcMaxEntries) &&
        Tmax <= 65535LL * 128 && max_tiles < (1LL << 24) &&
        (sms > 0 ? sms : 148) <= 255) {
      const int64_t P = sms > 0 ? sms : 148;
      const int64_t U = B * Hkv * rg;
      const int64_t slots = P + U;  // partial-state slots: CTA index + unit index
      pl.cfg.kernel = blkattn::Kernel::DecodeTc;
      pl.cfg.rows_per_cta = (int)R;
      pl.cfg.row_groups = (int)rg;
      pl.cfg.warps = 4;
      pl.cfg.stages = 5;
      pl.cfg.chunk = 0;  // the key ranges follow the device-resident lengths
      pl.cfg.n_splits = (int)slots;
      pl.tile = 128;
      pl.ctas = P;
      auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
      pl.ws_bytes = 2 * al(slots * R * 4) + al(slots * R * d * 4);
      pl.units = U;  // per-unit arrival counters
      return pl;
    }
  }
  size_t smem;
  bool tensor = (elt == Elt::BF16) && !force_cudacore;
  if (tensor) {
    // bf16: warp-level tensor cores, 16-row m-tiles (up to 3 per CTA)
    int64_t mt = (rows + 15) / 16;
    if (mt > 3) mt = 3;
    pl.cfg.kernel = blkattn::Kernel::TensorCore;
    pl.cfg.rows_per_cta = (int)(16 * mt);
    pl.cfg.warps = (int)(4 * mt);
    pl.cfg.stages = 3;
    pl.tile = 64;
    smem = blkattn::decode_mma_smem_bytes(d, (int)mt);
  } else {
    int R = 1;
    while (R < rows && R < 8) R *= 2;
    pl.cfg.kernel = blkattn::Kernel::CudaCore;
    pl.cfg.rows_per_cta = R;
    pl.cfg.warps = 4;
    pl.cfg.stages = (elt == Elt::BF16) ? 3 : 2;
    pl.tile = 16 * pl.cfg.warps;
    smem = blkattn::decode_smem_bytes(elt, d, pl.cfg);
  }
  pl.cfg.row_groups = (int)((rows + pl.cfg.rows_per_cta - 1) / pl.cfg.rows_per_cta);
  const int64_t units = B * Hkv * pl.cfg.row_groups;
  const int resident = resident_ctas_per_sm(smem);
  const int64_t target = (int64_t)(sms > 0 ? sms : 148) * resident * 4;  // ~4 waves
  int64_t chunk;
  if (units >= target) {
    chunk = Tmax;
  } else {
    // small problems: down to one tile per split (a 1000-key fp32 row in 16
    // splits took 19 us against 25 us in 8; launch latency dominates either way)
    chunk = (Tmax * units + target - 1) / target;
    const int64_t min_chunk = pl.tile;
    if (chunk < min_chunk) chunk = min_chunk;
  }
  if (const char* env = std::getenv("BLKATTN_CHUNK")) {  // tuning sweeps only
    const long v = std::strtol(env, nullptr, 10);
    if (v > 0) chunk = v;
  }
  chunk = (chunk + pl.tile - 1) / pl.tile * pl.tile;
  if (chunk > Tmax) chunk = (Tmax + pl.tile - 1) / pl.tile * pl.tile;
  if (chunk > 0x40000000) chunk = 0x40000000;
  pl.cfg.chunk = (int)chunk;
  pl.cfg.n_splits = (int)((Tmax + chunk - 1) / chunk);
  pl.ctas = (int64_t)pl.cfg.n_splits * Hkv * B * pl.cfg.row_groups;
  pl.ws_bytes = 0;
  if (pl.cfg.n_splits > 1)
    pl.ws_bytes = B * Hq * Tq * (int64_t)pl.cfg.n_splits * (d + 2) * 4 + 256 * 3;
  return pl;
}

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return BLKATTN_ERR_UNSUPPORTED;
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    if (cudaError_t e = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev); e != cudaSuccess)
      return cuda_fail(e);
    if (cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_error_word); e != cudaSuccess)
      return cuda_fail(e);
    s.ready = true;
  }
  *out = &s;
  return BLKATTN_OK;
}

// ---- tiled-TMA tensor maps for the K/V cache ----
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  if (g_encode) return BLKATTN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return cuda_fail(e != cudaSuccess ? e : cudaErrorNotSupported);
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return BLKATTN_OK;
}

struct MapKey {
  int dev;
  int dtype;
  int box_cols;
  int box_rows;
  const void* ptr;
  int64_t sizes[4];
  int64_t strides[3];
  bool operator==(const MapKey& o) const {
    return dev == o.dev && dtype == o.dtype && box_cols == o.box_cols && box_rows == o.box_rows && ptr == o.ptr &&
           std::memcmp(sizes, o.sizes, sizeof sizes) == 0 && std::memcmp(strides, o.strides, sizeof strides) == 0;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used = false;
};
constexpr int kMapCache = 32;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

// 4-D map over a view [B, H, T, d] (element strides, last = 1): dims
// {d, T, H, B}, box {box_cols, box_rows, 1, 1}, 128-byte swizzle (box_cols *
// element size = 128 bytes), zero fill past T.
// The map is copied into *out: a cache entry may be replaced by the next
// lookup of the same call (a hit followed by a miss landing on that entry),
// so no caller keeps a pointer into the cache.
int tensor_map(int dev, const blkattn_tensor* t, int box_cols, int box_rows, CUtensorMap* out) {
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.dev = dev;
  key.dtype = t->dtype;
  key.box_cols = box_cols;
  key.box_rows = box_rows;
  key.ptr = t->data;
  for (int i = 0; i < 4; ++i) key.sizes[i] = t->sizes[i];
  for (int i = 0; i < 3; ++i) key.strides[i] = t->strides[i];
  for (int i = 0; i < kMapCache; ++i)
    if (g_maps[i].used && g_maps[i].key == key) {
      *out = g_maps[i].map;
      return BLKATTN_OK;
    }
  int st = get_encoder();
  if (st != BLKATTN_OK) return st;
  MapEntry& e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCache;
  const bool f32 = t->dtype == BLKATTN_F32;
  const cuuint64_t eb = f32 ? 4 : 2;
  const cuuint64_t dims[4] = {(cuuint64_t)t->sizes[3], (cuuint64_t)t->sizes[2], (cuuint64_t)t->sizes[1],
                              (cuuint64_t)t->sizes[0]};
  const cuuint64_t strides[3] = {(cuuint64_t)t->strides[2] * eb, (cuuint64_t)t->strides[1] * eb,
                                 (cuuint64_t)t->strides[0] * eb};
  const cuuint32_t box[4] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(&e.map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                              t->data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    e.used = false;
    return cuda_fail(cudaErrorInvalidValue);  // the tensor map was refused
  }
  e.key = key;
  e.used = true;
  *out = e.map;
  return BLKATTN_OK;
}

// bf16 K/V cache or Q: boxes of 64 dims (128 bytes) x box_rows rows.
int kv_tensor_map(int dev, const blkattn_tensor* t, int box_rows, CUtensorMap* out) {
  return tensor_map(dev, t, 64, box_rows, out);
}

// Whether the output can be stored by tiled TMA from the prefill kernel:
// fp32, unit dim stride, 16-byte aligned base and strides.
bool out_tma_ok(const blkattn_tensor* out) {
  if (out->dtype != BLKATTN_F32 || out->strides[3] != 1) return false;
  if ((reinterpret_cast<uintptr_t>(out->data) % 16) != 0) return false;
  for (int i = 0; i < 3; ++i)
    if ((out->strides[i] * 4) % 16 != 0 || out->strides[i] <= 0) return false;
  return true;
}

// Grow-only per-device scratch, grown stream-ordered on the call's stream:
// the old buffer is released after the work already queued there
// (cudaFreeAsync) and the new one is allocated from the device's memory pool
// in stream order (cudaMallocAsync), so no call synchronises the device.
// Work on other streams that used the old buffer must be ordered before this
// call by the caller (calls on different streams must not overlap).  Growing
// while the stream is being captured is refused (a capture may not allocate).
int grow_stream_ordered(void** buf, size_t* have, size_t bytes, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaError_t e = cudaStreamIsCapturing(stream, &cs); e != cudaSuccess) return cuda_fail(e);
  if (cs != cudaStreamCaptureStatusNone) return BLKATTN_ERR_NO_WORKSPACE;
  if (*buf) {
    if (cudaError_t e = cudaFreeAsync(*buf, stream); e != cudaSuccess) return cuda_fail(e);
    *buf = nullptr;
    *have = 0;
  }
  if (cudaError_t e = cudaMallocAsync(buf, bytes, stream); e != cudaSuccess) {
    *buf = nullptr;
    return cuda_fail(e);
  }
  *have = bytes;
  return BLKATTN_OK;
}

int ensure_workspace(DeviceState* s, size_t bytes, cudaStream_t stream) {
  if (bytes <= s->ws_bytes) return BLKATTN_OK;
  return grow_stream_ordered(&s->ws, &s->ws_bytes, bytes, stream);
}

// Grow-only per-device counters, zeroed on the call's stream when they grow
// (the kernel leaves them zero).
int ensure_counters(DeviceState* s, int64_t n, cudaStream_t stream) {
  if ((size_t)n <= s->cnt_n) return BLKATTN_OK;
  void* buf = s->cnt;
  size_t bytes = s->cnt_n * sizeof(unsigned);
  const int st = grow_stream_ordered(&buf, &bytes, (size_t)n * sizeof(unsigned), stream);
  s->cnt = static_cast<unsigned*>(buf);
  s->cnt_n = bytes / sizeof(unsigned);
  if (st != BLKATTN_OK) return st;
  if (cudaError_t e = cudaMemsetAsync(s->cnt, 0, (size_t)n * sizeof(unsigned), stream); e != cudaSuccess) {
    // the counters cannot be trusted: drop them so the next call reallocates
    cudaFreeAsync(s->cnt, stream);
    s->cnt = nullptr;
    s->cnt_n = 0;
    return cuda_fail(e);
  }
  return BLKATTN_OK;
}

struct Checked {
  int32_t device;  // the ordinal every tensor of the call names
  int64_t B, Hq, Hkv, Tq, Tmax, d;
  int64_t window = 0;  // sliding window (0: none)
  Elt elt;
  bool prefill_ok;  // no bias and q rows movable by TMA (see make_plan)
  bool q_vec_ok;    // query rows contiguous and 16-byte aligned
};

int validate_fwd(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                 const blkattn_tensor* sl, const blkattn_tensor* qp, const blkattn_tensor* tree,
                 const blkattn_tensor* bias, const blkattn_tensor* out, const blkattn_tensor* lse,
                 Checked* c) {
  if (!dims_ok(q, 4) || !dims_ok(k, 4) || !dims_ok(v, 4) || !dims_ok(sl, 1) ||
      !dims_ok(qp, 2) || !dims_ok(out, 4) || !dims_ok(lse, 3))
    return BLKATTN_ERR_INVALID_ARG;
  if (bias && !dims_ok(bias, 4)) return BLKATTN_ERR_INVALID_ARG;
  if (tree && (!dims_ok(tree, 2) || tree->dtype != BLKATTN_I64)) return BLKATTN_ERR_INVALID_ARG;
  if (!is_float_dtype(q->dtype) || k->dtype != q->dtype || v->dtype != q->dtype)
    return BLKATTN_ERR_INVALID_ARG;
  if (sl->dtype != BLKATTN_I32 || qp->dtype != BLKATTN_I32) return BLKATTN_ERR_INVALID_ARG;
  if (!is_float_dtype(out->dtype) || lse->dtype != BLKATTN_F32) return BLKATTN_ERR_INVALID_ARG;
  if (bias && bias->dtype != BLKATTN_F32) return BLKATTN_ERR_INVALID_ARG;
  if (!same_device(q, {k, v, sl, qp, tree, bias, out, lse})) return BLKATTN_ERR_INVALID_ARG;
  c->device = q->device;

  c->B = q->sizes[0];
  c->Hq = q->sizes[1];
  c->Tq = q->sizes[2];
  c->d = q->sizes[3];
  c->Hkv = k->sizes[1];
  c->Tmax = k->sizes[2];
  const int64_t B = c->B, Hq = c->Hq, Tq = c->Tq, d = c->d, Hkv = c->Hkv, Tmax = c->Tmax;
  if (k->sizes[0] != B || v->sizes[0] != B || sl->sizes[0] != B || qp->sizes[0] != B ||
      out->sizes[0] != B || lse->sizes[0] != B)
    return BLKATTN_ERR_INVALID_ARG;
  if (out->sizes[1] != Hq || lse->sizes[1] != Hq || v->sizes[1] != Hkv)
    return BLKATTN_ERR_INVALID_ARG;
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return BLKATTN_ERR_INVALID_ARG;
  if (qp->sizes[1] != Tq || out->sizes[2] != Tq || lse->sizes[2] != Tq)
    return BLKATTN_ERR_INVALID_ARG;
  if (Tmax < 1 || v->sizes[2] != Tmax) return BLKATTN_ERR_INVALID_ARG;
  if (k->sizes[3] != d || v->sizes[3] != d || out->sizes[3] != d) return BLKATTN_ERR_INVALID_ARG;
  // a token tree: one 64-bit node mask per (sequence, query row)
  if (tree && (tree->sizes[0] != B || tree->sizes[1] != Tq || Tq > 64)) return BLKATTN_ERR_INVALID_ARG;
  if (bias) {  // each dim is full-size or 1 (a size-1 dim broadcasts)
    const int64_t full[4] = {B, Hq, Tq, Tmax};
    for (int i = 0; i < 4; ++i)
      if (bias->sizes[i] != full[i] && bias->sizes[i] != 1) return BLKATTN_ERR_INVALID_ARG;
  }
  // cache rows move with 16-byte bulk copies
  const int eb = elt_bytes(q->dtype);
  for (const blkattn_tensor* t : {k, v}) {
    if (t->strides[3] != 1) return BLKATTN_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
      if ((t->strides[i] * eb) % 16 != 0) return BLKATTN_ERR_INVALID_ARG;
  }
  const bool empty = (B == 0 || Tq == 0);
  if (!empty) {
    for (const blkattn_tensor* t : {q, k, v, sl, qp, out, lse})
      if (t->data == nullptr) return BLKATTN_ERR_INVALID_ARG;
    if (bias && bias->data == nullptr) return BLKATTN_ERR_INVALID_ARG;
    if (tree && tree->data == nullptr) return BLKATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k->data) | reinterpret_cast<uintptr_t>(v->data)) % 16 != 0)
      return BLKATTN_ERR_INVALID_ARG;
  }
  // 32-bit index ranges used on the device, grid limits
  if (B > 0x7fffffff || Hq > 0xffff || Hkv > 0xffff || Tq > 0x7fffffff || Tmax > 0x7fffffff)
    return BLKATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return BLKATTN_ERR_UNSUPPORTED;
  c->elt = (q->dtype == BLKATTN_BF16) ? Elt::BF16 : Elt::F32;
  c->q_vec_ok = q->strides[3] == 1 && (reinterpret_cast<uintptr_t>(q->data) % 16) == 0 &&
                (q->strides[0] * 2) % 16 == 0 && (q->strides[1] * 2) % 16 == 0 &&
                (q->strides[2] * 2) % 16 == 0;
  c->prefill_ok = bias == nullptr && tree == nullptr && c->q_vec_ok;
  return BLKATTN_OK;
}

// Kernel parameters of one call; `ws` holds the per-split partial states
// when the plan has more than one split (m, l, u in 256-byte aligned parts).
FwdParams fill_params(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                      const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                      const blkattn_tensor* tree, const blkattn_tensor* mask_bias, float scale,
                      const blkattn_tensor* out,
                      const blkattn_tensor* lse, const Checked& c, const Plan& pl, void* ws, int* err,
                      unsigned* counters) {
  const int eb = elt_bytes(q->dtype);
  FwdParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q->data;
  p.q_sb = q->strides[0]; p.q_sh = q->strides[1]; p.q_si = q->strides[2]; p.q_sd = q->strides[3];
  p.k = static_cast<const char*>(k->data);
  p.v = static_cast<const char*>(v->data);
  p.k_sb = k->strides[0] * eb; p.k_sh = k->strides[1] * eb; p.k_st = k->strides[2] * eb;
  p.v_sb = v->strides[0] * eb; p.v_sh = v->strides[1] * eb; p.v_st = v->strides[2] * eb;
  p.seqlens = static_cast<const int32_t*>(seqlens_k->data);
  p.sl_s = seqlens_k->strides[0];
  p.qpos = static_cast<const int32_t*>(q_logical_pos->data);
  p.qp_sb = q_logical_pos->strides[0]; p.qp_si = q_logical_pos->strides[1];
  if (mask_bias) {
    p.bias = static_cast<const float*>(mask_bias->data);
    int64_t bs[4];
    for (int i = 0; i < 4; ++i) bs[i] = mask_bias->sizes[i] == 1 ? 0 : mask_bias->strides[i];
    p.bi_sb = bs[0]; p.bi_sh = bs[1]; p.bi_si = bs[2]; p.bi_sj = bs[3];
  }
  if (tree) {
    p.tree = static_cast<const int64_t*>(tree->data);
    p.tr_sb = tree->strides[0];
    p.tr_si = tree->strides[1];
  }
  p.window = (int)c.window;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = out->data;
  p.out_bf16 = out->dtype == BLKATTN_BF16;
  p.o_sb = out->strides[0]; p.o_sh = out->strides[1]; p.o_si = out->strides[2]; p.o_sd = out->strides[3];
  p.lse = static_cast<float*>(lse->data);
  p.l_sb = lse->strides[0]; p.l_sh = lse->strides[1]; p.l_si = lse->strides[2];
  p.B = (int)c.B; p.Hq = (int)c.Hq; p.Hkv = (int)c.Hkv; p.G = (int)(c.Hq / c.Hkv);
  p.Tq = (int)c.Tq; p.Tmax = (int)c.Tmax;
  p.rows_per_head = (int)(p.G * c.Tq);
  p.row_groups = pl.cfg.row_groups;
  p.chunk = pl.cfg.chunk;
  p.n_splits = pl.cfg.n_splits;
  p.rows_cta = pl.cfg.rows_per_cta;
  p.unit_cnt = counters;
  if (pl.cfg.kernel == blkattn::Kernel::DecodeTc) {
    // per-CTA partial states: [slots][rows_cta] (m, l), [slots][rows_cta][d] (u)
    auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
    const int64_t n = (int64_t)pl.cfg.n_splits * pl.cfg.rows_per_cta;
    char* base = static_cast<char*>(ws);
    p.ws_m = reinterpret_cast<float*>(base);
    p.ws_l = reinterpret_cast<float*>(base + al(n * 4));
    p.ws_u = reinterpret_cast<float*>(base + 2 * al(n * 4));
  } else if (pl.cfg.n_splits > 1) {
    const int64_t n = c.B * c.Hq * c.Tq * (int64_t)pl.cfg.n_splits;
    char* base = static_cast<char*>(ws);
    p.ws_m = reinterpret_cast<float*>(base);
    p.ws_l = reinterpret_cast<float*>(base + ((n * 4 + 255) / 256) * 256);
    p.ws_u = reinterpret_cast<float*>(base + 2 * ((n * 4 + 255) / 256) * 256);
  }
  p.err = err;
  p.test_stall_cta = -1;
  // prefill dispatch groups: (sequence, head) pairs whose K and V take about
  // a quarter of the L2 cache together (129 MB on GB300; queried once per
  // device): with half, the causal prefill read its K/V 1.7 times from DRAM,
  // with a quarter once, in the same time
  {
    static int l2_bytes = 0;
    if (l2_bytes == 0) {
      int dev = 0, v = 0;
      if (cudaGetDevice(&dev) == cudaSuccess &&
          cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) == cudaSuccess && v > 0)
        l2_bytes = v;
      else
        l2_bytes = 64 << 20;
    }
    const int64_t kv_per_head = 2 * c.Tmax * c.d * elt_bytes(q->dtype);
    int64_t hg = (l2_bytes / 4) / (kv_per_head > 0 ? kv_per_head : 1);
    const int64_t heads = c.B * c.Hq;
    hg = hg < 1 ? 1 : (hg > heads ? heads : hg);
    p.head_group = (int)hg;
  }
  return p;
}

// Enqueue the split-KV kernel and, with more than one split, the merge.
int launch_fwd(const FwdParams& p, const Checked& c, const Plan& pl, const blkattn_tensor* q,
               const blkattn_tensor* k, const blkattn_tensor* v, const blkattn_tensor* out,
               cudaStream_t stream) {
  cudaError_t le;
  if (pl.cfg.kernel == blkattn::Kernel::DecodeTc) {
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_fail(e);
    CUtensorMap mk, mv;
    int st = kv_tensor_map(dev, k, 128, &mk);
    if (st != BLKATTN_OK) return st;
    st = kv_tensor_map(dev, v, 128, &mv);
    if (st != BLKATTN_OK) return st;
    FwdParams pt = p;
    if (g_stall_next >= 0) {  // test hook: one launch only
      pt.test_stall_cta = (int)(g_stall_next % pl.ctas);
      g_stall_next = -1;
    }
    le = blkattn::launch_decode_tc(pt, (int)pl.ctas, mk, mv, stream);
  } else if (pl.cfg.kernel == blkattn::Kernel::TensorCore || pl.cfg.kernel == blkattn::Kernel::Prefill) {
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_fail(e);
    CUtensorMap mk, mv;
    // K/V boxes: 64 keys for the split-KV kernel, 128 for the prefill kernel
    const int kv_rows = (pl.cfg.kernel == blkattn::Kernel::Prefill) ? 128 : 64;
    int st = kv_tensor_map(dev, k, kv_rows, &mk);
    if (st != BLKATTN_OK) return st;
    st = kv_tensor_map(dev, v, kv_rows, &mv);
    if (st != BLKATTN_OK) return st;
    if (pl.cfg.kernel == blkattn::Kernel::Prefill) {
      CUtensorMap mq;
      st = kv_tensor_map(dev, q, 128, &mq);
      if (st != BLKATTN_OK) return st;
      // whole output tiles by TMA where the output layout allows it
      FwdParams pp = p;
      CUtensorMap mo = mq;  // not read unless pp.o_tma
      pp.o_tma = 0;
      if (out_tma_ok(out)) {
        st = tensor_map(dev, out, 32, 32, &mo);
        if (st != BLKATTN_OK) return st;
        pp.o_tma = 1;
      }
      le = blkattn::launch_prefill_tc(pp, pl.cfg.row_groups, mq, mk, mv, mo, stream);
    } else {
      le = blkattn::launch_decode_mma(p, (int)c.d, pl.cfg, mk, mv, stream);
    }
  } else {
    le = blkattn::launch_decode_split(p, c.elt, (int)c.d, pl.cfg, stream);
  }
  if (le != cudaSuccess) return cuda_fail(le);
  if (g_split_event != nullptr)
    if (cudaError_t e = cudaEventRecord(g_split_event, stream); e != cudaSuccess) return cuda_fail(e);
  // the tcgen05 decode kernel folds its split units itself
  if (pl.cfg.kernel != blkattn::Kernel::DecodeTc && pl.cfg.n_splits > 1)
    if (cudaError_t e = blkattn::launch_split_merge(p, (int)c.d, stream); e != cudaSuccess) return cuda_fail(e);
  return BLKATTN_OK;
}

}  // namespace

namespace blkattn {

int validate_fwd_args(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                      const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                      const blkattn_tensor* mask_bias, const blkattn_tensor* out,
                      const blkattn_tensor* lse) {
  Checked c;
  return validate_fwd(q, k, v, seqlens_k, q_logical_pos, nullptr, mask_bias, out, lse, &c);
}

// blkattn_fwd with caller-provided scratch for the per-split states instead
// of the library's grow-only workspace.  Never allocates device memory.
int fwd_with_scratch(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                     const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                     const blkattn_tensor* tree, const blkattn_tensor* mask_bias, float scale,
                     const blkattn_tensor* out, const blkattn_tensor* lse, blkattn_stream_t stream_,
                     void* scratch, size_t scratch_bytes) {
  Checked c;
  int st = validate_fwd(q, k, v, seqlens_k, q_logical_pos, tree, mask_bias, out, lse, &c);
  if (st != BLKATTN_OK) return st;
  if (c.B == 0 || c.Tq == 0) return BLKATTN_OK;
  if ((st = check_current_device(c.device)) != BLKATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != BLKATTN_OK) return st;
  const Plan pl = make_plan(c.B, c.Hq, c.Hkv, c.Tq, c.Tmax, (int)c.d, c.elt, ds->sms,
                            c.prefill_ok && scale > 0.f, c.q_vec_ok);
  if ((pl.cfg.kernel == blkattn::Kernel::TensorCore || pl.cfg.kernel == blkattn::Kernel::CudaCore) &&
      c.B * pl.cfg.row_groups > 65535)
    return BLKATTN_ERR_UNSUPPORTED;  // grid z of the split-KV kernels
  // the last kStaticCounterBytes hold the per-unit counters (zero initially,
  // left zero by every call); plans get the rest
  if (scratch_bytes < blkattn::kStaticCounterBytes) return BLKATTN_ERR_SCRATCH_LIMIT;
  const size_t usable = scratch_bytes - blkattn::kStaticCounterBytes;
  if ((size_t)pl.ws_bytes > usable) return BLKATTN_ERR_SCRATCH_LIMIT;
  if ((size_t)pl.units * sizeof(unsigned) > blkattn::kStaticCounterBytes) return BLKATTN_ERR_SCRATCH_LIMIT;
  unsigned* counters = reinterpret_cast<unsigned*>(static_cast<char*>(scratch) + usable);
  const FwdParams p = fill_params(q, k, v, seqlens_k, q_logical_pos, tree, mask_bias, scale, out, lse, c,
                                  pl, scratch, ds->err, counters);
  return launch_fwd(p, c, pl, q, k, v, out, stream);
}

// blkattn_fwd and blkattn_fwd_tree: the library's grow-only workspace and
// per-unit counters.
int fwd_impl(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
             const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos, const blkattn_tensor* tree,
             int64_t window, const blkattn_tensor* mask_bias, float scale, const blkattn_tensor* out,
             const blkattn_tensor* lse, blkattn_stream_t stream_) {
  Checked c;
  int st = validate_fwd(q, k, v, seqlens_k, q_logical_pos, tree, mask_bias, out, lse, &c);
  if (st != BLKATTN_OK) return st;
  if (window < 0 || window > 0x7fffffff || (window > 0 && tree != nullptr)) return BLKATTN_ERR_INVALID_ARG;
  c.window = window;  // (the prefill kernel takes windows too: a first key tile per CTA and a window mask)
  if (c.B == 0 || c.Tq == 0) return BLKATTN_OK;
  if ((st = check_current_device(c.device)) != BLKATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != BLKATTN_OK) return st;
  const Plan pl = make_plan(c.B, c.Hq, c.Hkv, c.Tq, c.Tmax, (int)c.d, c.elt, ds->sms,
                            c.prefill_ok && scale > 0.f, c.q_vec_ok, c.window > 0);
  if ((pl.cfg.kernel == blkattn::Kernel::TensorCore || pl.cfg.kernel == blkattn::Kernel::CudaCore) &&
      c.B * pl.cfg.row_groups > 65535)
    return BLKATTN_ERR_UNSUPPORTED;  // grid z of the split-KV kernels
  if (pl.ws_bytes > 0) {
    st = ensure_workspace(ds, (size_t)pl.ws_bytes, stream);
    if (st != BLKATTN_OK) return st;
  }
  if (pl.units > 0) {
    st = ensure_counters(ds, pl.units, stream);
    if (st != BLKATTN_OK) return st;
  }
  const FwdParams p = fill_params(q, k, v, seqlens_k, q_logical_pos, tree, mask_bias, scale, out, lse, c, pl,
                                  ds->ws, ds->err, ds->cnt);
  return launch_fwd(p, c, pl, q, k, v, out, stream);
}

// CUDA failures of entry points outside this file: recorded for
// blkattn_last_cuda_error like the ones here.
int report_cuda_failure(cudaError_t e) { return cuda_fail(e); }

int device_error_word(int** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  const int st = device_state(&ds);
  if (st == BLKATTN_OK) *out = ds->err;
  return st;
}

namespace {

// fp32 gradient rows written with 16-byte vector stores: unit dim stride,
// 16-byte aligned base and strides.
bool grad_rows_ok(const blkattn_tensor* t) {
  if (t->dtype != BLKATTN_F32 || t->strides[3] != 1) return false;
  if ((reinterpret_cast<uintptr_t>(t->data) % 16) != 0) return false;
  for (int i = 0; i < 3; ++i)
    if ((t->strides[i] * 4) % 16 != 0) return false;
  return true;
}

// bf16 rows moved by tiled TMA: unit dim stride, 16-byte aligned base and strides.
bool tma_rows_ok(const blkattn_tensor* t) {
  if (t->dtype != BLKATTN_BF16 || t->strides[3] != 1) return false;
  if ((reinterpret_cast<uintptr_t>(t->data) % 16) != 0) return false;
  for (int i = 0; i < 3; ++i)
    if ((t->strides[i] * 2) % 16 != 0) return false;
  return true;
}

}  // namespace

int bwd_impl(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
             const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
             const blkattn_tensor* mask_bias, float scale, const blkattn_tensor* out,
             const blkattn_tensor* lse, const blkattn_tensor* dout, const blkattn_tensor* dq,
             const blkattn_tensor* dk, const blkattn_tensor* dv, int64_t window, blkattn_stream_t stream_) {
  if (window < 0 || window > 0x7fffffff) return BLKATTN_ERR_INVALID_ARG;
  Checked c;
  int st = validate_fwd(q, k, v, seqlens_k, q_logical_pos, nullptr, mask_bias, out, lse, &c);
  if (st != BLKATTN_OK) return st;
  if (!dims_ok(dout, 4) || !dims_ok(dq, 4) || !dims_ok(dk, 4) || !dims_ok(dv, 4)) return BLKATTN_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) {
    if (dout->sizes[i] != q->sizes[i] || dq->sizes[i] != q->sizes[i]) return BLKATTN_ERR_INVALID_ARG;
    if (dk->sizes[i] != k->sizes[i] || dv->sizes[i] != k->sizes[i]) return BLKATTN_ERR_INVALID_ARG;
  }
  if (dout->dtype != q->dtype || dq->dtype != BLKATTN_F32 || dk->dtype != BLKATTN_F32 || dv->dtype != BLKATTN_F32)
    return BLKATTN_ERR_INVALID_ARG;
  if (!same_device(q, {dout, dq, dk, dv})) return BLKATTN_ERR_INVALID_ARG;
  if (!(scale == scale) || scale == __builtin_huge_valf() || scale == -__builtin_huge_valf())
    return BLKATTN_ERR_INVALID_ARG;
  if (c.B == 0) return BLKATTN_OK;
  const bool rows = c.Tq > 0;
  if (dk->data == nullptr || dv->data == nullptr) return BLKATTN_ERR_INVALID_ARG;
  if (rows && (dout->data == nullptr || dq->data == nullptr)) return BLKATTN_ERR_INVALID_ARG;
  if (!grad_rows_ok(dk) || !grad_rows_ok(dv) || (rows && !grad_rows_ok(dq))) return BLKATTN_ERR_INVALID_ARG;
  // the tensor-core backward: bf16 operands, d = 128, TMA-movable Q and g_o
  // rows, at most 1024 query tiles of 128 rows per sequence
  if (c.elt != Elt::BF16 || c.d != 128 || c.Tq > 131072) return BLKATTN_ERR_UNSUPPORTED;
  if (rows && (!tma_rows_ok(q) || !tma_rows_ok(dout))) return BLKATTN_ERR_INVALID_ARG;
  if ((st = check_current_device(c.device)) != BLKATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != BLKATTN_OK) return st;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_fail(e);
  const int64_t n_qt = (c.Tq + 127) / 128;
  const int64_t n_kt = (c.Tmax + 127) / 128;
  const int64_t nrows = c.B * c.Hq * c.Tq;
  auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t ws = 2 * al(nrows * 4) + 2 * al(c.B * n_qt * 4);
  st = ensure_workspace(ds, (size_t)(ws > 0 ? ws : 256), stream);
  if (st != BLKATTN_OK) return st;
  CUtensorMap tmk, tmv, tmq, tmg;
  if ((st = kv_tensor_map(dev, k, 128, &tmk)) != BLKATTN_OK) return st;
  if ((st = kv_tensor_map(dev, v, 128, &tmv)) != BLKATTN_OK) return st;
  if (rows) {
    if ((st = kv_tensor_map(dev, q, 128, &tmq)) != BLKATTN_OK) return st;
    if ((st = kv_tensor_map(dev, dout, 128, &tmg)) != BLKATTN_OK) return st;
  } else {
    tmq = tmk;  // no query rows: the dK/dV kernel writes zeros and reads no query tile
    tmg = tmk;
  }
  BwdParams p{};
  p.out = out->data;
  p.out_bf16 = out->dtype == BLKATTN_BF16;
  p.out_vec = rows && out_tma_ok(out);  // fp32, unit dim stride, 16-byte aligned rows
  p.o_sb = out->strides[0]; p.o_sh = out->strides[1]; p.o_si = out->strides[2]; p.o_sd = out->strides[3];
  p.lse = static_cast<const float*>(lse->data);
  p.l_sb = lse->strides[0]; p.l_sh = lse->strides[1]; p.l_si = lse->strides[2];
  p.dout = dout->data;
  p.g_sb = dout->strides[0]; p.g_sh = dout->strides[1]; p.g_si = dout->strides[2];
  p.seqlens = static_cast<const int*>(seqlens_k->data);
  p.sl_s = seqlens_k->strides[0];
  p.qpos = static_cast<const int*>(q_logical_pos->data);
  p.qp_sb = q_logical_pos->strides[0]; p.qp_si = q_logical_pos->strides[1];
  p.bias = mask_bias ? static_cast<const float*>(mask_bias->data) : nullptr;
  if (mask_bias) {  // size-1 dims broadcast
    p.bi_sb = mask_bias->sizes[0] == 1 ? 0 : mask_bias->strides[0];
    p.bi_sh = mask_bias->sizes[1] == 1 ? 0 : mask_bias->strides[1];
    p.bi_si = mask_bias->sizes[2] == 1 ? 0 : mask_bias->strides[2];
    p.bi_sj = mask_bias->sizes[3] == 1 ? 0 : mask_bias->strides[3];
  }
  p.dq = static_cast<float*>(dq->data);
  p.dq_sb = dq->strides[0]; p.dq_sh = dq->strides[1]; p.dq_si = dq->strides[2];
  p.dk = static_cast<float*>(dk->data);
  p.dk_sb = dk->strides[0]; p.dk_sh = dk->strides[1]; p.dk_sj = dk->strides[2];
  p.dv = static_cast<float*>(dv->data);
  p.dv_sb = dv->strides[0]; p.dv_sh = dv->strides[1]; p.dv_sj = dv->strides[2];
  char* base = static_cast<char*>(ds->ws);
  p.ws_D = reinterpret_cast<float*>(base);
  p.ws_L = reinterpret_cast<float*>(base + al(nrows * 4));
  p.ws_end = reinterpret_cast<int*>(base + 2 * al(nrows * 4));
  p.ws_start = reinterpret_cast<int*>(base + 2 * al(nrows * 4) + al(c.B * n_qt * 4));
  p.window = (int)window;
  p.B = (int)c.B; p.Hq = (int)c.Hq; p.Hkv = (int)c.Hkv; p.G = (int)(c.Hq / c.Hkv);
  p.Tq = (int)c.Tq; p.Tmax = (int)c.Tmax; p.n_qt = (int)n_qt; p.n_kt = (int)n_kt;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = ds->err;
  {
    // L2-sized dispatch groups: half the L2 for the operands a group streams
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0) l2 = 64 << 20;
    const int64_t kv_head = 2 * c.Tmax * 128 * 2;              // K and V of one (sequence, KV head)
    const int64_t q_unit = 2 * (c.Hq / c.Hkv) * c.Tq * 128 * 2;  // Q and g_o of its G query heads
    auto clamp = [](int64_t x, int64_t hi) { return x < 1 ? 1 : (x > hi ? hi : x); };
    p.hg_q = (int)clamp((l2 / 2) / kv_head, c.B * c.Hq);
    p.hg_kv = (int)clamp((l2 / 2) / (q_unit > 0 ? q_unit : 1), c.B * c.Hkv);
  }
  if (cudaError_t e = launch_backward(p, tmq, tmg, tmk, tmv, stream); e != cudaSuccess) return cuda_fail(e);
  return BLKATTN_OK;
}

}  // namespace blkattn

extern "C" {

const char* blkattn_status_string(int status) {
  switch (status) {
    case BLKATTN_OK: return "ok";
    case BLKATTN_ERR_INVALID_ARG: return "invalid argument (shape, dtype, stride, alignment or head grouping)";
    case BLKATTN_ERR_UNSUPPORTED: return "unsupported configuration (head dim, dtype or size)";
    case BLKATTN_ERR_CUDA: return "CUDA runtime or launch error";
    case BLKATTN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
    case BLKATTN_ERR_NO_WORKSPACE: return "workspace would have to grow during stream capture";
    case BLKATTN_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed static maximum";
  }
  return "unknown status";
}

int blkattn_debug_plan(int64_t B, int64_t H_q, int64_t H_kv, int64_t T_q, int64_t T_max,
                       int64_t d, int32_t dtype, int32_t num_sms, blkattn_plan* plan) {
  if (plan == nullptr || B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || T_q < 0 ||
      T_max < 1 || (d != 64 && d != 128) || !is_float_dtype(dtype) || num_sms <= 0)
    return BLKATTN_ERR_INVALID_ARG;
  const Plan pl = make_plan(B, H_q, H_kv, T_q, T_max, (int)d,
                            dtype == BLKATTN_BF16 ? Elt::BF16 : Elt::F32, num_sms, true, true);
  plan->kernel = (int32_t)pl.cfg.kernel;
  plan->rows_per_cta = pl.cfg.rows_per_cta;
  plan->row_groups = pl.cfg.row_groups;
  plan->chunk_keys = pl.cfg.chunk;
  plan->n_splits = pl.cfg.n_splits;
  plan->tile_keys = pl.tile;
  plan->ctas = pl.ctas;
  plan->workspace_bytes = pl.ws_bytes;
  return BLKATTN_OK;
}

int blkattn_fwd(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                const blkattn_tensor* mask_bias, float scale, const blkattn_tensor* out,
                const blkattn_tensor* lse, blkattn_stream_t stream_) {
  return blkattn::fwd_impl(q, k, v, seqlens_k, q_logical_pos, nullptr, 0, mask_bias, scale, out, lse, stream_);
}

int blkattn_fwd_tree(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                     const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                     const blkattn_tensor* tree_mask, const blkattn_tensor* mask_bias, float scale,
                     const blkattn_tensor* out, const blkattn_tensor* lse, blkattn_stream_t stream_) {
  if (tree_mask == nullptr) return BLKATTN_ERR_INVALID_ARG;
  return blkattn::fwd_impl(q, k, v, seqlens_k, q_logical_pos, tree_mask, 0, mask_bias, scale, out, lse, stream_);
}

int blkattn_fwd_window(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                       const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos, int64_t window,
                       const blkattn_tensor* mask_bias, float scale, const blkattn_tensor* out,
                       const blkattn_tensor* lse, blkattn_stream_t stream_) {
  if (window < 1) return BLKATTN_ERR_INVALID_ARG;
  return blkattn::fwd_impl(q, k, v, seqlens_k, q_logical_pos, nullptr, window, mask_bias, scale, out, lse, stream_);
}

int blkattn_bwd(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos,
                const blkattn_tensor* mask_bias, float scale, const blkattn_tensor* out,
                const blkattn_tensor* lse, const blkattn_tensor* dout, const blkattn_tensor* dq,
                const blkattn_tensor* dk, const blkattn_tensor* dv, blkattn_stream_t stream) {
  if (!q || !k || !v || !seqlens_k || !q_logical_pos || !out || !lse || !dout || !dq || !dk || !dv)
    return BLKATTN_ERR_INVALID_ARG;
  return blkattn::bwd_impl(q, k, v, seqlens_k, q_logical_pos, mask_bias, scale, out, lse, dout, dq, dk, dv, 0,
                           stream);
}

int blkattn_bwd_window(const blkattn_tensor* q, const blkattn_tensor* k, const blkattn_tensor* v,
                       const blkattn_tensor* seqlens_k, const blkattn_tensor* q_logical_pos, int64_t window,
                       const blkattn_tensor* mask_bias, float scale, const blkattn_tensor* out,
                       const blkattn_tensor* lse, const blkattn_tensor* dout, const blkattn_tensor* dq,
                       const blkattn_tensor* dk, const blkattn_tensor* dv, blkattn_stream_t stream) {
  if (!q || !k || !v || !seqlens_k || !q_logical_pos || !out || !lse || !dout || !dq || !dk || !dv)
    return BLKATTN_ERR_INVALID_ARG;
  if (window < 1) return BLKATTN_ERR_INVALID_ARG;
  return blkattn::bwd_impl(q, k, v, seqlens_k, q_logical_pos, mask_bias, scale, out, lse, dout, dq, dk, dv,
                           window, stream);
}

int blkattn_merge(const blkattn_states* a, const blkattn_states* b, const blkattn_states* out,
                  blkattn_stream_t stream_) {
  if (!a || !b || !out) return BLKATTN_ERR_INVALID_ARG;
  if (a->rows != b->rows || a->rows != out->rows || a->d_v != b->d_v || a->d_v != out->d_v)
    return BLKATTN_ERR_INVALID_ARG;
  if (a->rows < 0 || a->d_v < 1 || a->d_v > 1024) return BLKATTN_ERR_INVALID_ARG;
  for (const blkattn_states* s : {a, b, out})
    if (s->u_row_stride < s->d_v) return BLKATTN_ERR_INVALID_ARG;
  if (a->rows == 0) return BLKATTN_OK;
  for (const blkattn_states* s : {a, b, out})
    if (s->m == nullptr || s->u == nullptr) return BLKATTN_ERR_INVALID_ARG;
  blkattn::MergeParams p;
  p.am = a->m; p.al = a->l; p.au = a->u; p.a_us = a->u_row_stride;
  p.bm = b->m; p.bl = b->l; p.bu = b->u; p.b_us = b->u_row_stride;
  p.om = out->m; p.ol = out->l; p.ou = out->u; p.o_us = out->u_row_stride;
  p.rows = a->rows;
  p.d = a->d_v;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaError_t e = blkattn::launch_state_merge(p, stream); e != cudaSuccess) return cuda_fail(e);
  return BLKATTN_OK;
}

void blkattn_debug_stall_next_decode(int32_t cta) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_stall_next = cta < 0 ? -1 : cta;
}

void blkattn_debug_set_split_event(void* ev) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_split_event = static_cast<cudaEvent_t>(ev);
}

const char* blkattn_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(g_last_cuda_error);
}

int blkattn_check_device_error(blkattn_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaError_t e = cudaStreamSynchronize(stream); e != cudaSuccess) return cuda_fail(e);
  int word = 0;
  if (cudaError_t e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof word); e != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    const int zero = 0;
    if (cudaError_t e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero); e != cudaSuccess) return cuda_fail(e);
    // a kernel that gave up may have left unit counters behind: restart them
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
      std::lock_guard<std::mutex> lock(g_mu);
      DeviceState& ds = g_dev[dev];
      if (ds.cnt)
        if (cudaError_t e = cudaMemset(ds.cnt, 0, ds.cnt_n * sizeof(unsigned)); e != cudaSuccess) return cuda_fail(e);
    }
    blkattn::clear_static_counters();
    return BLKATTN_ERR_DEVICE_TIMEOUT;
  }
  return BLKATTN_OK;
}

}  // extern "C"
