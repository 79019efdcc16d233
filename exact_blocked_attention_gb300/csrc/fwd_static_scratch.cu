// blkattn_fwd_static_scratch: blkattn_fwd for callers that must not allocate
// device memory at call time (a framework that owns all device memory through
// its own pool, a latency-critical loop that cannot take cudaMalloc's
// synchronisation, a runtime that forbids allocation after start-up).
//
// The split kernels' partial states go to one fixed array that is part of
// the library image, so the call allocates nothing.  The array is shared by
// every call on a device and keeps the last call's contents.  Its last
// kStaticCounterBytes hold the tcgen05 decode kernel's per-unit counters:
// zero when the library loads and left zero by every call; the rest never
// has to start at zero (each call writes every state it reads back).  Calls
// that overlap on the GPU race on it.
#include <mutex>

#include "blkattn.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = BLKATTN_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Resident on every device that loads the library, until the process exits.
// In host code this name is only a host-side handle: the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev_addr[kMaxDevices];  // per device, looked up once

// Device address of the array on the current device; the first call on a
// device looks it up (with that device current) and caches it.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BLKATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BLKATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr)
      return BLKATTN_ERR_CUDA;
    g_scratch_dev_addr[dev] = ptr;
  }
  *out = g_scratch_dev_addr[dev];
  return BLKATTN_OK;
}

}  // namespace

namespace blkattn {
// After a kernel gave up a bounded wait: zero the counters region of the
// array on the current device (if this device ever used it).
void clear_static_counters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev_addr[dev] != nullptr)
    cudaMemset(static_cast<char*>(g_scratch_dev_addr[dev]) + kScratchBytes - kStaticCounterBytes, 0,
               kStaticCounterBytes);
}
}  // namespace blkattn

extern "C" int blkattn_fwd_static_scratch(const blkattn_tensor* q, const blkattn_tensor* k,
                                          const blkattn_tensor* v, const blkattn_tensor* seqlens_k,
                                          const blkattn_tensor* q_logical_pos,
                                          const blkattn_tensor* mask_bias, float scale,
                                          const blkattn_tensor* out, const blkattn_tensor* lse,
                                          blkattn_stream_t stream) {
  // invalid requests fail before any CUDA call, as in blkattn_fwd
  int st = blkattn::validate_fwd_args(q, k, v, seqlens_k, q_logical_pos, mask_bias, out, lse);
  if (st != BLKATTN_OK) return st;
  if (q->sizes[0] == 0 || q->sizes[2] == 0) return BLKATTN_OK;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != BLKATTN_OK) return st;
  return blkattn::fwd_with_scratch(q, k, v, seqlens_k, q_logical_pos, nullptr, mask_bias, scale, out, lse,
                                   stream, scratch, kScratchBytes);
}
