/*
 * libblkattn — exact blocked attention over a KV cache on GB300 (sm_103a).
 *
 * C ABI.  No torch types, no C++ types; every pointer in a descriptor is a
 * DEVICE pointer on the current CUDA device unless stated otherwise.  The
 * caller owns every buffer it passes.  No call reads device memory from the
 * host (cache lengths and positions stay on the device), so a call can be
 * captured in a CUDA graph once the library's workspace has been sized by an
 * earlier uncaptured call of the same or a larger problem.
 *
 * What is computed ("Chapter 33: inference compute optimisation", §33.2,
 * eq. 33.2): for every query row (b, h, i)
 *
 *     z_j = scale * (q[b,h,i,:] . k[b,hk,j,:]) + M[b,h,i,j]
 *     out[b,h,i,:] = sum_j e^{z_j} v[b,hk,j,:] / sum_j e^{z_j}
 *     lse[b,h,i]   = ln sum_j e^{z_j}
 *
 * over the VALID keys j, with hk = floor(h / (H_q / H_kv)) (grouped-query
 * heads, contiguous groups; the head-grouping condition of §33.3 "interface,
 * backend and correctness conditions").  Key j is valid for row (b, h, i) iff
 *
 *     j < min(seqlens_k[b], T_max)              (the key exists in the cache)
 *     j <= q_logical_pos[b, i]                  (causal by LOGICAL position)
 *     M[b,h,i,j] != -inf                        (additive mask, when given)
 *
 * Logical positions follow "Generation and Caching with the Same Model"
 * (cache reuse: after a cache of length t the new queries sit at t, t+1, ...)
 * and §33.3 of Chapter 33 (a decode row must not be aligned from zero).  A
 * non-causal row is expressed with q_logical_pos >= seqlens_k[b] - 1.
 *
 * A row with no valid key gets out = 0 (all +0.0) and lse = -inf: the defined
 * output that §33.2 asks an interface to fix for a fully masked row (the
 * paragraph after eq. 33.5, and Exercise 33.3).  No NaN is produced for it.
 *
 * The result is computed with the sufficient statistics (m, l, u) of eq. 33.3
 * and the merge rule of eqs. 33.4–33.5 (Algorithm 33.1): exact up to rounding
 * order; the T_q x T_k score matrix is never written to memory.
 */
#ifndef BLKATTN_H_
#define BLKATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (cudaStream_t / CUstream); NULL = legacy stream. */
typedef struct CUstream_st* blkattn_stream_t;

/* ---------------------------------------------------------------- status */
enum {
  BLKATTN_OK = 0,
  BLKATTN_ERR_INVALID_ARG = -1,   /* bad shape, dtype, stride, alignment, H_q % H_kv, NULL */
  BLKATTN_ERR_UNSUPPORTED = -2,   /* a valid request the library has no kernel for (e.g. d not in {64,128}) */
  BLKATTN_ERR_CUDA = -3,          /* a CUDA runtime call or kernel launch failed */
  BLKATTN_ERR_DEVICE_TIMEOUT = -4,/* a kernel's bounded wait ran out (reported by blkattn_check_device_error) */
  BLKATTN_ERR_NO_WORKSPACE = -5,  /* the workspace must grow while the stream is being captured */
  BLKATTN_ERR_SCRATCH_LIMIT = -6  /* blkattn_fwd_static_scratch: more scratch needed than it has */
};

/* ---------------------------------------------------------------- tensors */
enum {
  BLKATTN_BF16 = 1,  /* bfloat16 */
  BLKATTN_F32 = 2,   /* IEEE binary32 */
  BLKATTN_I32 = 3,   /* int32 */
  BLKATTN_I64 = 4    /* int64 (token-tree node masks) */
};

/*
 * A strided view.  sizes/strides are in ELEMENTS; a stride of 0 broadcasts.
 * Only the first ndim entries are read.  `device` is the CUDA device ordinal
 * of the memory `data` points to.  Every tensor of one call must name the
 * same device and that device must be current when the call is made;
 * otherwise the call returns BLKATTN_ERR_INVALID_ARG ("Generation and
 * Caching with the Same Model", the cache-reuse forward: cached K/V and the
 * new tokens must be on one device; Chapter 33 §33.3, interface, backend
 * and correctness conditions: the backend follows the device).  A negative
 * ordinal (host memory) is refused the same way.  The library never switches
 * the current device.
 */
typedef struct {
  void* data;
  int32_t dtype;      /* BLKATTN_BF16 | BLKATTN_F32 | BLKATTN_I32 | BLKATTN_I64 */
  int32_t ndim;
  int64_t sizes[4];
  int64_t strides[4];
  int32_t device;     /* CUDA device ordinal holding `data` */
} blkattn_tensor;

/*
 * blkattn_fwd — exact attention of T_q query rows per sequence over a KV cache.
 *
 * q             [B, H_q, T_q, d_h]   bf16 or f32.  Any strides.
 * k             [B, H_kv, T_max, d_h] same dtype as q.  Last stride 1; the
 *               other strides and the base address must be multiples of 16
 *               bytes (rows are moved with bulk asynchronous copies).
 * v             [B, H_kv, T_max, d_v] same dtype and rules as k; d_v == d_h.
 * seqlens_k     [B] int32: valid cache length of each sequence (clamped to
 *               [0, T_max] on the device).
 * q_logical_pos [B, T_q] int32: logical position of each query row (the same
 *               for every head of a sequence).  Negative: no key is visible.
 * mask_bias     NULL, or f32 [B, H_q, T_q, T_max] view; a dim of size 1 or
 *               stride 0 broadcasts (e.g. [B, 1, T_q, T_max] for all heads)
 *               holding the additive M_j of eq. 33.2: finite or -inf.  +inf or
 *               NaN entries are out of contract (the result is then undefined).
 * scale         multiplies q.k (eq. 33.2 uses 1/sqrt(d_h)).
 * out           [B, H_q, T_q, d_v] bf16 or f32, any strides: written.
 * lse           [B, H_q, T_q] f32, any strides: written (natural log).
 * stream        the stream every kernel of the call is enqueued on.
 *
 * Supported: d_h = d_v in {64, 128}; q/k/v all bf16 or all f32.  H_q % H_kv
 * must be 0.  B, T_q >= 0 (0 is a no-op), T_max >= 1.
 * Returns BLKATTN_OK after enqueuing the work (asynchronous), or a negative
 * status without enqueuing anything.  Library-owned scratch (per-split
 * partial states, and per-unit counters that every call leaves at zero)
 * comes from per-device, grow-only buffers.  They grow stream-ordered on the
 * call's stream (cudaFreeAsync of the old buffer, cudaMallocAsync of the
 * new one, counters zeroed by cudaMemsetAsync), so a call never synchronises
 * the device; growth during stream capture is refused with
 * BLKATTN_ERR_NO_WORKSPACE.  Calls on different streams of one device must
 * not overlap in time (they share the buffers): order them with events.
 */
int blkattn_fwd(const blkattn_tensor* q, const blkattn_tensor* k,
                const blkattn_tensor* v, const blkattn_tensor* seqlens_k,
                const blkattn_tensor* q_logical_pos,
                const blkattn_tensor* mask_bias, float scale,
                const blkattn_tensor* out, const blkattn_tensor* lse,
                blkattn_stream_t stream);

/*
 * blkattn_fwd_tree — blkattn_fwd for a token tree of draft rows.
 *
 * "推理加速算法" (inference acceleration algorithms) §7.2.2 Medusa, tree
 * attention verification: a tree of candidate continuations is verified in
 * one pass, every node attending to the cached prefix and to its own
 * ancestors, never to another branch.
 *
 * Arguments as blkattn_fwd, plus
 * tree_mask     int64 [B, T_q], any strides, device (required; T_q <= 64).
 *               The T_q query rows of sequence b are the tree's nodes and
 *               the last T_q cache entries [len_b - T_q, len_b) hold their
 *               keys, node k at key len_b - T_q + k.  Bit k of
 *               tree_mask[b, i] set = row i sees node k (normally its
 *               ancestors and itself).
 * Visibility of key j for row (b, h, i): j < len_b, j <= q_logical_pos[b, i]
 * (pass len_b - 1 to leave the tree region to the mask), the bias is not
 * -inf, and either j < len_b - T_q or bit (j - len_b + T_q) of
 * tree_mask[b, i] is set.  Bits for nodes at or past len_b are ignored.
 * Served by the decode/verify kernels (never the prefill kernel).
 * Returns as blkattn_fwd; BLKATTN_ERR_INVALID_ARG also for a NULL tree_mask,
 * a dtype other than BLKATTN_I64, sizes other than [B, T_q] or T_q > 64.
 */
int blkattn_fwd_tree(const blkattn_tensor* q, const blkattn_tensor* k,
                     const blkattn_tensor* v, const blkattn_tensor* seqlens_k,
                     const blkattn_tensor* q_logical_pos,
                     const blkattn_tensor* tree_mask,
                     const blkattn_tensor* mask_bias, float scale,
                     const blkattn_tensor* out, const blkattn_tensor* lse,
                     blkattn_stream_t stream);

/*
 * blkattn_fwd_window — blkattn_fwd with sliding-window attention.
 *
 * "Chapter 33: inference compute optimisation" §33.7 (the paragraph of
 * eq. 33.16): only the keys of the prescribed range stay visible.
 * Arguments as blkattn_fwd, plus window >= 1: a row at logical position pos
 * sees only keys j with pos - window < j <= pos (the window most recent
 * positions up to its own), on top of the length, position and bias
 * conditions.  The kernels skip the key tiles before their rows' earliest
 * visible key (the tcgen05 decode kernel per unit, the prefill kernel per
 * CTA); the tcgen05 decode kernel takes at most 512 (sequence x row group)
 * units of window calls (more go to the split kernels).  Returns as blkattn_fwd;
 * BLKATTN_ERR_INVALID_ARG also for window < 1 or window > 2^31 - 1.
 */
int blkattn_fwd_window(const blkattn_tensor* q, const blkattn_tensor* k,
                       const blkattn_tensor* v, const blkattn_tensor* seqlens_k,
                       const blkattn_tensor* q_logical_pos, int64_t window,
                       const blkattn_tensor* mask_bias, float scale,
                       const blkattn_tensor* out, const blkattn_tensor* lse,
                       blkattn_stream_t stream);

/*
 * blkattn_spec_sample — one speculative-decoding verification step per
 * sequence ("Chapter 33: inference compute optimisation" §33.5,
 * eqs. 33.10–33.13; §33.6 for the in-order rule).
 *
 * p           f32 [B, k+1, V]: target probabilities after the confirmed
 *             prefix and after each candidate (row k: past all of them);
 *             vocabulary stride 1.
 * q           f32 [B, k, V]: the draft probabilities the candidates were
 *             drawn from; vocabulary stride 1.
 * draft       int32 [B, k]: the candidates x_1..x_k.
 * u_accept    f32 [B, k]: uniforms in [0, 1), one per candidate.
 * u_sample    int32 [B]: one 32-bit uniform integer per sequence (the bits
 *             are read as unsigned).
 * n_accepted  int32 [B], written: candidates kept (0..k).
 * token       int32 [B], written: the token emitted after them.
 * Candidate x_i is kept iff u_i * q_i(x_i) < p_i(x_i) (computed in fp64,
 * exact for fp32 operands), in order, up to the first rejection; then the
 * token is drawn from the residual [p_i - q_i]_+ of that position, or from
 * p_{k+1} when all are kept, by inverse CDF in fixed point (mass: the exact
 * difference p - q of the fp32 values, as eq. 33.12 writes it, or p,
 * clamped to [0, 2]; weight floor(mass * 2^40); integer prefix sums;
 * threshold floor(s * Z / 2^32); the smallest token whose prefix sum
 * exceeds it).  A rejection meeting a zero
 * residual keeps the candidate; a candidate outside [0, V) or with q = 0 is
 * rejected (its position having no residual mass, the token is drawn from
 * p_i); a distribution with no mass at 2^-40 resolution gives token 0.
 * k = 0 is allowed (q, draft, u_accept may then be empty).  The caller owns
 * every buffer; the call enqueues one kernel on the stream and never reads
 * device data on the host.  Returns BLKATTN_OK, BLKATTN_ERR_INVALID_ARG
 * (shapes, dtypes, strides, NULL data, tensors on another device than the
 * current one) or BLKATTN_ERR_CUDA (launch).
 */
int blkattn_spec_sample(const blkattn_tensor* p, const blkattn_tensor* q,
                        const blkattn_tensor* draft, const blkattn_tensor* u_accept,
                        const blkattn_tensor* u_sample, const blkattn_tensor* n_accepted,
                        const blkattn_tensor* token, blkattn_stream_t stream);

/*
 * blkattn_fwd_static_scratch — blkattn_fwd that allocates no device memory.
 *
 * No counterpart on the pages: this is a deployment variant of blkattn_fwd.
 * It is for callers that must not allocate device memory at call time: a
 * host framework that owns every byte of device memory through its own pool
 * or budget, a latency-critical loop that cannot afford the device-wide
 * synchronisation cudaMalloc/cudaFree may bring, or a runtime that forbids
 * dynamic device allocation after start-up.
 *
 * Same arguments, layouts, semantics and results as blkattn_fwd.  The
 * per-split partial states live in one fixed array compiled into the library
 * (BLKATTN_STATIC_SCRATCH_BYTES, 16 MiB, held on every device that loads the
 * library until the process exits) instead of the grow-only workspace; the
 * call makes no cudaMalloc, cudaFree or other allocating call.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - The last 256 KiB of the array hold 32-bit per-unit counters of the
 *     tcgen05 decode kernel (one per sequence x KV head x row group); they
 *     are zero when the library loads and every call leaves them zero.  A
 *     problem whose plan needs more than the remaining 15.75 MiB
 *     (blkattn_debug_plan's workspace_bytes) or more than 65536 units is
 *     rejected with BLKATTN_ERR_SCRATCH_LIMIT before anything is enqueued.
 *   - Every call shares the one array and leaves its contents behind.  Apart
 *     from the counters nothing has to start at zero: each call writes every
 *     partial state it later reads.  Calls whose kernels overlap on the GPU
 *     (concurrent streams, several host threads) race on the array:
 *     serialise them.
 */
#define BLKATTN_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int blkattn_fwd_static_scratch(const blkattn_tensor* q, const blkattn_tensor* k,
                               const blkattn_tensor* v, const blkattn_tensor* seqlens_k,
                               const blkattn_tensor* q_logical_pos,
                               const blkattn_tensor* mask_bias, float scale,
                               const blkattn_tensor* out, const blkattn_tensor* lse,
                               blkattn_stream_t stream);

/*
 * blkattn_bwd — gradients of blkattn_fwd with respect to q, k and v.
 *
 * "Chapter 33: inference compute optimisation" §33.3, eqs. 33.6–33.8: the
 * probabilities are recomputed block by block from the scores and the saved
 * lse (P = exp(S - lse)), never stored; with the upstream gradient g_o,
 *   dv = P^T g_o,  dP = g_o v^T,  dS = P (dP - D),  D_i = g_o,i . o_i,
 *   dq = scale dS k,  dk = scale dS^T q,
 * where `scale` takes the place of eq. 33.8's 1/sqrt(d_h) and D is eq.
 * 33.7's row sum in the form of Exercise 33.4.  Visibility is blkattn_fwd's
 * (length, position, bias); invisible keys and empty rows get no gradient.
 * With grouped heads, dk and dv of a KV head sum over its G query heads.
 *
 *   q, k, v, seqlens_k, q_logical_pos, mask_bias, scale: as for the
 *        blkattn_fwd call whose gradients are wanted (bf16, d_h = 128; q rows
 *        as k/v rows: unit dim stride, 16-byte aligned base and strides)
 *   out  the forward output o [B,H_q,T_q,d] (bf16 or f32, any strides)
 *   lse  the forward lse [B,H_q,T_q] (f32, natural log, -inf = empty row)
 *   dout g_o [B,H_q,T_q,d], bf16, laid out like q
 *   dq   f32 [B,H_q,T_q,d]; dk, dv f32 [B,H_kv,T_max,d]: unit dim stride,
 *        16-byte aligned base and strides.  Every element is written (0 for
 *        cache rows no query sees, including [len, T_max)).
 * The products take P and dS as bf16 operands with fp32 accumulation; the
 * result does not depend on the schedule (no atomics: deterministic).
 * Uses the library's grow-only workspace (D and the base-2 lse per row).
 * Returns as blkattn_fwd; BLKATTN_ERR_UNSUPPORTED for f32, d_h != 128 or
 * T_q > 131072;
 * BLKATTN_ERR_INVALID_ARG also for a non-finite scale or mismatched
 * gradient shapes, dtypes or layouts.
 */
int blkattn_bwd(const blkattn_tensor* q, const blkattn_tensor* k,
                const blkattn_tensor* v, const blkattn_tensor* seqlens_k,
                const blkattn_tensor* q_logical_pos,
                const blkattn_tensor* mask_bias, float scale,
                const blkattn_tensor* out, const blkattn_tensor* lse,
                const blkattn_tensor* dout, const blkattn_tensor* dq,
                const blkattn_tensor* dk, const blkattn_tensor* dv,
                blkattn_stream_t stream);

/*
 * blkattn_bwd_window — blkattn_bwd for a blkattn_fwd_window call: the same
 * arguments plus window >= 1 (keys pos - window < j <= pos, "Chapter 33"
 * §33.7, the paragraph of eq. 33.16).  Each dQ block starts at the key tile
 * of its rows' earliest visible key and each dK/dV block visits only the
 * query tiles whose windows reach it.  Returns as blkattn_bwd;
 * BLKATTN_ERR_INVALID_ARG also for window < 1 or window > 2^31 - 1.
 */
int blkattn_bwd_window(const blkattn_tensor* q, const blkattn_tensor* k,
                       const blkattn_tensor* v, const blkattn_tensor* seqlens_k,
                       const blkattn_tensor* q_logical_pos, int64_t window,
                       const blkattn_tensor* mask_bias, float scale,
                       const blkattn_tensor* out, const blkattn_tensor* lse,
                       const blkattn_tensor* dout, const blkattn_tensor* dq,
                       const blkattn_tensor* dk, const blkattn_tensor* dv,
                       blkattn_stream_t stream);

/*
 * Attention states of rows, in the sufficient statistics of eq. 33.3:
 *   m [rows]           f32, the maximum score (natural-log units); -inf = empty
 *   l [rows]           f32, sum e^{z_j - m}; NULL means "normalised": l = 1 and
 *                      u holds o = u / l (then m is the row's lse, so the
 *                      (out, lse) pair blkattn_fwd writes IS a state)
 *   u [rows, d_v]      f32, sum e^{z_j - m} v_j, row stride u_row_stride elements
 * An empty state (no valid key) is m = -inf; its l and u are not read.
 */
typedef struct {
  float* m;
  float* l;
  float* u;
  int64_t rows;
  int32_t d_v;
  int64_t u_row_stride;
} blkattn_states;

/*
 * blkattn_merge — row-wise merge of two disjoint-key states, eqs. 33.4–33.5
 * (m = max(m_a, m_b); l and u rescaled by e^{m_x - m}), with the valid-flag
 * rule: an empty side contributes nothing and -inf - (-inf) is never formed.
 * out may alias a or b.  If out->l is NULL the result is written normalised
 * (u <- u / l, m <- m + ln l); an empty result is then u = 0, m = -inf.
 * rows and d_v must agree across a, b and out; d_v in [1, 1024].
 * Asynchronous on stream; returns a status as blkattn_fwd does.
 */
int blkattn_merge(const blkattn_states* a, const blkattn_states* b,
                  const blkattn_states* out, blkattn_stream_t stream);

/* Human-readable text for a status code (static storage). */
const char* blkattn_status_string(int status);

/*
 * The CUDA runtime's text for the error behind the calling thread's last
 * BLKATTN_ERR_CUDA (static storage; "no CUDA error recorded" before any).
 */
const char* blkattn_last_cuda_error(void);

/*
 * Test hook: synchronises the stream, then reads and clears the library's
 * device error word.  Returns BLKATTN_OK, BLKATTN_ERR_DEVICE_TIMEOUT when a
 * kernel gave up a bounded wait (the per-unit counters of the current device
 * are then reset to zero, since the kernel that gave up may have left some
 * behind), or BLKATTN_ERR_CUDA if the sync failed.
 */
int blkattn_check_device_error(blkattn_stream_t stream);

/*
 * Host-only view of the split plan blkattn_fwd would use (no CUDA call).
 * Keys [0, T_max) are cut into n_splits consecutive chunks of chunk_keys
 * (the last may be shorter); rows_per_cta query rows of one KV head share a
 * CTA.  kernel: 0 = CUDA-core split-KV kernel (f32 inputs), 1 = warp-level
 * tensor-core split-KV kernel (bf16 inputs), 2 = tcgen05 prefill kernel
 * (bf16, d = 128, T_q >= 64, no bias, scale > 0; the plan shown assumes no
 * bias, a positive scale and 16-byte aligned query rows).
 * Returns BLKATTN_OK or BLKATTN_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t kernel;
  int32_t rows_per_cta;
  int32_t row_groups;     /* CTAs along the query rows of one KV head */
  int32_t chunk_keys;
  int32_t n_splits;
  int32_t tile_keys;      /* keys per pipeline stage */
  int64_t ctas;           /* grid size */
  int64_t workspace_bytes;
} blkattn_plan;

int blkattn_debug_plan(int64_t B, int64_t H_q, int64_t H_kv, int64_t T_q,
                       int64_t T_max, int64_t d, int32_t dtype,
                       int32_t num_sms, blkattn_plan* plan);

/*
 * Measurement hook: when ev is not NULL (a cudaEvent_t of the calling
 * process), every later blkattn_fwd records it on its stream right after the
 * main attention kernel and before the split-merge kernel, so a caller can
 * time the two kernels separately with events on the launch stream.  NULL
 * switches it off.  Process-wide; not for concurrent callers.
 */
void blkattn_debug_set_split_event(void* ev);

/*
 * Test hook of the bounded waits (no counterpart on the pages; it exercises
 * the rule of Chapter 33 §33.2 that undefined values must not propagate, here
 * for a kernel that cannot finish).  After this call, the NEXT launch of the
 * tcgen05 decode kernel (a blkattn_fwd call that blkattn_debug_plan reports
 * as kernel 3) makes the MMA-issuing thread of CTA (cta mod the launch's CTA
 * count) wait on a barrier that nothing completes.  That wait gives up after
 * 1 ms; the thread then issues no product, and the CTA's other roles give up
 * their own bounded waits (2 s each), let the copies they issued land, free
 * tensor memory and return.  The call's output is undefined;
 * blkattn_check_device_error then reports BLKATTN_ERR_DEVICE_TIMEOUT and
 * resets the per-unit counters the stopped CTA left behind, so the next call
 * is correct.  No fault and no unbounded wait is involved.  cta < 0 cancels a
 * pending request.  Process-wide; not for concurrent callers.
 */
void blkattn_debug_stall_next_decode(int32_t cta);

#ifdef __cplusplus
}
#endif

#endif /* BLKATTN_H_ */
