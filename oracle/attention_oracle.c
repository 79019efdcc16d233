/*
 * Exact attention oracle — TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, fp64 statement of what the attention path
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header or constant with the CUDA
 * library and must never be reached from the product path.
 *
 * Definition followed ("Chapter 33: inference compute optimisation",
 * §33.2, eq. 33.2): for one query row
 *
 *     z_j = q . k_j / sqrt(d_h) + M_j            (scale passed explicitly)
 *     o   = sum_j e^{z_j} v_j / sum_j e^{z_j}    over the valid keys j
 *
 * The score vector of a row is formed explicitly, key by key; the softmax is
 * evaluated with the usual subtraction of the row maximum (an identity of the
 * quotient, not a blocking); no tiling, splitting or merging happens here.
 *
 * Which keys are valid (readings of the pages, stated once here):
 *   - causal visibility is by LOGICAL position ("Generation and Caching with the
 *     Same Model", the section on cache reuse: new queries after a cache of
 *     length t sit at positions t, t+1, ...; and §33.3 "interface and
 *     correctness conditions" of Chapter 33): key j is visible to a row at
 *     logical position pos iff j <= pos;
 *   - a key must exist in the cache: j < min(seqlen_b, T_max) (seqlen < 0 -> 0);
 *   - an additive bias of -inf masks the key (M_j in eq. 33.2); finite biases
 *     are added after scaling; +inf / NaN biases are out of contract and make
 *     the call return an error;
 *   - a row with no valid key (the empty set of §33.2, the last paragraph
 *     before Example 25.1) gets the defined output out = 0, lse = -inf.
 *   - lse is the natural logarithm of sum_j e^{z_j}.
 *   - token-tree verification ("推理加速算法" (inference acceleration
 *     algorithms) §7.2.2 Medusa, tree attention verification and its figure
 *     of a candidate tree): when a tree is given, the T_q query rows of a
 *     sequence are the nodes of a candidate tree and the last T_q cache
 *     entries [len - T_q, len) hold those nodes' keys, node k at key
 *     len - T_q + k.  A node sees the whole earlier cache and, inside the
 *     tree, only the nodes named in its mask (its ancestors and itself): bit k
 *     of tree[b, i] set = node i sees node k.  The plainest reading of
 *     "verify every candidate path in one pass": no node sees a sibling
 *     branch.  This is one more condition on top of the three above.
 *   - sliding-window attention ("Chapter 33: inference compute
 *     optimisation" §33.7, the paragraph of eq. 33.16: only the keys of
 *     the prescribed range stay visible): with a window of W keys a row at
 *     logical position pos sees only keys j > pos - W, i.e. the W most
 *     recent positions up to its own; another condition on top of the
 *     others.  W = 0 means no window.
 *   - grouped-query heads: query head h reads KV head floor(h / (H_q/H_kv)).
 *
 * Inputs may be float64, float32 or bfloat16 (raw 16-bit patterns); every
 * element is widened exactly to double before use.  Arrays are contiguous,
 * row-major: q [B,H_q,T_q,d_h], k [B,H_kv,T_max,d_h], v [B,H_kv,T_max,d_v],
 * seqlens [B] int32, qpos [B,T_q] int32, bias addressed through four element
 * strides (zero strides broadcast), out [nrows,d_v], lse [nrows].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F64 = 0, OR_F32 = 1, OR_BF16 = 2 };

static double widen(const void* p, int type, int64_t i) {
  if (type == OR_F64) return ((const double*)p)[i];
  if (type == OR_F32) return (double)((const float*)p)[i];
  /* bfloat16: the upper half of an IEEE binary32 pattern */
  uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  int B, Hq, Hkv, Tq, Tmax, dh, dv;
  const void* q; int q_type;
  const void* k; int k_type;
  const void* v; int v_type;
  const int32_t* seqlens;
  const int32_t* qpos;
  const void* bias; int bias_type;  /* may be NULL */
  int64_t bias_stride[4];
  const int64_t* tree;              /* may be NULL: [B, T_q] node masks, T_q <= 64 */
  int64_t window;                   /* 0: none; else keys j > pos - window */
  double scale;
} oracle_problem;

/* One query row, explicit scores (eq. 33.2).  Returns 0, or -2 on a bias that
 * is +inf or NaN.  zbuf has room for T_max doubles. */
static int one_row(const oracle_problem* P, int64_t row, double* zbuf,
                   double* out, double* lse, int32_t* n_vis, int32_t* first,
                   int32_t* last) {
  const int64_t i = row % P->Tq;
  const int64_t h = (row / P->Tq) % P->Hq;
  const int64_t b = row / ((int64_t)P->Tq * P->Hq);
  const int64_t group = P->Hq / P->Hkv;
  const int64_t hk = h / group;
  int64_t len = P->seqlens[b];
  if (len < 0) len = 0;
  if (len > P->Tmax) len = P->Tmax;
  const int64_t pos = P->qpos[b * P->Tq + i];

  const int64_t q_off = ((b * P->Hq + h) * P->Tq + i) * P->dh;
  const int64_t kv_head = (b * P->Hkv + hk) * (int64_t)P->Tmax;

  /* explicit score vector: z_j for every key, -inf where the key is invalid */
  double m = -INFINITY;
  int32_t count = 0, fst = -1, lst = -1;
  for (int64_t j = 0; j < P->Tmax; ++j) {
    zbuf[j] = -INFINITY;
    if (!(j < len && j <= pos)) continue;
    if (P->window > 0 && j <= pos - P->window) continue; /* outside the window */
    if (P->tree) {
      const int64_t base = len - P->Tq; /* key of tree node 0 */
      if (j >= base) {
        const int64_t node = j - base;  /* 0 <= node < T_q because j < len */
        if (!((((uint64_t)P->tree[b * P->Tq + i]) >> node) & 1u)) continue;
      }
    }
    double bias = 0.0;
    if (P->bias) {
      const int64_t bi = b * P->bias_stride[0] + h * P->bias_stride[1] +
                         i * P->bias_stride[2] + j * P->bias_stride[3];
      bias = widen(P->bias, P->bias_type, bi);
      if (isnan(bias) || bias == INFINITY) return -2;
      if (bias == -INFINITY) continue; /* masked by M_j */
    }
    double dot = 0.0;
    for (int t = 0; t < P->dh; ++t)
      dot += widen(P->q, P->q_type, q_off + t) *
             widen(P->k, P->k_type, (kv_head + j) * P->dh + t);
    const double z = P->scale * dot + bias;
    zbuf[j] = z;
    if (z > m) m = z;
    if (fst < 0) fst = (int32_t)j;
    lst = (int32_t)j;
    ++count;
  }
  *n_vis = count;
  *first = fst;
  *last = lst;
  if (count == 0) { /* no valid key: the defined output */
    for (int t = 0; t < P->dv; ++t) out[t] = 0.0;
    *lse = -INFINITY;
    return 0;
  }
  double denom = 0.0;
  for (int t = 0; t < P->dv; ++t) out[t] = 0.0;
  for (int64_t j = 0; j < P->Tmax; ++j) {
    if (zbuf[j] == -INFINITY) continue;
    const double w = exp(zbuf[j] - m);
    denom += w;
    for (int t = 0; t < P->dv; ++t)
      out[t] += w * widen(P->v, P->v_type, (kv_head + j) * P->dv + t);
  }
  for (int t = 0; t < P->dv; ++t) out[t] /= denom;
  *lse = m + log(denom);
  return 0;
}

/*
 * oracle_attention: rows == NULL means every row 0..B*H_q*T_q-1 in order;
 * otherwise the flattened row ids ((b*H_q + h)*T_q + i) listed in rows.
 * Integer outputs (may be NULL): visible-key count, first and last visible
 * key index (-1 when none).  nthreads <= 0 uses the OpenMP default.
 * Returns 0, -1 on bad sizes, -2 on an out-of-contract bias, -3 on no memory.
 */
int oracle_attention_masks(int B, int Hq, int Hkv, int Tq, int Tmax, int dh, int dv,
                           const void* q, int q_type, const void* k, int k_type,
                           const void* v, int v_type, const int32_t* seqlens,
                           const int32_t* qpos, const void* bias, int bias_type,
                           const int64_t* bias_stride, const int64_t* tree,
                           int64_t window, double scale, const int64_t* rows,
                           int64_t nrows, double* out, double* lse,
                           int32_t* n_vis, int32_t* first, int32_t* last,
                           int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Tq < 0 || Tmax < 0 || dh <= 0 ||
      dv <= 0 || Hq % Hkv != 0 || (tree && Tq > 64) || window < 0)
    return -1;
  oracle_problem P;
  memset(&P, 0, sizeof P);
  P.B = B; P.Hq = Hq; P.Hkv = Hkv; P.Tq = Tq; P.Tmax = Tmax; P.dh = dh;
  P.dv = dv; P.q = q; P.q_type = q_type; P.k = k; P.k_type = k_type;
  P.v = v; P.v_type = v_type; P.seqlens = seqlens; P.qpos = qpos;
  P.bias = bias; P.bias_type = bias_type; P.scale = scale; P.tree = tree;
  P.window = window;
  if (bias)
    for (int s = 0; s < 4; ++s) P.bias_stride[s] = bias_stride[s];
  const int64_t total = (int64_t)B * Hq * Tq;
  if (rows == NULL) nrows = total;
  for (int64_t r = 0; rows && r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -1;

  int status = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
  {
    double* zbuf = (double*)malloc(sizeof(double) * (size_t)(Tmax > 0 ? Tmax : 1));
    int32_t nv, fs, ls;
    /* every thread enters the work-sharing loop, even without a buffer */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
      const int64_t row = rows ? rows[r] : r;
      int rc = -3;
      nv = 0; fs = -1; ls = -1;
      if (zbuf) rc = one_row(&P, row, zbuf, out + r * dv, lse + r, &nv, &fs, &ls);
      if (rc != 0) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
        status = rc;
      }
      if (n_vis) n_vis[r] = nv;
      if (first) first[r] = fs;
      if (last) last[r] = ls;
    }
    free(zbuf);
  }
  return status;
}

/* The same with a tree and no window. */
int oracle_attention_tree(int B, int Hq, int Hkv, int Tq, int Tmax, int dh, int dv,
                          const void* q, int q_type, const void* k, int k_type,
                          const void* v, int v_type, const int32_t* seqlens,
                          const int32_t* qpos, const void* bias, int bias_type,
                          const int64_t* bias_stride, const int64_t* tree,
                          double scale, const int64_t* rows, int64_t nrows,
                          double* out, double* lse, int32_t* n_vis,
                          int32_t* first, int32_t* last, int nthreads) {
  return oracle_attention_masks(B, Hq, Hkv, Tq, Tmax, dh, dv, q, q_type, k, k_type, v, v_type,
                                seqlens, qpos, bias, bias_type, bias_stride, tree, 0, scale,
                                rows, nrows, out, lse, n_vis, first, last, nthreads);
}

/* The same without a tree. */
int oracle_attention(int B, int Hq, int Hkv, int Tq, int Tmax, int dh, int dv,
                     const void* q, int q_type, const void* k, int k_type,
                     const void* v, int v_type, const int32_t* seqlens,
                     const int32_t* qpos, const void* bias, int bias_type,
                     const int64_t* bias_stride, double scale,
                     const int64_t* rows, int64_t nrows, double* out,
                     double* lse, int32_t* n_vis, int32_t* first,
                     int32_t* last, int nthreads) {
  return oracle_attention_tree(B, Hq, Hkv, Tq, Tmax, dh, dv, q, q_type, k, k_type, v, v_type,
                               seqlens, qpos, bias, bias_type, bias_stride, NULL, scale, rows,
                               nrows, out, lse, n_vis, first, last, nthreads);
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
