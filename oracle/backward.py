"""Attention backward pass — TEST INFRASTRUCTURE ONLY.

Plain numpy fp64 statement of the gradients of "Chapter 33: inference compute
optimisation" §33.3 (the paragraph on block size, parallelism and
recomputation, eqs. 33.6–33.8, and Exercise 33.4).  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import it; it
shares no code with the CUDA library.

With P = softmax(S) over the visible keys of each row, O = P V and upstream
gradient G_O:

  G_V = P^T G_O,  G_P = G_O V^T                               eq. 33.6
  (G_S)_ij = P_ij [ (G_P)_ij - sum_k P_ik (G_P)_ik ]          eq. 33.7
  G_Q = scale * G_S K,  G_K = scale * G_S^T Q                 eq. 33.8

S_ij = scale * q_i . k_j + M_ij on the visible keys; the pages write 1/sqrt(d_h)
where the interface takes `scale`, and eq. 33.8's 1/sqrt(d_h) is the same
factor.  Visibility is the forward's: key j is visible to row (b, h, i) iff
j < len_b, j <= pos[b, i] and M[b, h, i, j] != -inf, and, with a sliding
window of W keys (§33.7, the paragraph of eq. 33.16), j > pos[b, i] - W.  Invisible keys have
P = 0 and take no gradient; a row with no visible key has P = 0 everywhere
(its forward output is the defined 0) and contributes nothing.  Grouped
query attention: query head h reads KV head h // G, so G_K and G_V of a KV
head sum the contributions of its G query heads.

The row sum in eq. 33.7 is taken literally (sum of P G_P over the row);
Exercise 33.4's solution identifies it with g_o . o, which the tests check
separately.  Rows are processed in chunks of query rows only to bound memory:
each row's arithmetic is the definition above, and a chunk boundary only
splits the fp64 sums of G_K and G_V over rows.

Besides the gradients the function returns, per element, the sum of the
absolute values of the terms a computation with bf16-rounded P and G_S
operands and fp32 accumulation adds up (the scale of its rounding error):
  dv_abs = P^T |G_O|
  dq_abs = scale * E |K|,  dk_abs = scale * E^T |Q|,
  E_ij = |G_S,ij| + 2^-8 P_ij (sum_t |G_O,it| |V_jt| + sum_t |G_O,it| |O_it|)
(the second part of E bounds the fp32 cancellation in G_P - D).
"""
from __future__ import annotations

import numpy as np

_CHUNK = 1024  # query rows per chunk


def _f64(x):
    """fp64 numpy copy of a CPU array or tensor (bf16 widened exactly)."""
    if hasattr(x, "detach"):
        import torch
        t = x.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle inputs must live on the CPU")
        return t.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def attention_backward(q, k, v, seqlens, qpos, scale, dout, bias=None, units=None,
                       with_abs: bool = True, window: int = 0):
    """Gradients of exact attention (eqs. 33.6–33.8) in fp64.

    q [B,H_q,T_q,d], k, v [B,H_kv,T_max,d], seqlens int [B], qpos int [B,T_q],
    dout [B,H_q,T_q,d] (the upstream gradient G_O), bias None or broadcastable
    to [B,H_q,T_q,T_max] (finite or -inf).  units: None for every (b, kv head),
    else a list of (b, kv_head) pairs to compute (the others stay zero).
    window: 0, or W > 0 for sliding-window visibility.

    Returns dict(dq [B,H_q,T_q,d], dk, dv [B,H_kv,T_max,d], o [B,H_q,T_q,d],
    lse [B,H_q,T_q] (natural log, -inf for rows with no visible key),
    D [B,H_q,T_q] (the row sums of eq. 33.7), and with with_abs the error
    scales dq_abs, dk_abs, dv_abs of the same shapes).
    """
    Q, K, V, GO = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Tq, d = Q.shape
    Hkv, Tmax = K.shape[1], K.shape[2]
    G = Hq // Hkv
    sl = np.asarray(_f64(seqlens), dtype=np.int64).reshape(B)
    qp = np.asarray(_f64(qpos), dtype=np.int64).reshape(B, Tq)
    Mb = None if bias is None else np.broadcast_to(_f64(bias), (B, Hq, Tq, Tmax))

    out = {name: np.zeros_like(Q) for name in ("dq", "o")}
    out.update({name: np.zeros_like(K) for name in ("dk", "dv")})
    out["lse"] = np.full((B, Hq, Tq), -np.inf)
    out["D"] = np.zeros((B, Hq, Tq))
    if with_abs:
        out.update({"dq_abs": np.zeros_like(Q), "dk_abs": np.zeros_like(K), "dv_abs": np.zeros_like(K)})
    todo = [(b, hk) for b in range(B) for hk in range(Hkv)] if units is None else list(units)
    keys = np.arange(Tmax)
    for b, hk in todo:
        length = min(max(int(sl[b]), 0), Tmax)
        Kb, Vb = K[b, hk], V[b, hk]
        for h in range(hk * G, (hk + 1) * G):
            for r0 in range(0, Tq, _CHUNK):
                r1 = min(r0 + _CHUNK, Tq)
                Qh, GOh = Q[b, h, r0:r1], GO[b, h, r0:r1]
                # visibility (the forward's rule)
                vis = (keys[None, :] < length) & (keys[None, :] <= qp[b, r0:r1, None])
                if window > 0:
                    vis &= keys[None, :] > qp[b, r0:r1, None] - window
                S = scale * (Qh @ Kb.T)
                if Mb is not None:
                    Mh = Mb[b, h, r0:r1]
                    vis &= ~np.isneginf(Mh)
                    S = S + np.where(vis, Mh, 0.0)
                S = np.where(vis, S, -np.inf)
                any_vis = vis.any(axis=1)
                m = np.where(any_vis, S.max(axis=1, initial=-np.inf), 0.0)
                W = np.where(vis, np.exp(S - m[:, None]), 0.0)
                ell = W.sum(axis=1)
                P = np.divide(W, ell[:, None], out=np.zeros_like(W), where=any_vis[:, None])
                O = P @ Vb
                GP = GOh @ Vb.T                                    # eq. 33.6
                D = (P * GP).sum(axis=1)                           # eq. 33.7, the row sum
                GS = P * (GP - D[:, None])                         # eq. 33.7
                out["dq"][b, h, r0:r1] = scale * (GS @ Kb)         # eq. 33.8
                out["dk"][b, hk] += scale * (GS.T @ Qh)            # eq. 33.8
                out["dv"][b, hk] += P.T @ GOh                      # eq. 33.6
                out["o"][b, h, r0:r1] = O
                out["lse"][b, h, r0:r1] = np.where(any_vis, m + np.log(np.where(any_vis, ell, 1.0)), -np.inf)
                out["D"][b, h, r0:r1] = D
                if with_abs:
                    A = np.abs(GOh) @ np.abs(Vb).T
                    Bo = (np.abs(GOh) * np.abs(O)).sum(axis=1)
                    E = np.abs(GS) + 2.0 ** -8 * P * (A + Bo[:, None])
                    out["dq_abs"][b, h, r0:r1] = scale * (E @ np.abs(Kb))
                    out["dk_abs"][b, hk] += scale * (E.T @ np.abs(Qh))
                    out["dv_abs"][b, hk] += P.T @ np.abs(GOh)
    return out
