"""Exact-attention oracle — TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 CPU statement of what the attention path computes, written
from "Chapter 33: inference compute optimisation" §33.2 (eqs. 33.2–33.5,
Example 25.1, Algorithm 33.1) and from "Generation and Caching with the Same
Model" (logical-position alignment of cached decoding).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library in
``exact_blocked_attention_gb300`` and neither imports the other.

Contents
  attention(...)   explicit eq. 33.2 per row (C, fp64, OpenMP), plus the
                   integer facts per row: visible-key count, first and last
                   visible key.  Pinned by tests/test_oracle_pins.py against
                   Example 25.1, exact rational brute force, closed forms and
                   the cache-alignment example.  Optional token-tree
                   visibility ("推理加速算法" §7.2.2 Medusa, tree attention
                   verification), pinned by brute force over random trees;
                   optional sliding window (§33.7), pinned by the bound of
                   eq. 33.16 and by brute force.
  states           the sufficient statistics (m, l, u) of eq. 33.3, the merge
                   rule of eqs. 33.4–33.5 and Algorithm 33.1, in numpy fp64.
  spec_sampling    speculative-sampling acceptance and residual sampling
                   (§33.5 eqs. 33.10–33.13, the in-order rule of §33.6),
                   pinned by tests/test_spec_sampling_pins.py against
                   Example 25.2 and Exercises 33.7 and 33.9.
  backward         the gradients of eqs. 33.6–33.8 (§33.3) in numpy fp64,
                   pinned by tests/test_backward_pins.py against finite
                   differences of attention(), fp64 autograd of a separate
                   dense formulation, Exercise 33.4's row-sum identity and
                   closed forms.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

F64, F32, BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (fp64, no fast-math, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_attention.restype = I
            lib.oracle_attention.argtypes = [
                I, I, I, I, I, I, I,          # B Hq Hkv Tq Tmax dh dv
                P, I, P, I, P, I,             # q k v (+types)
                P, P,                         # seqlens qpos
                P, I, P,                      # bias, type, strides
                ctypes.c_double,              # scale
                P, ctypes.c_int64,            # rows, nrows
                P, P, P, P, P,                # out lse n_vis first last
                I]                            # nthreads
            lib.oracle_attention_masks.restype = I
            lib.oracle_attention_masks.argtypes = [
                I, I, I, I, I, I, I,          # B Hq Hkv Tq Tmax dh dv
                P, I, P, I, P, I,             # q k v (+types)
                P, P,                         # seqlens qpos
                P, I, P,                      # bias, type, strides
                P, ctypes.c_int64,            # tree masks, window
                ctypes.c_double,              # scale
                P, ctypes.c_int64,            # rows, nrows
                P, P, P, P, P,                # out lse n_vis first last
                I]                            # nthreads
            lib.oracle_attention_tree.restype = I
            lib.oracle_attention_tree.argtypes = [
                I, I, I, I, I, I, I,          # B Hq Hkv Tq Tmax dh dv
                P, I, P, I, P, I,             # q k v (+types)
                P, P,                         # seqlens qpos
                P, I, P,                      # bias, type, strides
                P,                            # tree masks int64 [B, T_q]
                ctypes.c_double,              # scale
                P, ctypes.c_int64,            # rows, nrows
                P, P, P, P, P,                # out lse n_vis first last
                I]                            # nthreads
            lib.oracle_max_threads.restype = I
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_array(x):
    """numpy view of a CPU array or CPU torch tensor (no copy when contiguous)."""
    if hasattr(x, "detach"):  # torch tensor, CPU only
        import torch
        t = x.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle inputs must live on the CPU")
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), BF16
        if t.dtype == torch.float32:
            return t.numpy(), F32
        if t.dtype == torch.float64:
            return t.numpy(), F64
        if t.dtype == torch.int32:
            return t.numpy(), None
        raise TypeError(f"unsupported oracle dtype {t.dtype}")
    a = np.ascontiguousarray(x)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.int32:
        return a, None
    raise TypeError(f"unsupported oracle dtype {a.dtype}")


def attention(q, k, v, seqlens, qpos, scale, bias=None, rows=None,
              nthreads: int = 0, tree=None, window: int = 0):
    """Explicit exact attention (eq. 33.2), one row at a time, in fp64.

    q [B,H_q,T_q,d_h], k [B,H_kv,T_max,d_h], v [B,H_kv,T_max,d_v] (float64,
    float32 or bfloat16; bf16 is widened exactly), seqlens int32 [B], qpos
    int32 [B,T_q] (logical position of each query row), bias None or any
    array/tensor broadcastable to [B,H_q,T_q,T_max] (values finite or -inf).
    rows: None for all rows, or flattened row ids (b*H_q + h)*T_q + i.
    tree: None, or int64 [B,T_q] node masks of a candidate token tree whose
    nodes' keys are the last T_q cache entries of each sequence (bit k of
    tree[b,i] set = row i sees tree node k; T_q <= 64).
    window: 0, or W > 0 for sliding-window attention (a row at position pos
    sees only keys j > pos - W).

    Returns dict(out [n,d_v] f64, lse [n] f64, n_visible, first, last int32 [n]).
    """
    lib = _load()
    qa, qt = _as_array(q)
    ka, kt = _as_array(k)
    va, vt = _as_array(v)
    B, Hq, Tq, dh = qa.shape
    Bk, Hkv, Tmax, dhk = ka.shape
    dv = va.shape[3]
    if Bk != B or dhk != dh or va.shape[:3] != ka.shape[:3]:
        raise ValueError("shape mismatch between q, k, v")
    sl, _ = _as_array(seqlens)
    qp, _ = _as_array(qpos)
    sl = np.ascontiguousarray(sl, dtype=np.int32).reshape(B)
    qp = np.ascontiguousarray(qp, dtype=np.int32).reshape(B, Tq)
    bias_ptr, bias_type, strides = None, 0, None
    keep = []
    if bias is not None:
        if hasattr(bias, "detach"):
            import torch
            bt = bias.detach()
            if bt.device.type != "cpu":
                raise ValueError("oracle inputs must live on the CPU")
            if bt.dtype not in (torch.float32, torch.float64):
                bt = bt.float()
            bias = bt.numpy()  # keeps zero (broadcast) strides
        ba = np.asarray(bias)
        if ba.dtype not in (np.float32, np.float64):
            ba = ba.astype(np.float64)
        ba = np.broadcast_to(ba, (B, Hq, Tq, Tmax))
        bias_type = F32 if ba.dtype == np.float32 else F64
        strides = np.array([s // ba.itemsize for s in ba.strides], dtype=np.int64)
        keep.append(ba)
        bias_ptr = ba.ctypes.data
    if rows is None:
        rows_arr = None
        n = B * Hq * Tq
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        n = rows_arr.size
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    nvis = np.zeros(n, dtype=np.int32)
    first = np.zeros(n, dtype=np.int32)
    last = np.zeros(n, dtype=np.int32)
    tr = None
    if tree is not None:
        tr = np.asarray(tree.detach().cpu().numpy() if hasattr(tree, "detach") else tree)
        tr = np.ascontiguousarray(tr.astype(np.int64, copy=False)).reshape(B, Tq)
    P = lambda a: None if a is None else a.ctypes.data
    rc = lib.oracle_attention_masks(
        B, Hq, Hkv, Tq, Tmax, dh, dv,
        P(qa), qt, P(ka), kt, P(va), vt,
        P(sl), P(qp),
        bias_ptr, bias_type, P(strides),
        P(tr), int(window),
        float(scale),
        P(rows_arr), int(n),
        P(out), P(lse), P(nvis), P(first), P(last),
        int(nthreads))
    del keep
    if rc == -2:
        raise ValueError("bias holds +inf or NaN on a visible key (out of contract)")
    if rc != 0:
        raise ValueError(f"oracle_attention failed with status {rc}")
    return {"out": out, "lse": lse, "n_visible": nvis, "first": first, "last": last}
