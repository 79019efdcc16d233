"""Sufficient statistics and their merge rule — TEST INFRASTRUCTURE ONLY.

fp64 numpy statement of "Chapter 33: inference compute optimisation" §33.2:

  * eq. 33.3   state of a non-empty valid key set A:
               m_A = max_{j in A} z_j,
               l_A = sum_{j in A} e^{z_j - m_A},
               u_A = sum_{j in A} e^{z_j - m_A} v_j
  * eqs. 33.4–33.5  merge of two disjoint valid sets with m = max(m_A, m_B):
               l = e^{m_A - m} l_A + e^{m_B - m} l_B,
               u = e^{m_A - m} u_A + e^{m_B - m} u_B,  and o = u / l
  * the empty-set rule (the paragraph after eq. 33.5): an empty set is carried
    as an explicit EMPTY marker, the first non-empty block initialises the
    state, and -inf - (-inf) is never evaluated;
  * Algorithm 33.1 (blocked exact attention for one query): start from EMPTY,
    per block score and mask, skip a block with no valid key, merge its state,
    finish with u / l or the defined fully-masked output.

A state is the tuple (m, l, u) with u a 1-D float64 array, or ``EMPTY``.
Only tests may import this module; the CUDA library does not use it.
"""
from __future__ import annotations

import math

import numpy as np

EMPTY = None  # the explicit "no valid key yet" state


def block_state(z, v, valid=None):
    """eq. 33.3 for the valid keys of one block; EMPTY when none is valid.

    z: scores [n]; v: values [n, d_v]; valid: bool [n] or None (all valid).
    """
    z = np.asarray(z, dtype=np.float64).reshape(-1)
    v = np.asarray(v, dtype=np.float64).reshape(z.size, -1)
    keep = np.ones(z.size, bool) if valid is None else np.asarray(valid, bool)
    if not keep.any():
        return EMPTY
    zk = z[keep]
    m = float(zk.max())
    w = np.exp(zk - m)
    return (m, float(w.sum()), (w[:, None] * v[keep]).sum(axis=0))


def merge(a, b):
    """eqs. 33.4–33.5; either argument may be EMPTY (no arithmetic on it)."""
    if a is EMPTY:
        return b
    if b is EMPTY:
        return a
    ma, la, ua = a
    mb, lb, ub = b
    m = max(ma, mb)
    ca = math.exp(ma - m)
    cb = math.exp(mb - m)
    return (m, ca * la + cb * lb, ca * ua + cb * ub)


def finish(state, d_v):
    """o = u / l and lse = m + ln l; the fully-masked row gives (0, -inf)."""
    if state is EMPTY:
        return np.zeros(d_v), -math.inf
    m, l, u = state
    return u / l, m + math.log(l)


def blocked_attention(z, v, valid, blocks):
    """Algorithm 33.1: fold the blocks (lists of key indices, any order) into
    one state with the merge rule, then finish.  Returns (o, lse, state)."""
    z = np.asarray(z, dtype=np.float64).reshape(-1)
    v = np.asarray(v, dtype=np.float64).reshape(z.size, -1)
    valid = np.ones(z.size, bool) if valid is None else np.asarray(valid, bool)
    state = EMPTY
    for idx in blocks:
        idx = np.asarray(idx, dtype=np.int64)
        if idx.size == 0 or not valid[idx].any():
            continue  # a fully masked block contributes nothing
        state = merge(state, block_state(z[idx], v[idx], valid[idx]))
    o, lse = finish(state, v.shape[1])
    return o, lse, state
