"""Speculative-sampling acceptance and residual sampling — TEST INFRASTRUCTURE ONLY.

Plain numpy statement of "Chapter 33: inference compute optimisation" §33.5
(eqs. 33.10–33.13) and the in-order rule of §33.6.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import it; it
shares no code with the CUDA library.

Distributions (fp64, the formulas as printed):
  a(x)  = min(1, p(x)/q(x))                      eq. 33.10 (q(x) > 0)
  A     = sum_x min(p(x), q(x)) = 1 - TV(p, q)   eq. 33.11
  r(x)  = [p(x) - q(x)]_+ / Z,  Z = 1 - A        eq. 33.12 (not formed when Z = 0)
  out   = min(p, q) + Z r = p                    eq. 33.13

One verification step (the integer decisions the kernel must reproduce):
  candidates x_1..x_k are taken in order; x_i is accepted iff
  u_i * q_i(x_i) < p_i(x_i), evaluated in fp64 (exact for fp32 inputs:
  a 24-bit by 24-bit product), which is u_i < a(x_i) for u_i in [0, 1).
  At the first rejection the emitted token is drawn from the residual of
  that position; if every candidate is accepted it is drawn from the next
  target distribution p_{k+1}.  The draw is an inverse CDF in fixed point:
  the mass of x is m = p(x) - q(x) for a residual, the EXACT difference of
  the two fp32 values as eq. 33.12 writes it (no rounding), or p(x) for a
  target; it is clamped to [0, 2] and becomes the weight
  F(m) = floor(m * 2^40); integer prefix sums C, Z_int = C(V-1),
  threshold T = floor(s * Z_int / 2^32) for the 32-bit uniform integer s, and
  the token is the smallest x with C(x) > T.  Integer sums make the choice
  independent of summation order.  When a rejection meets a zero residual
  (Z_int = 0, which eq. 33.12 leaves unformed: rejection then has probability
  zero) the candidate is accepted instead.  A candidate with q_i(x_i) = 0, or
  outside the vocabulary, cannot have been proposed; it is rejected, and if
  its position has no residual mass either the token is drawn from p_i
  itself (p = q there).  A distribution with no mass at 2^-40 resolution
  (not a distribution) gives token 0.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

FIX_BITS = 40  # fractional bits of the fixed-point weights


def acceptance(p, q):
    """Eqs. 33.10–33.13 for one pair of distributions (1-D arrays, fp64).
    Returns dict(a, accepted_mass, A, Z, residual (None when Z == 0), out)."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    a = np.where(q > 0, np.minimum(1.0, np.divide(p, q, out=np.zeros_like(p), where=q > 0)), 0.0)
    accepted = np.minimum(p, q)                  # q(x) a(x)
    A = float(accepted.sum())                    # eq. 33.11, first form
    pos = np.maximum(p - q, 0.0)
    Z = float(pos.sum())                         # equals 1 - A when both sum to 1
    residual = None if Z == 0.0 else pos / Z     # eq. 33.12
    out = accepted + (0.0 if residual is None else Z * residual)  # eq. 33.13
    return {"a": a, "accepted_mass": accepted, "A": A, "Z": Z, "residual": residual, "out": out}


def fixed(m) -> np.ndarray:
    """F(m) = floor(clamp(m, 0, 2) * 2^40) (int64) of fp64 masses, exact:
    scaling by a power of two only moves the exponent (NaN counts as 0, like
    a min/max that skips NaN)."""
    m = np.fmin(np.fmax(np.asarray(m, dtype=np.float64), 0.0), 2.0)
    return np.floor(m * float(1 << FIX_BITS)).astype(np.int64)


def fixed_exact(m: Fraction) -> int:
    """F(m) for an exact rational mass."""
    m = min(max(m, Fraction(0)), Fraction(2))
    return math.floor(m * (1 << FIX_BITS))


def weights(p_row, q_row=None) -> np.ndarray:
    """Fixed-point weights F([p - q]_+) of eq. 33.12's residual, with p - q
    the exact difference of the fp32 values, or F(p) of a target row.

    A nonzero fp32 value has all its bits between 2^(e-24) and 2^(e-1), e its
    binary exponent (np.frexp), so the difference of two finite fp32 values
    needs at most |e_p - e_q| + 25 bits: an fp64 subtraction is exact when the
    exponents are at most 28 apart (or either value is 0).  The other entries
    are subtracted as rationals."""
    p = np.asarray(p_row, dtype=np.float32).astype(np.float64)
    if q_row is None:
        return fixed(p)
    q = np.asarray(q_row, dtype=np.float32).astype(np.float64)
    with np.errstate(invalid="ignore"):  # inf - inf is NaN, which F counts as 0
        w = fixed(p - q)
    _, ep = np.frexp(p)
    _, eq = np.frexp(q)
    wide = np.isfinite(p) & np.isfinite(q) & (p != 0) & (q != 0) & (np.abs(ep - eq) > 28)
    for x in np.flatnonzero(wide):
        w.flat[x] = fixed_exact(Fraction(float(p.flat[x])) - Fraction(float(q.flat[x])))
    return w


def inverse_cdf(w: np.ndarray, s: int) -> int:
    """Smallest x with C(x) > floor(s * Z / 2^32), C the prefix sums of w."""
    Z = int(w.sum())
    T = (int(s) * Z) >> 32
    c = 0
    for x, wx in enumerate(w.tolist()):
        c += int(wx)
        if c > T:
            return x
    raise ValueError("empty distribution")


def verify_step(p, q, draft, u_accept, u_sample):
    """One speculative verification step per row.

    p float32 [B, k+1, V] target probabilities, q float32 [B, k, V] draft
    probabilities, draft int32 [B, k] candidates, u_accept float32 [B, k] in
    [0, 1), u_sample uint32 [B].  Returns (n_accepted int32 [B], token
    int32 [B]): the number of candidates kept and the token emitted after them.
    """
    p = np.asarray(p, dtype=np.float32)
    q = np.asarray(q, dtype=np.float32)
    draft = np.asarray(draft, dtype=np.int64)
    u_accept = np.asarray(u_accept, dtype=np.float32)
    u_sample = np.asarray(u_sample, dtype=np.uint64)
    B, k1, V = p.shape
    k = k1 - 1
    n_acc = np.zeros(B, dtype=np.int32)
    token = np.zeros(B, dtype=np.int32)
    for b in range(B):
        chosen = None
        i = 0
        while i < k:
            x = int(draft[b, i])
            if x < 0 or x >= V:  # cannot have been proposed
                px = qx = 0.0
            else:
                px = float(p[b, i, x])
                qx = float(q[b, i, x])
            valid = qx > 0.0
            if valid and float(u_accept[b, i]) * qx < px:
                i += 1
                continue
            # rejected: the residual of position i
            w = weights(p[b, i], q[b, i])
            if int(w.sum()) == 0:
                if valid:  # rejection has probability zero here: keep the candidate
                    i += 1
                    continue
                # an impossible candidate and no residual (p = q here): the target itself
                w = weights(p[b, i])
                chosen = inverse_cdf(w, int(u_sample[b])) if int(w.sum()) > 0 else 0
                break
            chosen = inverse_cdf(w, int(u_sample[b]))
            break
        if chosen is None:  # every candidate kept: the next target distribution
            w = weights(p[b, k])
            # no mass at 2^-40 resolution (not a distribution): token 0 by definition
            chosen = inverse_cdf(w, int(u_sample[b])) if int(w.sum()) > 0 else 0
        n_acc[b] = i
        token[b] = chosen
    return n_acc, token
