"""Pins of the speculative-sampling oracle (oracle/spec_sampling.py) against
"Chapter 33: inference compute optimisation" §33.5: the printed Example 25.2
and Exercises 33.7 and 33.9, the identities of eqs. 33.11 and 33.13, and the
exact boundaries of the fixed-point inverse CDF."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import spec_sampling as ss

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "speculative_sampling.json")


def frac(x):
    return float(Fraction(x))


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["example_25_2", "exercise_33_7"])
def test_printed_examples(name):
    g = golden()[name]
    r = ss.acceptance(g["p"], g["q"])
    np.testing.assert_allclose(r["a"], [frac(x) for x in g["acceptance_probabilities"]], atol=1e-15)
    np.testing.assert_allclose(r["accepted_mass"], [frac(x) for x in g["accepted_mass"]], atol=1e-15)
    assert r["A"] == pytest.approx(frac(g["total_acceptance"]), abs=1e-15)
    np.testing.assert_allclose(r["Z"] * r["residual"], [frac(x) for x in g["positive_residual"]], atol=1e-15)
    np.testing.assert_allclose(r["out"], [frac(x) for x in g["final"]], atol=1e-15)
    np.testing.assert_allclose(r["out"], g["p"], atol=1e-15)  # eq. 33.13


def test_example_25_2_residual_and_wrong_branch():
    g = golden()["example_25_2"]
    r = ss.acceptance(g["p"], g["q"])
    assert r["Z"] == pytest.approx(frac(g["rejection_mass"]), abs=1e-15)
    np.testing.assert_allclose(r["residual"], [frac(x) for x in g["residual_distribution"]], atol=1e-15)
    # negative control: resampling from p after a rejection changes the target
    wrong = r["accepted_mass"] + r["Z"] * np.asarray(g["p"])
    np.testing.assert_allclose(wrong, [frac(x) for x in g["wrong_branch_resample_from_p"]], atol=1e-15)
    assert not np.allclose(wrong, g["p"])
    # after a rejection the first token is certain, whatever the 32-bit draw
    p = np.array(g["p"], dtype=np.float32)[None, None, :].repeat(2, axis=1)
    q = np.array(g["q"], dtype=np.float32)[None, None, :]
    for s in (0, 1, 2**31, 2**32 - 1):
        n, tok = ss.verify_step(p, q, [[1]], [[0.99]], [s])  # 0.99 * 0.5 >= 0.3: rejected
        assert n[0] == 0 and tok[0] == 0


def test_exercise_33_9_temperatures():
    g = golden()["exercise_33_9"]
    logits = np.array([math.log(4.0), 0.0])
    softmax = lambda z: np.exp(z - z.max()) / np.exp(z - z.max()).sum()
    p = softmax(logits / g["target_temperature"])
    q = softmax(logits / g["draft_temperature"])
    np.testing.assert_allclose(p, [frac(x) for x in g["p"]], atol=1e-15)
    np.testing.assert_allclose(q, [frac(x) for x in g["q"]], atol=1e-15)
    r = ss.acceptance(p, q)
    np.testing.assert_allclose(r["a"], [frac(x) for x in g["acceptance_probabilities"]], atol=1e-15)
    np.testing.assert_allclose(r["accepted_mass"], [frac(x) for x in g["accepted_mass"]], atol=1e-15)
    assert r["Z"] == pytest.approx(frac(g["rejection_mass"]), abs=1e-15)
    np.testing.assert_allclose(r["out"], [frac(x) for x in g["final"]], atol=1e-15)


def test_acceptance_is_one_minus_total_variation():
    rng = np.random.default_rng(3)
    for _ in range(20):
        p = rng.dirichlet(np.ones(50)); q = rng.dirichlet(np.ones(50) * 0.3)
        r = ss.acceptance(p, q)
        assert r["A"] == pytest.approx(1 - 0.5 * np.abs(p - q).sum(), abs=1e-14)   # eq. 33.11
        assert r["Z"] == pytest.approx(1 - r["A"], abs=1e-14)
        np.testing.assert_allclose(r["out"], p, atol=1e-14)                         # eq. 33.13


def test_zero_residual_is_not_formed():
    r = ss.acceptance([0.25, 0.75], [0.25, 0.75])
    assert r["Z"] == 0.0 and r["residual"] is None
    np.testing.assert_allclose(r["out"], [0.25, 0.75])


def test_inverse_cdf_boundaries_are_exact():
    """Draw s maps to x iff C(x-1) 2^32 <= s Z < C(x) 2^32: check both sides
    of every boundary, and that each token's share of the 2^32 draws is its
    weight's share of Z to within one draw."""
    rng = np.random.default_rng(4)
    for _ in range(10):
        w = rng.integers(0, 2**38, size=12, dtype=np.int64)
        w[rng.integers(0, 12, size=3)] = 0
        Z = int(w.sum())
        C = np.cumsum(w).tolist()
        starts = [0]
        for c in C:
            starts.append(-(-c * 2**32 // Z))  # ceil(c 2^32 / Z)
        for x in range(12):
            count = starts[x + 1] - starts[x]
            assert abs(count - int(w[x]) * 2**32 / Z) < 1.0
            if count == 0:
                assert w[x] == 0 or count == 0
                continue
            assert ss.inverse_cdf(w, starts[x]) == x
            assert ss.inverse_cdf(w, starts[x + 1] - 1) == x
            if starts[x] > 0:
                assert ss.inverse_cdf(w, starts[x] - 1) < x


def test_acceptance_boundary_in_fp32():
    """u * q(x) < p(x) in fp64 from fp32 operands: the decision flips exactly
    between adjacent fp32 u around p/q."""
    p = np.array([[[0.3, 0.7], [0.5, 0.5]]], dtype=np.float32)
    q = np.array([[[0.45, 0.55]]], dtype=np.float32)
    ratio = float(p[0, 0, 0]) / float(q[0, 0, 0])
    u_hi = np.float32(ratio)
    while float(u_hi) * float(q[0, 0, 0]) < float(p[0, 0, 0]):
        u_hi = np.nextafter(u_hi, np.float32(1))
    u_lo = np.nextafter(u_hi, np.float32(0))
    n_lo, _ = ss.verify_step(p, q, [[0]], [[u_lo]], [0])
    n_hi, _ = ss.verify_step(p, q, [[0]], [[u_hi]], [0])
    assert n_lo[0] == 1 and n_hi[0] == 0


def test_in_order_rule_and_bonus_token():
    V = 4
    p = np.full((1, 3, V), 0.25, dtype=np.float32)
    q = np.full((1, 2, V), 0.25, dtype=np.float32)
    p[0, 2] = [0.0, 0.0, 0.5, 0.5]
    # both candidates kept (p = q: always accepted): the bonus comes from p_3
    n, tok = ss.verify_step(p, q, [[1, 3]], [[0.9, 0.9]], [0])
    assert n[0] == 2 and tok[0] == 2
    n, tok = ss.verify_step(p, q, [[1, 3]], [[0.9, 0.9]], [2**32 - 1])
    assert tok[0] == 3
    # a zero-probability candidate cannot have been proposed: rejected, and
    # the later candidate is never looked at
    q2 = q.copy(); q2[0, 0] = [0.5, 0.0, 0.5, 0.0]
    p2 = p.copy(); p2[0, 0] = [0.1, 0.4, 0.1, 0.4]
    n, tok = ss.verify_step(p2, q2, [[1, 3]], [[0.0, 0.0]], [0])
    assert n[0] == 0 and tok[0] in (1, 3)


def test_sampled_output_follows_the_target():
    """Eq. 33.13 by simulation: many independent draws of one verification
    (k = 1) reproduce p within sampling error."""
    rng = np.random.default_rng(5)
    V, N = 6, 40000
    p = rng.dirichlet(np.ones(V)).astype(np.float32); p /= p.sum()
    q = rng.dirichlet(np.ones(V)).astype(np.float32); q /= q.sum()
    q64 = q.astype(np.float64)
    x = rng.choice(V, size=N, p=q64 / q64.sum())
    u = rng.random(N, dtype=np.float32)
    s = rng.integers(0, 2**32, size=N, dtype=np.uint64)
    P = np.broadcast_to(np.stack([p, p])[None], (N, 2, V))
    Q = np.broadcast_to(q[None, None], (N, 1, V))
    n, tok = ss.verify_step(P, Q, x[:, None], u[:, None], s)
    emitted = np.where(n == 1, x, tok)
    freq = np.bincount(emitted, minlength=V) / N
    assert np.all(np.abs(freq - p) < 5 * np.sqrt(p * (1 - p) / N) + 1e-3)


# ---- eq. 33.12's residual [p - q]_+ is the EXACT difference of the fp32 values

EXACT_RESIDUAL_CASES = [
    # (p, q, F(p - q)) worked out by hand: F(m) = floor(m 2^40)
    (1 - 2.0**-24, 2.0**-30, 2**40 - 2**16 - 2**10),  # an fp32 subtraction returns p
    (1 - 2.0**-24, 2.0**-80, 2**40 - 2**16 - 1),      # 80 significant bits: an fp64 subtraction rounds too
    (0.75, 3 * 2.0**-40, 3 * 2**38 - 3),
    (0.5, 3 * 2.0**-27, 2**39 - 3 * 2**13),            # fp32 rounds 0.5 - 0.75 ulp to 0.5 - 1 ulp
    (2.0**-10 + 2.0**-33, 2.0**-10, 2**7),             # cancellation (exact in any precision)
    (2.0**-17, 2.0**-60, 2**23 - 1),                   # just below an integer weight
    (0.25, 0.25, 0), (0.1, 0.2, 0),                    # [.]_+ clips
    (2.0**-41, 0.0, 0), (2.0**-40, 0.0, 1), (3 * 2.0**-41, 2.0**-149, 1),
]


@pytest.mark.parametrize("p,q,want", EXACT_RESIDUAL_CASES)
def test_residual_weight_is_the_exact_difference(p, q, want):
    assert np.float32(p) == p and np.float32(q) == q  # the operands are fp32 values
    assert int(ss.weights(np.array([p], np.float32), np.array([q], np.float32))[0]) == want


def test_exact_residual_cases_discriminate_rounding():
    """The first cases are ones where a rounded subtraction gives another weight
    (a planted fp32 or fp64 residual would fail the pins above)."""
    for p, q, want in EXACT_RESIDUAL_CASES[:4]:
        m32 = float(np.float32(p) - np.float32(q))
        assert math.floor(m32 * 2**40) != want
    p, q, want = EXACT_RESIDUAL_CASES[1]
    assert math.floor((p - q) * 2**40) != want


def test_residual_weights_brute_force_wide_exponents():
    """Random fp32 pairs whose exponents lie up to 60 binades apart, against
    the exact rational difference formed from integer numerators (every
    exponent gap, so the rule for where fp64 is exact is pinned too)."""
    rng = np.random.default_rng(11)
    n = 4000
    p = (rng.random(n) * 2.0 ** -rng.integers(0, 30, n)).astype(np.float32)
    q = (rng.random(n) * 2.0 ** -rng.integers(0, 60, n)).astype(np.float32)
    q[::7] = p[::7]
    q[1::7] = np.nextafter(p[1::7], np.float32(0))
    w = ss.weights(p, q)
    for x in range(n):
        a, da = float(p[x]).as_integer_ratio()
        b, db = float(q[x]).as_integer_ratio()
        num, den = a * db - b * da, da * db  # p - q = num / den exactly
        want = 0 if num <= 0 else min((num << 40) // den, 2**41)
        assert int(w[x]) == want, (x, float(p[x]), float(q[x]))
    gaps = np.abs(np.frexp(p.astype(np.float64))[1] - np.frexp(q.astype(np.float64))[1])
    assert (gaps > 28).sum() > 500 and (gaps <= 28).sum() > 500


def test_token_follows_the_exact_residual():
    """A draw on the boundary that the exact residual moves: V = 3, the
    candidate (token 2, p = 0) is rejected, the residual weights are
    w = (2^39 - 3 2^13, 2^38, 0) (by hand, as above), and the first draw s
    with floor(s Z / 2^32) >= w_0 emits token 1 while s - 1 emits token 0.
    With the residual rounded to fp32 (w_0 = 2^39 - 2^14) both give token 0."""
    p = np.array([[[0.5, 0.25, 0.0], [1.0, 0.0, 0.0]]], np.float32)
    q = np.array([[[3 * 2.0**-27, 0.0, 0.5]]], np.float32)
    w0, w1 = 2**39 - 3 * 2**13, 2**38
    Z = w0 + w1
    s = -(-(w0 << 32) // Z)  # ceil(w0 2^32 / Z)
    assert (s * Z) >> 32 == w0 and ((s - 1) * Z) >> 32 < w0
    assert tuple(x[0] for x in ss.verify_step(p, q, [[2]], [[0.5]], [s])) == (0, 1)
    assert tuple(x[0] for x in ss.verify_step(p, q, [[2]], [[0.5]], [s - 1])) == (0, 0)
    w0r = 2**39 - 2**14  # the rounded residual would put s below its boundary
    assert (s * (w0r + w1)) >> 32 < w0r
