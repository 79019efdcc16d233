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
