"""The sampling kernel's short weight form, checked on the host.

For masses already in [0, 1] the kernel (csrc/spec_sample.cu,
add_entry_unit) forms F = floor((p - q) 2^40) for p > q (0 otherwise) from
seven fp32 operations with directed rounding instead of the exact TwoSum
pair.  This test restates those seven operations with exact rational
arithmetic and IEEE binary32 rounding written out here (round toward -inf,
round to nearest even; subnormals kept), and checks the result against the
exact floor on random, nearly equal, far-apart, subnormal and boundary
masses.  It shares no code with the kernel or the oracle; it pins the
derivation the kernel's comment gives ("Chapter 33: inference compute
optimisation" eq. 33.12: the residual is the exact difference)."""
import math
from fractions import Fraction as Fr

import numpy as np
import pytest

MAGIC = Fr(3 * 2 ** 22)  # 1.5 * 2^23
TWO20, TWO40, TWOM20 = Fr(2 ** 20), Fr(2 ** 40), Fr(1, 2 ** 20)


def _ulp(a: Fr) -> Fr:
    """Spacing of binary32 numbers at |a| > 0 (subnormal spacing 2^-149)."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fr(2) ** e > a:
        e -= 1
    while Fr(2) ** (e + 1) <= a:
        e += 1
    return Fr(2) ** max(e - 23, -149)


def rd(x: Fr) -> Fr:
    """Round toward -inf to binary32 (no overflow in these ranges)."""
    if x == 0:
        return Fr(0)
    if x < 0:  # toward -inf: the magnitude rounds up
        a = -x
        u = _ulp(a)
        return -a if a % u == 0 else -((a // u + 1) * u)
    u = _ulp(x)
    return (x // u) * u


def rn(x: Fr) -> Fr:
    """Round to nearest, ties to even, to binary32."""
    if x == 0:
        return Fr(0)
    sgn = 1 if x > 0 else -1
    a = abs(x)
    u = _ulp(a)
    q, r = divmod(a, u)
    if 2 * r > u or (2 * r == u and q % 2 == 1):
        q += 1
    return sgn * q * u


def short_form(p: float, q: float) -> int:
    """The kernel's seven operations on binary32 inputs p, q in [0, 1]."""
    p, q = Fr(float(np.float32(p))), Fr(float(np.float32(q)))
    qs = min(q, p)                       # fminf
    y = rd(p - qs)                       # __fadd_rd(p, -qs)
    mh = rd(y * TWO20 + MAGIC)           # __fmaf_rd(y, 2^20, 1.5 2^23)
    hf = rn(mh - MAGIC)                  # __fsub_rn
    d = rn(-hf * TWOM20 + p)             # __fmaf_rn(-hf, 2^-20, p)
    assert d == p - hf * TWOM20, "D must be exact"
    t = rd(d - qs)                       # __fadd_rd(d, -qs)
    ml = rd(t * TWO40 + MAGIC)           # __fmaf_rd(t, 2^40, 1.5 2^23)
    h, l = mh - MAGIC, ml - MAGIC
    assert h.denominator == 1 and l.denominator == 1 and 0 <= l < 2 ** 20
    return int(h) * 2 ** 20 + int(l)


def exact(p: float, q: float) -> int:
    m = Fr(float(np.float32(p))) - Fr(float(np.float32(q)))
    return max(0, math.floor(m * TWO40))


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    f32 = np.float32
    out = [(1.0, 0.0), (1.0, 1.0), (0.0, 0.0), (1.0, float(np.nextafter(f32(1), f32(0)))), (1.4e-45, 0.0),
           (1.0, 1.4e-45), (2.0 ** -20, 0.0), (2.0 ** -20, 2.0 ** -60), (2.0 ** -17, 2.0 ** -41), (0.5, 0.25)]
    for _ in range(n):
        kind = int(rng.integers(6))
        if kind == 0:
            p, q = rng.random(), rng.random()
        elif kind == 1:
            p = rng.random()
            q = p * (1 - 10 ** -rng.uniform(0, 8))
        elif kind == 2:
            p, q = 2.0 ** -rng.uniform(0, 140), 2.0 ** -rng.uniform(0, 140)
        elif kind == 3:
            p, q = 2.0 ** -rng.uniform(0, 30), 0.0
        elif kind == 4:
            p = rng.random()
            q = float(np.nextafter(f32(p), f32(0)))
        else:
            p = 2.0 ** -int(rng.integers(0, 60))
            q = 2.0 ** -int(rng.integers(0, 60)) * rng.random()
        out.append((float(f32(min(p, 1.0))), float(f32(min(q, 1.0)))))
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_short_form_equals_the_exact_floor(seed):
    for p, q in _cases(1500, seed):
        assert short_form(p, q) == exact(p, q), (p, q)


def test_rounding_helpers_against_numpy():
    """The hand-written binary32 rounding agrees with numpy's float32 casts
    (round to nearest) and with the neighbouring float below (round down)."""
    rng = np.random.default_rng(9)
    for _ in range(500):
        x = Fr(float(rng.standard_normal())) * Fr(2) ** int(rng.integers(-130, 20)) / 3
        assert rn(x) == Fr(float(np.float32(float(x)))) or abs(x) < Fr(2) ** -120  # (double rounding far below)
        r = rd(x)
        assert r <= x and rd(r) == r
        f = np.float32(float(r))
        assert Fr(float(np.nextafter(f, np.float32(np.inf)))) > x
