"""Exact-arithmetic references for float32 chains (test helpers).

Everything here works on exact rationals (``fractions.Fraction``) and rounds
to binary32 by the IEEE 754 rule written out (nearest value, ties to the even
significand), so it depends on neither the host's FPU nor numpy's casts.  It
holds the alternative ways a dot product can be evaluated, so that a test can
check that the oracle and the GPU evaluate the indexer score as the in-order
fused chain that the library defines and not as one of the others.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

_MIN_EXP = -149          # binary32: the smallest subnormal is 2^-149
_MAX_FINITE = Fraction((1 << 24) - 1) * Fraction(2) ** 104


def round_f32(x: Fraction) -> np.float32:
    """The binary32 value nearest to the rational x, ties to an even significand."""
    if x == 0:
        return np.float32(0.0)
    neg = x < 0
    a = -x if neg else x
    # exponent e of the last significand bit: 2^23 <= a / 2^e < 2^24 (normal range)
    e = a.numerator.bit_length() - a.denominator.bit_length() - 24
    while a / Fraction(2) ** e >= (1 << 24):
        e += 1
    while a / Fraction(2) ** e < (1 << 23):
        e -= 1
    e = max(e, _MIN_EXP)                 # subnormals share the fixed quantum 2^-149
    m = a / Fraction(2) ** e
    n = m.numerator // m.denominator
    rest = m - n
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = Fraction(n) * Fraction(2) ** e
    assert v <= _MAX_FINITE, "overflow is outside what these tests use"
    f = np.float32(float(v))             # n * 2^e is a binary32 value, so this is exact
    assert Fraction(float(f)) == v
    return np.float32(-f) if neg else f


def fma_chain(q, r, order=None) -> np.float32:
    """s = 0; s = fma(q[i], r[i], s) over i in `order` (default 0..d-1): one rounding per step."""
    idx = range(len(q)) if order is None else order
    s = np.float32(0.0)
    for i in idx:
        s = round_f32(Fraction(float(q[i])) * Fraction(float(r[i])) + Fraction(float(s)))
    return s


def unfused_chain(q, r) -> np.float32:
    """s = 0; s = (s + round(q[i] * r[i])) rounded: two roundings per step."""
    s = np.float32(0.0)
    for i in range(len(q)):
        p = round_f32(Fraction(float(q[i])) * Fraction(float(r[i])))
        s = round_f32(Fraction(float(s)) + Fraction(float(p)))
    return s


def exact_dot_rounded_once(q, r) -> np.float32:
    """The exact dot product, rounded once to binary32."""
    return round_f32(sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(q, r)), Fraction(0)))


def double_dot_rounded_once(q, r) -> np.float32:
    """A double accumulation of the products (each step rounded to binary64), then one binary32 rounding."""
    s = 0.0
    for a, b in zip(q, r):
        s = s + float(a) * float(b)
    return round_f32(Fraction(s))


def distinguishing_pairs(n_pairs: int, d: int, seed: int):
    """Deterministic (q, row) float32 pairs of width d on which the in-order fused
    chain differs from the reversed fused chain, the unfused chain, the exact dot
    rounded once and the double-accumulated dot.  Values have full 24-bit
    significands so that every step rounds."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n_pairs:
        q = rng.uniform(-2.0, 2.0, d).astype(np.float32)
        r = rng.uniform(-2.0, 2.0, d).astype(np.float32)
        s = fma_chain(q, r)
        alts = (fma_chain(q, r, range(d - 1, -1, -1)), unfused_chain(q, r), exact_dot_rounded_once(q, r),
                double_dot_rounded_once(q, r))
        if all(a != s for a in alts):
            out.append((q, r, s))
    return out
