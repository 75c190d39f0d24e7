"""The division method the merge passes use, checked in exact arithmetic.

The passes divide s by the round's divisor d (the worker count, or the token
total) with the reciprocal held as two binary32 terms, y = RN(1/d) and
y_lo = RN(1/d - y), and one of Markstein's corrections (P. Markstein,
"Computation of elementary functions on the IBM RISC System/6000 processor",
IBM J. Res. Develop. 34(1), 1990):

    q0 = RN(s*y + RN(s*y_lo)),  r = s - d*q0 (exact),  q = RN(q0 + r*y),

for |s| in [2^max(-100, e-124), 2^min(126, e+124)) where d lies in
[2^(e-1), 2^e) inside [2^-100, 2^100]; every other dividend takes the
division instruction. The claim is that q is the correctly rounded s/d. Here
every binary32 operation is carried out on exact rationals and rounded to
nearest-even by hand, so the claim is checked independently of any
floating-point unit: on random dividends of every admitted exponent and on the
range's end points, for divisors from 2^-99 to 2^99, including significands of
all ones. The GPU tests check the kernels' bits against IEEE division on every
binary32 dividend for two divisors.
"""
from __future__ import annotations

import math
import random
import struct
from fractions import Fraction as Q

import pytest

INF = Q(10) ** 400  # stands for an overflow to infinity (never reached in range)


def rn32(x: Q) -> Q:
    """x rounded to the nearest binary32 value, ties to even, subnormals kept."""
    if x == 0:
        return Q(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Q(2) ** e > a:
        e -= 1
    if Q(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    quantum = Q(2) ** (e - 23)
    m = a / quantum
    n = m.numerator // m.denominator
    rest = m - n
    if rest > Q(1, 2) or (rest == Q(1, 2) and n % 2 == 1):
        n += 1
    v = n * quantum
    return sign * (INF if v >= Q(2) ** 128 else v)


def as_f32(x: float) -> Q:
    return Q(struct.unpack("<f", struct.pack("<f", x))[0])


def plan(d: Q) -> tuple[int, int]:
    _, e = math.frexp(float(d))
    return max(-100, e - 124), min(126, e + 124)


def two_term_quotient(s: Q, d: Q) -> Q:
    y = rn32(1 / d)
    y_lo = rn32(Q(1.0 / float(d) - float(y)))  # binary64 1/d - y, as the host forms it
    q0 = rn32(s * y + rn32(s * y_lo))
    r = s - d * q0
    assert rn32(r) == r, "the remainder is not representable"
    return rn32(q0 + r * y)


DIVISORS = [3, 5, 6, 7, 10, 1000, 123_457, (1 << 24) - 1, (1 << 24) + 2, 999_999_999,
            (1 << 31) - 1, 3 * (1 << 40) + 12_345, 1 << 56, 1.0000001, 1.9999999, 0.3, 1e-20,
            7e25, 2.0 ** -99, 2.0 ** 99]


@pytest.mark.parametrize("divisor", DIVISORS)
def test_two_term_quotient_is_correctly_rounded(divisor):
    d = as_f32(float(divisor))
    lo_e, hi_e = plan(d)
    rng = random.Random(int(float(d) * 1e6) % (1 << 31) + hi_e)
    cases = []
    for e in (lo_e, hi_e - 1):  # the range's ends
        for mant in (0, 1, (1 << 22), (1 << 23) - 1):
            cases.append(Q(2) ** e * (1 + Q(mant, 1 << 23)))
    for _ in range(400):
        e = rng.randint(lo_e, hi_e - 1)
        cases.append(Q(2) ** e * (1 + Q(rng.randint(0, (1 << 23) - 1), 1 << 23)))
    for s in cases:
        for v in (s, -s):
            assert two_term_quotient(v, d) == rn32(v / d), (float(v), float(d))


def test_rounding_helper_against_known_values():
    # the hand-written rounding agrees with the machine's binary32 conversion
    # on values whose nearest binary32 neighbour is known
    for x in (1 / 3, 2 / 3, 0.1, 1e-40, 3.4e38, 1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24):
        assert rn32(Q(x)) == as_f32(x)
    assert rn32(Q(1) + Q(1, 1 << 24)) == 1  # a tie goes to the even neighbour
    assert rn32(Q(1) + Q(3, 1 << 24)) == Q(1) + Q(2, 1 << 23)
