"""Exact rational evaluation of IEEE-754 binary32 arithmetic for the tests.

Each f32 operation of a definition is evaluated on exact rationals and then
rounded to the nearest binary32 value, ties to even (IEEE-754 section 4.3.1).
This gives expected results that do not depend on any floating-point unit or
on the code under test.
"""
from fractions import Fraction

import numpy as np

_HALF = Fraction(1, 2)


def f32_round(x: Fraction) -> Fraction:
    """Round an exact rational to the nearest binary32 value (ties to even)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = -x if x < 0 else x
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)  # subnormals share the smallest exponent
    ulp = Fraction(2) ** (e - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    r = q - n
    if r > _HALF or (r == _HALF and n % 2 == 1):
        n += 1
    return sign * n * ulp


def F(v) -> Fraction:
    """Exact value of a float (or float32)."""
    return Fraction(float(v))


def to_f32(x: Fraction) -> np.float32:
    y = np.float32(float(x))
    assert Fraction(float(y)) == x, "value is not a binary32 number"
    return y


def round_half_even(x: Fraction) -> int:
    n = x.numerator // x.denominator
    r = x - n
    if r > _HALF or (r == _HALF and n % 2 == 1):
        n += 1
    return n
