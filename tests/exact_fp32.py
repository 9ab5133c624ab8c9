"""Exact IEEE-754 binary32 rounding with Python rationals (test helper).

Used to pin the requantiser's float32 arithmetic independently of numpy and
of the GPU: every quotient is formed exactly as a Fraction and rounded to the
nearest binary32 value, ties to even, with gradual underflow.
"""

from fractions import Fraction

import numpy as np


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_fp32(x: Fraction, mant_bits: int = 23) -> Fraction:
    """Nearest binary32 value to the rational x (ties to even); finite range only.
    ``mant_bits`` = 7 gives bfloat16 (binary32's exponent range, 8 significant bits)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = max(_floor_log2(a), -126)
    quantum = Fraction(2) ** (e - mant_bits)
    n = a / quantum
    m = round(n)  # Python rounds a Fraction half to even
    return sign * m * quantum


def f32(v) -> Fraction:
    return Fraction(float(np.float32(v)))


def to_f32(fr: Fraction) -> np.float32:
    return np.float32(float(fr))
