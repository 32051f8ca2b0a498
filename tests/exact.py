"""Exact rational arithmetic with an independent round-to-nearest-even.

Used by the oracle's pins: the oracle's binary32 / BF16 operations are
re-derived here from exact rationals and an explicit rounding rule, so a wrong
order, index, rounding or dropped term in the C code shows up as a mismatch.
Nothing here calls the oracle or the CUDA library.
"""
import struct
from fractions import Fraction

import numpy as np

F32 = (24, -126, 127)   # significand bits (with the hidden one), emin, emax
BF16 = (8, -126, 127)
F16 = (11, -14, 15)


def _round_half_even(q: Fraction) -> int:
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem == Fraction(1, 2):
        return fl + (fl & 1)
    return fl


def rn(x: Fraction, fmt=F32):
    """Nearest value of the format to x (ties to even), with subnormals and
    overflow to +-inf.  Returns a Fraction, or a float infinity."""
    p, emin, emax = fmt
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, emin) - p + 1)
    n = _round_half_even(a / quantum)
    v = n * quantum
    largest = (Fraction(2) - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if v > largest:
        return float("inf") * sign
    return sign * v


def f32_bits(v) -> int:
    return struct.unpack("<I", struct.pack("<f", float(v)))[0]


def bf16_bits_of(v) -> int:
    """Bit pattern of a value that is exactly representable in BF16."""
    b = f32_bits(v)
    assert b & 0xFFFF == 0, "value is not a BF16 number"
    return b >> 16


def bf16_value(bits: int) -> Fraction:
    return Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))


def f32_value(x) -> Fraction:
    return Fraction(float(np.float32(x)))
