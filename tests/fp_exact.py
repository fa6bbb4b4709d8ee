"""Exact rational arithmetic with explicit IEEE-754 rounding, for pinning the oracle.

Every binary32 operation the oracle claims to perform is "the exact result,
rounded to nearest, ties to even".  These helpers compute exactly that with
Python Fractions and integers, independently of any floating-point unit.
"""
from fractions import Fraction
import math
import struct

import numpy as np


def f32_bits(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(np.float32(x))))[0]


def bits_f32(b: int) -> np.float32:
    return np.frombuffer(struct.pack("<I", b & 0xFFFFFFFF), dtype=np.float32)[0]


def exact(x) -> Fraction:
    """Exact rational value of a finite binary32/binary64 number."""
    return Fraction(float(x))


def _round_scaled(a: Fraction, quantum: Fraction) -> Fraction:
    """a rounded to an integer multiple of quantum, ties to even."""
    q = a / quantum
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n * quantum


def rn(a: Fraction, mant_bits: int, emin: int, emax: int) -> float:
    """Round a rational to the binary format with `mant_bits` significand bits
    (including the hidden bit), minimum normal exponent emin, maximum exponent emax."""
    if a == 0:
        return 0.0
    sign = -1 if a < 0 else 1
    a = abs(a)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # now 2^e <= a < 2^(e+1)
    e = max(e, emin)
    quantum = Fraction(2) ** (e - (mant_bits - 1))
    r = _round_scaled(a, quantum)
    if r >= Fraction(2) ** (emax + 1):
        return sign * math.inf
    return sign * float(r)


def rn32(a: Fraction) -> np.float32:
    return np.float32(rn(a, 24, -126, 127))


def rn64(a: Fraction) -> float:
    return rn(a, 53, -1022, 1023)


def rn_bf16_bits(x: np.float32) -> int:
    """bf16 nearest to a finite binary32 value (ties to even), as bits."""
    r = rn(exact(x), 8, -126, 127)
    if math.isinf(r):
        return 0x7F80 | (0x8000 if r < 0 else 0)
    b = f32_bits(np.float32(r))
    assert b & 0xFFFF == 0
    hi = b >> 16
    if r == 0 and math.copysign(1.0, float(x)) < 0:
        hi = 0x8000
    return hi


def sqrt_rn32(a: Fraction) -> np.float32:
    """Correctly rounded binary32 square root of a non-negative rational."""
    if a == 0:
        return np.float32(0.0)
    # scale so that the integer square root carries far more than 24 bits
    k = 200
    scaled = a * Fraction(2) ** (2 * k)
    n = scaled.numerator // scaled.denominator
    s = math.isqrt(n)
    # sqrt(a) lies in [s, s+1) / 2^k; with 200 extra bits the rounding decision is
    # exact unless sqrt(a) * 2^k is an integer, which isqrt detects
    if s * s == n and scaled.denominator == 1:
        return rn32(Fraction(s, 2 ** k))
    # irrational (or not exactly representable): use the midpoint of the bracket,
    # which cannot straddle a rounding boundary of a 24-bit result
    return rn32(Fraction(2 * s + 1, 2 ** (k + 1)))


def add(a, b):
    return rn32(exact(a) + exact(b))


def sub(a, b):
    return rn32(exact(a) - exact(b))


def mul(a, b):
    return rn32(exact(a) * exact(b))


def div(a, b):
    return rn32(exact(a) / exact(b))


def sqrt(a):
    return sqrt_rn32(exact(a))
