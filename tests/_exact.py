"""Exact rounding in rational arithmetic, for pinning the oracle.

This is an independent restatement of IEEE round-to-nearest-even onto a binary
format (p significand bits, minimum normal exponent emin, maximum exponent
emax), done with Python integers and fractions.  Values from mpmath are
converted exactly (an mpf is man * 2^exp) before rounding.
"""
from fractions import Fraction
import math
import struct

import mpmath


def to_fraction(x) -> Fraction:
    if isinstance(x, Fraction):
        return x
    if isinstance(x, int):
        return Fraction(x)
    if isinstance(x, float):
        return Fraction(x)
    x = mpmath.mpf(x)
    if not mpmath.isfinite(x):
        raise ValueError("exact rounding needs a finite value")
    sign, man, exp, _ = x._mpf_
    man = -int(man) if sign else int(man)
    exp = int(exp)
    return Fraction(man * 2 ** exp) if exp >= 0 else Fraction(man, 2 ** (-exp))


def round_fraction(x: Fraction, p: int, emin: int, emax: int):
    """RN-even of exact x onto the format; returns a Fraction or +-inf float."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    # E = floor(log2(a))
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    if Fraction(2) ** (E + 1) <= a:
        E += 1
    E = max(E, emin)
    q = Fraction(2) ** (E - (p - 1))
    k = a / q
    fl = k.numerator // k.denominator
    rem = k - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * q
    max_finite = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if r > max_finite:
        return sign * math.inf
    return sign * r


def rn32(x) -> float:
    r = round_fraction(to_fraction(x), 24, -126, 127)
    return float(r)


def rn16_bits(x) -> int:
    """bf16 bit pattern of RN16(x) for an exact (non-NaN) value x."""
    fx = to_fraction(x)
    r = round_fraction(fx, 8, -126, 127)
    if isinstance(r, float):  # infinity
        return 0xFF80 if r < 0 else 0x7F80
    f = float(r)
    bits = struct.unpack("<I", struct.pack("<f", f))[0]
    assert bits & 0xFFFF == 0
    b = bits >> 16
    if r == 0 and fx < 0:
        b = 0x8000
    return b


def rn16_of_rn32_bits(x) -> int:
    """bf16 bits of RN16(RN32(x)) for exact x."""
    fx = to_fraction(x)
    r32 = round_fraction(fx, 24, -126, 127)
    if isinstance(r32, float):
        return 0xFF80 if r32 < 0 else 0x7F80
    if r32 == 0:
        return 0x8000 if fx < 0 else 0
    return rn16_bits(r32)


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0]


def is_nan_bits(bits: int) -> bool:
    return (bits & 0x7F80) == 0x7F80 and (bits & 0x007F) != 0
