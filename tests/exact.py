"""Exact rational arithmetic helpers for the brute-force pins (pure Python).

Written from the IEEE-754 definition of round-to-nearest-even on the bf16
grid (8 significant bits, exponent range of binary32), with Fractions, so it
shares nothing with the oracle's C code."""

from fractions import Fraction
import math
import struct


def bf16_bits_to_fraction(h: int) -> Fraction:
    f = struct.unpack("<f", struct.pack("<I", (h & 0xFFFF) << 16))[0]
    if math.isinf(f) or math.isnan(f):
        raise ValueError("non-finite")
    return Fraction(f)


def round_bf16(x: Fraction) -> Fraction:
    """Nearest bf16 value to x, ties to even; overflow returns +-inf as float."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    # binade: 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 7)
    q, rem = divmod(a, ulp)
    q = int(q)
    half = ulp / 2
    if rem > half or (rem == half and q % 2 == 1):
        q += 1
    r = q * ulp
    if r >= Fraction(2) ** 128:
        return sign * math.inf
    return sign * r


def bf16_sum(a_bits: int, b_bits: int):
    return round_bf16(bf16_bits_to_fraction(a_bits) + bf16_bits_to_fraction(b_bits))


def argmax_lowest(values) -> int:
    best, idx = None, 0
    for i, v in enumerate(values):
        if best is None or v > best:
            best, idx = v, i
    return idx
