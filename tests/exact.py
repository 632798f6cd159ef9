"""Exact rational arithmetic for pinning the oracle (test helper).

Round-to-nearest-even into BF16 is written here from the IEEE 754 definition
over Python ``Fraction``s: find the binade, scale by the unit in the last
place, round the quotient half to even, rescale. Nothing here shares code
with the oracle's bit-twiddling rounding or with the GPU path.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

import numpy as np

BF16_MANT = 8          # significand bits, implicit bit included
BF16_EMIN = -126       # smallest normal exponent
BF16_EMAX = 127
F32_MANT = 24


def bits_to_value(h: int):
    """BF16 bits -> exact Fraction (or a float inf/nan)."""
    f = struct.unpack("<f", struct.pack("<I", (int(h) & 0xFFFF) << 16))[0]
    if math.isinf(f) or math.isnan(f):
        return f
    return Fraction(f)


def f32_to_value(x: float):
    f = float(np.float32(x))
    if math.isinf(f) or math.isnan(f):
        return f
    return Fraction(f)


def _round_half_even(q: Fraction) -> int:
    fl = math.floor(q)
    rem = q - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def rne(q: Fraction, mant: int = BF16_MANT, emin: int = BF16_EMIN, emax: int = BF16_EMAX):
    """Round an exact rational to the nearest binary float with ``mant``
    significand bits (ties to even). Returns a Fraction, or +-inf."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix floating error of log2 on huge/small rationals
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - (mant - 1))
    n = _round_half_even(a / ulp)
    r = n * ulp
    if r >= Fraction(2) ** (emax + 1):
        return sign * math.inf
    return sign * r


def value_to_bf16_bits(v, negative_zero: bool = False) -> int:
    """Exact BF16-representable value -> bits."""
    if isinstance(v, float) and math.isinf(v):
        return 0xFF80 if v < 0 else 0x7F80
    f = float(v)
    u = struct.unpack("<I", struct.pack("<f", f))[0]
    assert u & 0xFFFF == 0, "value is not representable in BF16"
    h = u >> 16
    if f == 0 and negative_zero:
        h = 0x8000
    return h


def rne_bf16_bits(q) -> int:
    return value_to_bf16_bits(rne(q))


def rne_f32(q: Fraction):
    return rne(q, mant=F32_MANT, emin=-126, emax=127)
