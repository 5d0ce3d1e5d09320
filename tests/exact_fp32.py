"""Exact IEEE-754 binary32 arithmetic on rationals, for pinning the oracle.

Every value is a ``fractions.Fraction``; ``f32(q)`` rounds an exact rational
to the nearest binary32 value (ties to even), returning +-inf on overflow.
The oracle's float32 steps are checked against these exact roundings, which
do not depend on the host's floating-point unit, compiler flags or FMA
contraction.
"""
from fractions import Fraction
import math
import struct

INF = float("inf")


def f32(q):
    """Round an exact rational (or +-inf) to the nearest binary32 value."""
    if isinstance(q, float) and math.isinf(q):
        return q
    q = Fraction(q)
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = -q if q < 0 else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp_exp = max(e, -126) - 23
    m = round(a / Fraction(2) ** ulp_exp)          # Fraction.__round__: ties to even
    r = m * Fraction(2) ** ulp_exp
    if r >= Fraction(2) ** 128:
        return sign * INF
    return sign * r


def mul(a, b):
    if isinstance(a, float) or isinstance(b, float):
        return f32(float(a) * float(b))
    return f32(Fraction(a) * Fraction(b))


def add(a, b):
    if isinstance(a, float) or isinstance(b, float):
        return f32(float(a) + float(b))
    return f32(Fraction(a) + Fraction(b))


def rne_int(t):
    """Round to the nearest integer, ties to even (inf passes through)."""
    if isinstance(t, float):
        return t
    return Fraction(round(t))


def clamp_i8(t):
    if isinstance(t, float):
        return 127 if t > 0 else -128
    return int(max(Fraction(-128), min(Fraction(127), t)))


def as_f32(x):
    """The exact value of a Python/numpy float after rounding to binary32."""
    v = struct.unpack("<f", struct.pack("<f", float(x)))[0]
    if math.isinf(v):
        return v
    return Fraction(v)


def recip_in_double_then_f32(scale):
    """(float)(1.0 / scale) with 1.0/scale a correctly rounded binary64 division."""
    return as_f32(1.0 / float(scale))
