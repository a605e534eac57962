"""Exact-arithmetic helpers for the oracle pins (tests only).

Everything here is independent of the C oracle: rationals from ``fractions``,
square roots and trig functions from ``decimal`` at 60 significant digits,
and a bf16 rounding written on rationals.  A pin that compares the oracle
with these helpers therefore checks the oracle against arithmetic that shares
none of its code.
"""
from __future__ import annotations

import struct
from decimal import Decimal, getcontext
from fractions import Fraction

getcontext().prec = 60

_BF16_MAX = Fraction((2**8 - 1) * 2**120)          # (2 - 2^-7) * 2^127
_BF16_OVERFLOW = Fraction(2**128 - 2**119)         # max + half a quantum


def bits_to_fraction(bits: int) -> Fraction:
    """bf16 bit pattern -> exact rational (finite values only)."""
    f = struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]
    return Fraction(f)


def f32_to_fraction(v: float) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<f", v))[0])


def _round_half_even(q: Fraction) -> int:
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def round_bf16(q) -> int:
    """Exact rational (or Decimal) -> nearest bf16 bit pattern, ties to even."""
    if isinstance(q, Decimal):
        q = Fraction(q)
    q = Fraction(q)
    if q == 0:
        return 0x0000
    sign = 0x8000 if q < 0 else 0
    a = -q if q < 0 else q
    # exponent e with 2^(e-1) <= a < 2^e
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    while Fraction(2) ** e <= a:
        e += 1
    qexp = max(e - 8, -133)
    quantum = Fraction(2) ** qexp
    n = _round_half_even(a / quantum)
    r = n * quantum
    if a >= _BF16_OVERFLOW:
        return sign | 0x7F80
    assert r <= _BF16_MAX
    f = float(r)  # exact: r has at most 8 significant bits
    u = struct.unpack("<I", struct.pack("<f", f))[0]
    return sign | (u >> 16)


def dsqrt(q: Fraction) -> Decimal:
    return (Decimal(q.numerator) / Decimal(q.denominator)).sqrt()


def to_dec(q: Fraction) -> Decimal:
    return Decimal(q.numerator) / Decimal(q.denominator)


_PI = Decimal("3.14159265358979323846264338327950288419716939937510582097494459")


def _reduce(a: Decimal) -> Decimal:
    two_pi = 2 * _PI
    k = (a / two_pi).to_integral_value()
    return a - k * two_pi


def dcos(a: Decimal) -> Decimal:
    """cos by Taylor series after reduction to [-pi, pi]; 60-digit context."""
    x = _reduce(a)
    term = Decimal(1)
    s = Decimal(1)
    x2 = x * x
    for k in range(1, 80):
        term = -term * x2 / ((2 * k - 1) * (2 * k))
        s += term
        if abs(term) < Decimal(10) ** -58:
            break
    return s


def dsin(a: Decimal) -> Decimal:
    x = _reduce(a)
    term = x
    s = x
    x2 = x * x
    for k in range(1, 80):
        term = -term * x2 / ((2 * k) * (2 * k + 1))
        s += term
        if abs(term) < Decimal(10) ** -58:
            break
    return s


def dec_to_f32(d: Decimal) -> float:
    """Nearest binary32 of a Decimal (via the exact rational)."""
    q = Fraction(d)
    # round to float32 exactly: use the bf16-style routine generalised to 24 bits
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    while Fraction(2) ** e <= a:
        e += 1
    qexp = max(e - 24, -149)
    quantum = Fraction(2) ** qexp
    n = _round_half_even(a / quantum)
    return sign * float(n * quantum)


def ulp_distance_bf16(a_bits, b_bits):
    """Element-wise distance in bf16 units in the last place between two arrays
    of bit patterns, on the sign-magnitude ordering (so +0 and -0 are 0 apart)."""
    import numpy as np
    a = np.asarray(a_bits, dtype=np.uint16).astype(np.int32)
    b = np.asarray(b_bits, dtype=np.uint16).astype(np.int32)

    def ordered(u):
        mag = u & 0x7FFF
        return np.where(u & 0x8000, -mag, mag)

    return np.abs(ordered(a) - ordered(b))


def bits_to_f64(bits):
    import numpy as np
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


_F16_OVERFLOW = Fraction(65520)  # 65504 + half a quantum: ties to 2^16 (even) -> inf


def round_f16(q) -> int:
    """Exact rational -> nearest IEEE binary16 bit pattern, ties to even."""
    q = Fraction(q)
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = -q if q < 0 else q
    if a >= _F16_OVERFLOW:
        return sign | 0x7C00
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    while Fraction(2) ** e <= a:
        e += 1
    qexp = max(e - 11, -24)
    n = _round_half_even(a / Fraction(2) ** qexp)
    r = n * Fraction(2) ** qexp
    import numpy as np
    return sign | int(np.array([float(r)], dtype=np.float16).view(np.uint16)[0])


def f16_bits_to_f64(bits):
    import numpy as np
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)
