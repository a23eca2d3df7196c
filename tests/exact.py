"""Exact-arithmetic helpers for pinning the oracle (test code, independent of it).

Every BF16 value is a dyadic rational, so sums of BF16 products are computed
exactly with ``fractions.Fraction``; SiLU is evaluated with ``decimal`` at 60
significant digits; BF16 rounding is decided by exact comparison with the
midpoints between neighbouring BF16 values. None of this shares code with
``oracle/``.
"""
from __future__ import annotations

import decimal
from fractions import Fraction

_CTX = decimal.Context(prec=60)


def bf16_fraction(bits: int) -> Fraction:
    """Decode a BF16 bit pattern field by field (finite values only)."""
    bits = int(bits) & 0xFFFF
    sign = -1 if bits & 0x8000 else 1
    exp = (bits >> 7) & 0xFF
    man = bits & 0x7F
    assert exp != 0xFF, "inf/nan"
    if exp == 0:
        return sign * Fraction(man, 1 << 133)            # subnormal: man * 2^-133
    val = Fraction(128 + man, 128)                        # 1.man
    e = exp - 127
    return sign * (val * (Fraction(2) ** e))


def exact_dot(a_bits, w_bits) -> Fraction:
    s = Fraction(0)
    for a, w in zip(a_bits, w_bits):
        s += bf16_fraction(a) * bf16_fraction(w)
    return s


def frac_to_decimal(x: Fraction) -> decimal.Decimal:
    return _CTX.divide(decimal.Decimal(x.numerator), decimal.Decimal(x.denominator))


def silu_decimal(g: decimal.Decimal) -> decimal.Decimal:
    """SiLU(g) = g / (1 + e^-g) at 60 digits."""
    return _CTX.divide(g, _CTX.add(decimal.Decimal(1), _CTX.exp(-g)))


def _bf16_grid_neighbours(x: Fraction):
    """(lo, hi, lo_is_even_significand) with lo <= |x| < hi on the BF16 grid."""
    ax = abs(x)
    # exponent of the binade holding ax (clamped to the subnormal range)
    e = -126
    if ax >= Fraction(2) ** -126:
        e = ax.numerator.bit_length() - ax.denominator.bit_length()
        while Fraction(2) ** e > ax:
            e -= 1
        while Fraction(2) ** (e + 1) <= ax:
            e += 1
    spacing = Fraction(2) ** (e - 7)
    q = ax // spacing                      # floor(ax / spacing)
    lo = q * spacing
    return lo, lo + spacing, int(q) % 2 == 0


def round_bf16_exact(x) -> int:
    """Exact value (Fraction or Decimal) -> BF16 bits by RNE, decided exactly."""
    if isinstance(x, decimal.Decimal):
        x = Fraction(x)
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    lo, hi, lo_even = _bf16_grid_neighbours(x)
    ax = abs(x)
    mid = (lo + hi) / 2
    if ax < mid or (ax == mid and lo_even):
        v = lo
    else:
        v = hi
    if v >= Fraction(2) ** 128:
        return sign | 0x7F80
    return sign | _encode_grid_value(v)


def _encode_grid_value(v: Fraction) -> int:
    if v == 0:
        return 0
    if v < Fraction(2) ** -126:
        units = v / Fraction(2) ** -133
        assert units.denominator == 1
        return int(units)
    e = v.numerator.bit_length() - v.denominator.bit_length()
    while Fraction(2) ** e > v:
        e -= 1
    while Fraction(2) ** (e + 1) <= v:
        e += 1
    man = v / Fraction(2) ** e - 1
    man128 = man * 128
    assert man128.denominator == 1
    return ((e + 127) << 7) | int(man128)


def near_tie(x: decimal.Decimal, rel: float = 1e-12) -> bool:
    """True when x lies within rel of a BF16 rounding midpoint (skip those)."""
    fx = Fraction(x)
    if fx == 0:
        return False
    lo, hi, _ = _bf16_grid_neighbours(fx)
    mid = (lo + hi) / 2
    return abs(abs(fx) - mid) <= Fraction(rel) * abs(fx)


def e4m3_fraction(bits: int) -> Fraction:
    """Decode an FP8 E4M3 pattern field by field (finite values only)."""
    bits = int(bits) & 0xFF
    sign = -1 if bits & 0x80 else 1
    exp = (bits >> 3) & 0xF
    man = bits & 0x7
    assert not (exp == 0xF and man == 0x7), "nan"
    if exp == 0:
        return sign * Fraction(man, 1 << 9)
    return sign * Fraction(8 + man, 8) * (Fraction(2) ** (exp - 7))
