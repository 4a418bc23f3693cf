"""Exact rational arithmetic for pinning the oracle's IEEE roundings.

Each helper rounds an exact rational value with the textbook definition
(nearest representable value, ties to the even significand), independently of
any floating-point unit, so that the oracle's binary32 division, its
half-even rounding to an integer and its bf16 conversion are each checked
against their definitions rather than against a re-run of the same float code.
"""
from fractions import Fraction as F
import struct


def f32_from_bits(u: int) -> F:
    return F(struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0])


def bits_from_f32(v: F) -> int:
    """Bits of a rational that is exactly a binary32 value."""
    f = float(v)
    assert F(f) == v, "not exactly representable"
    return struct.unpack("<I", struct.pack("<f", f))[0]


def round_to_precision(v: F, p: int, emin: int) -> F:
    """Round v to p significant bits, ties to even; normal numbers only (the
    exponent of the result must be >= emin)."""
    if v == 0:
        return F(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    while F(2) ** (e + 1) <= a:
        e += 1
    assert e >= emin, "subnormal range not modelled"
    unit = F(2) ** (e - (p - 1))
    q = a / unit
    m = q.numerator // q.denominator
    rem = q - m
    if rem > F(1, 2) or (rem == F(1, 2) and m % 2 == 1):
        m += 1
    return sign * m * unit


def rn_f32(v: F) -> F:
    return round_to_precision(v, 24, -126)


def rn_bf16(v: F) -> F:
    return round_to_precision(v, 8, -126)


def bf16_bits_of(v: F, negative_zero: bool = False) -> int:
    """bf16 bits of a rational that is exactly a bf16 value."""
    if v == 0:
        return 0x8000 if negative_zero else 0
    b = bits_from_f32(v)
    assert b & 0xFFFF == 0, "not a bf16 value"
    return b >> 16


def rint_half_even(v: F) -> int:
    fl = v.numerator // v.denominator
    rem = v - fl
    if rem > F(1, 2) or (rem == F(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def expected_code(x: F, s: F) -> int:
    """clamp(round_half_even(fl32(x / s)), -127, 127); 0 when s == 0."""
    if s == 0:
        return 0
    r = rint_half_even(rn_f32(x / s))
    return max(-127, min(127, r))


def expected_row_scale(xs) -> F:
    return rn_f32(max(abs(x) for x in xs) / 127)


def expected_dequant_bits(q: int, s: F) -> int:
    """bf16 bits of rn_bf16(rn_f32(q * s)).  A zero product carries IEEE's sign:
    float(q) is +0 for q == 0, and the scales used in tests are never -0, so
    the product is -0 exactly when q < 0 and s == 0."""
    v = rn_bf16(rn_f32(F(q) * s))
    if v == 0:
        return bf16_bits_of(v, negative_zero=(q < 0 and s == 0))
    return bf16_bits_of(v)
