"""Exact reference arithmetic for pinning the oracle.

Values are computed with Python's Fraction and big integers, then rounded to
binary32 by the IEEE 754 rule (nearest, ties to even, gradual underflow,
overflow to infinity). Nothing here calls the oracle or the C library's
float routines.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

F32_MAX_EXP = 127
F32_MIN_EXP = -126
F32_MANT = 23
POS_INF = 0x7F800000
CANON_NAN = 0x7FFFFFFF


def bits_to_fraction(bits: int):
    """Returns ('nan'|'inf'|'fin', sign, Fraction magnitude) for f32 bits."""
    sign = (bits >> 31) & 1
    e = (bits >> 23) & 0xFF
    m = bits & 0x7FFFFF
    if e == 0xFF:
        return ("nan" if m else "inf"), sign, None
    if e == 0:
        mag = Fraction(m, 1 << 149)
    else:
        mag = Fraction((1 << 23) | m, 1) * Fraction(2) ** (e - 150)
    return "fin", sign, mag


def value(bits: int):
    kind, sign, mag = bits_to_fraction(bits)
    if kind != "fin":
        return kind, sign
    return "fin", (-mag if sign else mag), sign


def round_f32(x: Fraction, zero_sign: int = 0) -> int:
    """Rounds an exact rational to binary32 bits (nearest, ties to even)."""
    if x == 0:
        return zero_sign << 31
    sign = 1 if x < 0 else 0
    a = -x if sign else x
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if e >= F32_MIN_EXP:
        q_exp = e - F32_MANT
    else:
        q_exp = F32_MIN_EXP - F32_MANT  # subnormal quantum 2^-149
    m = a / (Fraction(2) ** q_exp)
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    # re-normalise
    if n >= (1 << 24):
        n >>= 1
        q_exp += 1
    if n == 0:
        return sign << 31
    if n < (1 << 23):
        assert q_exp == F32_MIN_EXP - F32_MANT
        return (sign << 31) | n  # subnormal
    biased = q_exp + F32_MANT + 127
    if biased >= 0xFF:
        return (sign << 31) | POS_INF
    return (sign << 31) | (biased << 23) | (n & 0x7FFFFF)


def f32_bits(f: float) -> int:
    return struct.unpack("<I", struct.pack("<f", f))[0]


def bits_f32(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def add(a: int, b: int, sub: bool = False) -> int:
    ka, sa, ma = bits_to_fraction(a)
    kb, sb, mb = bits_to_fraction(b)
    if sub:
        sb ^= 1
    if ka == "nan" or kb == "nan":
        return CANON_NAN
    if ka == "inf" and kb == "inf":
        return CANON_NAN if sa != sb else (sa << 31) | POS_INF
    if ka == "inf":
        return (sa << 31) | POS_INF
    if kb == "inf":
        return (sb << 31) | POS_INF
    x = (-ma if sa else ma) + (-mb if sb else mb)
    if x == 0:
        # exact zero: -0 only when both operands are -0 (round to nearest)
        zs = 1 if (sa and sb and ma == 0 and mb == 0) else 0
        return round_f32(x, zs)
    return round_f32(x)


def mul(a: int, b: int) -> int:
    ka, sa, ma = bits_to_fraction(a)
    kb, sb, mb = bits_to_fraction(b)
    s = sa ^ sb
    if ka == "nan" or kb == "nan":
        return CANON_NAN
    if ka == "inf" or kb == "inf":
        if (ka == "fin" and ma == 0) or (kb == "fin" and mb == 0):
            return CANON_NAN
        return (s << 31) | POS_INF
    return round_f32(ma * mb * (-1 if s else 1), s)


def div(a: int, b: int) -> int:
    ka, sa, ma = bits_to_fraction(a)
    kb, sb, mb = bits_to_fraction(b)
    s = sa ^ sb
    if ka == "nan" or kb == "nan":
        return CANON_NAN
    if ka == "inf" and kb == "inf":
        return CANON_NAN
    if ka == "inf":
        return (s << 31) | POS_INF
    if kb == "inf":
        return s << 31
    if mb == 0:
        if ma == 0:
            return CANON_NAN
        return (s << 31) | POS_INF
    return round_f32(ma / mb * (-1 if s else 1), s)


def fma(a: int, b: int, c: int) -> int:
    ka, sa, ma = bits_to_fraction(a)
    kb, sb, mb = bits_to_fraction(b)
    kc, sc, mc = bits_to_fraction(c)
    if "nan" in (ka, kb, kc):
        return CANON_NAN
    sp = sa ^ sb
    if ka == "inf" or kb == "inf":
        if (ka == "fin" and ma == 0) or (kb == "fin" and mb == 0):
            return CANON_NAN
        if kc == "inf" and sc != sp:
            return CANON_NAN
        return (sp << 31) | POS_INF
    if kc == "inf":
        return (sc << 31) | POS_INF
    prod = ma * mb * (-1 if sp else 1)
    x = prod + (-mc if sc else mc)
    if x == 0:
        prod_zero_neg = (ma * mb == 0) and sp
        zs = 1 if (prod_zero_neg and sc and mc == 0) else 0
        return round_f32(x, zs)
    return round_f32(x)


def sqrt(a: int) -> int:
    ka, sa, ma = bits_to_fraction(a)
    if ka == "nan":
        return CANON_NAN
    if ma == 0 and ka == "fin":
        return sa << 31  # sqrt(-0) = -0
    if sa:
        return CANON_NAN
    if ka == "inf":
        return POS_INF
    # correctly rounded sqrt: find candidate via integer sqrt at high precision
    # r = sqrt(ma) exactly bracketed: scale so that the integer part has >= 60 bits
    k = 200
    num = ma.numerator << (2 * k)
    den = ma.denominator
    # sqrt(num/den) = sqrt(num*den)/den
    s = math.isqrt(num * den)
    # sqrt(ma) in [s/den, (s+1)/den) * 2^-k
    lo = Fraction(s, den) / (Fraction(2) ** k)
    hi = Fraction(s + 1, den) / (Fraction(2) ** k)
    r_lo, r_hi = round_f32(lo), round_f32(hi)
    if r_lo == r_hi:
        return r_lo
    # decide exactly: compare ma with the square of the midpoint between r_lo and r_hi
    m = (bits_to_fraction(r_lo)[2] + bits_to_fraction(r_hi)[2]) / 2
    if ma > m * m:
        return r_hi
    if ma < m * m:
        return r_lo
    return r_lo if (r_lo & 1) == 0 else r_hi


def int_to_f32(v: int) -> int:
    return round_f32(Fraction(v))


def f32_to_int(bits: int, mode: str, width: int, signed: bool) -> int:
    kind, sign, mag = bits_to_fraction(bits)
    if kind == "nan":
        return 0
    lo = -(1 << (width - 1)) if signed else 0
    hi = (1 << (width - 1)) - 1 if signed else (1 << width) - 1
    if kind == "inf":
        v = hi if not sign else lo
    else:
        x = -mag if sign else mag
        if mode == "rzi":
            v = math.trunc(x)
        elif mode == "rmi":
            v = math.floor(x)
        elif mode == "rpi":
            v = math.ceil(x)
        else:  # rni: nearest, ties to even
            f = math.floor(x)
            d = x - f
            v = f + (1 if d > Fraction(1, 2) or (d == Fraction(1, 2) and f % 2 == 1) else 0)
        v = max(lo, min(hi, v))
    return v & ((1 << width) - 1)


def cmp_f32(a: int, b: int, op: str) -> bool:
    ka, sa, ma = bits_to_fraction(a)
    kb, sb, mb = bits_to_fraction(b)
    if ka == "nan" or kb == "nan":
        return False
    big = Fraction(2) ** 200
    x = (big if ka == "inf" else ma) * (-1 if sa else 1)
    y = (big if kb == "inf" else mb) * (-1 if sb else 1)
    return {"eq": x == y, "ne": x != y, "lt": x < y, "le": x <= y, "gt": x > y, "ge": x >= y}[op]
