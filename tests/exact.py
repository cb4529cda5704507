"""Exact rational arithmetic for pinning the oracle (test helper).

Independent of the oracle: bf16 patterns are decoded from their sign,
exponent and fraction fields (IEEE-754 §3.4), sums are exact rationals, and
rounding to a binary format is done by scaling to the format's quantum and
rounding the integer part half-to-even (IEEE-754 §4.3.1, §7.4 overflow).
"""
from __future__ import annotations

from fractions import Fraction

INF = "inf"
NINF = "-inf"

# binary formats: (precision p incl. the implicit bit, emin, emax)
BINARY32 = (24, -126, 127)
BFLOAT16 = (8, -126, 127)


def decode_bf16(bits: int):
    """bf16 pattern -> (Fraction value, is_negative_zero) or INF/NINF/None(NaN)."""
    s = (bits >> 15) & 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0xFF:
        if f:
            return None
        return NINF if s else INF
    if e == 0:
        mag = Fraction(f, 128) * Fraction(2) ** -126
    else:
        mag = (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127)
    if mag == 0:
        return (Fraction(0), bool(s))
    return (-mag if s else mag, False)


def _floor_log2(a: Fraction) -> int:
    # largest e with 2^e <= a  (a > 0)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_to(x: Fraction, fmt) -> Fraction | str:
    """Round an exact nonzero rational to the format, ties to even."""
    p, emin, emax = fmt
    neg = x < 0
    a = -x if neg else x
    e = max(_floor_log2(a), emin)
    q = Fraction(2) ** (e - p + 1)          # quantum of the binade
    m = a / q
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * q
    if r >= Fraction(2) ** (emax + 1):
        return NINF if neg else INF
    return -r if neg else r


def encode_bf16(v) -> int:
    """Exact bf16-representable value (Fraction, neg-zero flag) -> pattern."""
    if v == INF:
        return 0x7F80
    if v == NINF:
        return 0xFF80
    val, negzero = v
    if val == 0:
        return 0x8000 if negzero else 0x0000
    s = 1 if val < 0 else 0
    a = -val if s else val
    e = _floor_log2(a)
    if e < -126:                       # subnormal: a = f/128 * 2^-126
        f = a / Fraction(2) ** -126 * 128
        assert f.denominator == 1
        return (s << 15) | int(f)
    f = (a / Fraction(2) ** e - 1) * 128
    assert f.denominator == 1, "value not representable in bf16"
    return (s << 15) | ((e + 127) << 7) | int(f)


def add32(acc, x):
    """binary32 addition of two binary32 values given exactly; returns the
    rounded result as (Fraction, negzero) or INF/NINF/None."""
    if acc is None or x is None:
        return None
    if acc in (INF, NINF) or x in (INF, NINF):
        vals = {v for v in (acc, x) if v in (INF, NINF)}
        return None if len(vals) == 2 else vals.pop()
    (a, az), (b, bz) = acc, x
    s = a + b
    if s == 0:
        # exact zero sum: -0 only when both operands are -0 (roundTiesToEven)
        both_negzero = (a == 0 and az) and (b == 0 and bz)
        return (Fraction(0), both_negzero)
    r = round_to(s, BINARY32)
    if r in (INF, NINF):
        return r
    return (r, False)


def to_bf16_bits(acc) -> int:
    if acc is None:
        return 0x7FC0
    if acc in (INF, NINF):
        return encode_bf16(acc)
    val, negzero = acc
    if val == 0:
        return encode_bf16((val, negzero))
    r = round_to(val, BFLOAT16)
    if r in (INF, NINF):
        return encode_bf16(r)
    return encode_bf16((r, False))


def fold_bits(values: list[int]) -> int:
    """Exact model of the fixed-order fold: acc = x0; acc = rnd32(acc + xp);
    result = rnd_bf16(acc)."""
    acc = decode_bf16(values[0])
    for b in values[1:]:
        acc = add32(acc, decode_bf16(b))
    return to_bf16_bits(acc)


def decode_f32(bits: int):
    """binary32 pattern -> (Fraction value, is_negative_zero) or INF/NINF/None(NaN)."""
    s = (bits >> 31) & 1
    e = (bits >> 23) & 0xFF
    f = bits & 0x7FFFFF
    if e == 0xFF:
        if f:
            return None
        return NINF if s else INF
    if e == 0:
        mag = Fraction(f, 1 << 23) * Fraction(2) ** -126
    else:
        mag = (1 + Fraction(f, 1 << 23)) * Fraction(2) ** (e - 127)
    if mag == 0:
        return (Fraction(0), bool(s))
    return (-mag if s else mag, False)


def encode_f32(v) -> int:
    """Exact binary32-representable value (Fraction, neg-zero flag) -> pattern."""
    if v == INF:
        return 0x7F800000
    if v == NINF:
        return 0xFF800000
    val, negzero = v
    if val == 0:
        return 0x80000000 if negzero else 0
    s = 1 if val < 0 else 0
    a = -val if s else val
    e = _floor_log2(a)
    if e < -126:
        f = a / Fraction(2) ** -126 * (1 << 23)
        assert f.denominator == 1
        return (s << 31) | int(f)
    f = (a / Fraction(2) ** e - 1) * (1 << 23)
    assert f.denominator == 1
    return (s << 31) | ((e + 127) << 23) | int(f)


def add_exact(x, y):
    """IEEE-754 binary32 addition of two decoded operands (§6.1, §6.3):
    infinities, signed zeros under round-to-nearest, and one rounding of the
    exact sum.  None stands for NaN."""
    if x is None or y is None:
        return None
    if x in (INF, NINF) or y in (INF, NINF):
        if x in (INF, NINF) and y in (INF, NINF) and x != y:
            return None
        return x if x in (INF, NINF) else y
    (vx, zx), (vy, zy) = x, y
    t = vx + vy
    if t == 0:
        # exact zero sum: -0 only when both operands are -0 (§6.3)
        return (Fraction(0), vx == 0 and vy == 0 and zx and zy)
    r = round_to(t, BINARY32)
    if r in (INF, NINF):
        return r
    return (r, r == 0 and t < 0)
