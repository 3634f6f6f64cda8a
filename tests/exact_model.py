"""Exact rational model of binary floating-point rounding, for pinning the oracle.

An independent restatement of IEEE 754 round-to-nearest-even on a binary grid
(p significant bits, smallest normal exponent emin, largest exponent emax) in
exact rational arithmetic (``fractions.Fraction``). The oracle (binary64 C) and
this model share nothing but the rule they follow, so agreement between them
checks the oracle's arithmetic, not a retyping of it.

BF16 is (p=8, emin=-126, emax=127); binary32 is (p=24, emin=-126, emax=127).
"""
from fractions import Fraction
import math
import struct

BF16 = (8, -126, 127)
F32 = (24, -126, 127)

INF = float("inf")


def _floor_log2(a: Fraction) -> int:
    """Largest e with 2^e <= a (a > 0)."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_ne(q, fmt):
    """Nearest value of the format to the rational q, ties to even.

    Returns a Fraction (possibly 0) or +-inf on overflow. The sign of an exact
    zero result is the caller's business (see ``to_bits``).
    """
    p, emin, emax = fmt
    if isinstance(q, float) and math.isinf(q):
        return q
    q = Fraction(q)
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = -q if q < 0 else q
    e = max(_floor_log2(a), emin)
    ulp = Fraction(2) ** (e - (p - 1))
    t = a / ulp
    r = t.numerator // t.denominator
    d = t - r
    if d > Fraction(1, 2) or (d == Fraction(1, 2) and r % 2 == 1):
        r += 1
    res = r * ulp
    if res >= Fraction(2) ** (emax + 1):
        return sign * INF
    return sign * res


def to_bits_bf16(value, negative_zero=False) -> int:
    """BF16 pattern of a value already on the BF16 grid (Fraction, float or inf)."""
    if value == 0:
        return 0x8000 if negative_zero else 0x0000
    f = float(value)
    if math.isinf(f):
        return 0xFF80 if f < 0 else 0x7F80
    (u,) = struct.unpack("<I", struct.pack("<f", f))
    if u & 0xFFFF:
        raise ValueError(f"{value!r} is not on the BF16 grid")
    return u >> 16


def from_bits_bf16(b: int) -> Fraction:
    """Exact value of a finite BF16 pattern."""
    (f,) = struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))
    if math.isinf(f) or math.isnan(f):
        raise ValueError("not finite")
    return Fraction(f)


def is_negative_zero_bits(b: int) -> bool:
    return (b & 0xFFFF) == 0x8000


def bf16_of_rational(q) -> int:
    """BF16 pattern nearest to q (positive zero for an exact zero)."""
    return to_bits_bf16(round_ne(q, BF16))


def f32_add(a, b, a_negzero=False, b_negzero=False):
    """binary32 a + b (ties to even) with IEEE signed-zero rules.

    Values are Fractions on the binary32 grid; zeros carry their sign in the
    flags. Returns (value, is_negative_zero).
    """
    if any(isinstance(v, float) and math.isinf(v) for v in (a, b)):
        return float(a) + float(b), False
    s = Fraction(a) + Fraction(b)
    if s == 0:
        # Exact zero sum: -0 only when both operands are -0 (round to nearest).
        both_neg = (a == 0 and a_negzero) and (b == 0 and b_negzero)
        return Fraction(0), both_neg
    r = round_ne(s, F32)
    return r, False


def gemm_exact_bits(x_rows, w_rows):
    """out[m][n] = BF16(sum_k x[m][k] w[n][k]) with the sum exact (Fractions)."""
    out = []
    for xr in x_rows:
        row = []
        for wr in w_rows:
            s = sum((Fraction(a) * Fraction(b) for a, b in zip(xr, wr)), Fraction(0))
            row.append(bf16_of_rational(s))
        out.append(row)
    return out


def reduce_bits(slot_bits, residual_bits=None):
    """One column of the reduce: binary32 rank-order sum from slot 0, BF16 rounding,
    optional binary32 residual add, BF16 rounding. Inputs and result are patterns."""
    s = from_bits_bf16(slot_bits[0])
    neg = is_negative_zero_bits(slot_bits[0])
    for b in slot_bits[1:]:
        s, neg = f32_add(s, from_bits_bf16(b), neg, is_negative_zero_bits(b))
    a = round_ne(s, BF16)
    # A zero after rounding keeps the sign of what was rounded (IEEE 754).
    a_neg = (neg if s == 0 else s < 0) if a == 0 else False
    if residual_bits is None:
        return to_bits_bf16(a, a_neg)
    h, h_neg = f32_add(a, from_bits_bf16(residual_bits), a_neg,
                       is_negative_zero_bits(residual_bits))
    hr = round_ne(h, BF16)
    return to_bits_bf16(hr, (h_neg if h == 0 else h < 0) if hr == 0 else False)
