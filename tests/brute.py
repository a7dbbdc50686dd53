"""Independent brute force for pinning the oracle.

Softmax by Python ``decimal`` at 60 significant digits (its own exp, not the C
library's), and rounding to f32 / bf16 / f16 by exact rational arithmetic
(``fractions.Fraction``, round half to even). Nothing here is shared with the
oracle or with the CUDA path.
"""
from __future__ import annotations

import decimal
import math
from fractions import Fraction

import numpy as np

F32, BF16, F16 = 0, 1, 2
# (significand bits, smallest normal exponent, largest finite exponent)
FORMATS = {F32: (24, -126, 127), BF16: (8, -126, 127), F16: (11, -14, 15)}

CTX = decimal.Context(prec=60, rounding=decimal.ROUND_HALF_EVEN, Emin=-999999, Emax=999999)


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_exact(q: Fraction, dtype: int) -> float:
    """Nearest-even rounding of an exact rational to the format; returned as a float."""
    p, emin, emax = FORMATS[dtype]
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    e = _floor_log2(a)
    qe = max(e, emin) - (p - 1)
    r = round(a / Fraction(2) ** qe)  # Fraction.__round__ rounds half to even
    val = Fraction(r) * Fraction(2) ** qe
    if val >= Fraction(2) ** (emax + 1):
        return sign * math.inf
    return sign * float(val)  # exactly representable in double


def softmax_decimal(x) -> list:
    """Softmax of one row of floats at 60 digits; entries may be +-inf or NaN."""
    with decimal.localcontext(CTX):
        xs = [decimal.Decimal(float(v)) for v in x]
        if any(v.is_nan() for v in xs):
            return [decimal.Decimal("NaN")] * len(xs)
        m = max(xs)
        if m.is_infinite():
            # m = +inf: inf - inf is undefined; m = -inf: every term is 0/0.
            return [decimal.Decimal("NaN")] * len(xs)
        e = [(v - m).exp() for v in xs]
        s = sum(e)
        return [t / s for t in e]


def softmax_exact_cast(x, dtype: int) -> np.ndarray:
    """Brute-force softmax of one row, rounded once to the dtype, as float64 values."""
    ys = softmax_decimal(x)
    out = np.empty(len(ys), dtype=np.float64)
    for k, y in enumerate(ys):
        out[k] = math.nan if y.is_nan() else round_exact(Fraction(y), dtype)
    return out


def softmax_decimal_f64(x) -> np.ndarray:
    return np.array([float(y) for y in softmax_decimal(x)], dtype=np.float64)
