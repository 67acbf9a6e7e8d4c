"""Exact bf16 arithmetic for the tests, from the format definition alone.

bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
Normal values are (-1)^s * 2^(e-127) * (1 + f/128); subnormals (e = 0) are
(-1)^s * f * 2^-133; e = 255 is inf (f = 0) or NaN.  Rounding here works on
exact rationals (``fractions.Fraction``), so it shares nothing with the
oracle's bit-level rounding or with the CUDA conversion instructions.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

BF16_MAX = Fraction(255, 128) * Fraction(2) ** 127        # 0x7F7F
POS_INF, NEG_INF, QNAN = 0x7F80, 0xFF80, 0x7FC0


def decode(b: int):
    """bf16 pattern -> Fraction, or float('inf')/-inf/nan."""
    s = -1 if b & 0x8000 else 1
    e = (b >> 7) & 0xFF
    f = b & 0x7F
    if e == 0xFF:
        return float("nan") if f else s * float("inf")
    if e == 0:
        return s * Fraction(f) * Fraction(2) ** -133
    return s * (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127)


def is_nan(b: int) -> bool:
    return ((b >> 7) & 0xFF) == 0xFF and (b & 0x7F) != 0


def round_rne(q) -> int:
    """Exact rational (or +-0.0/inf/nan float) -> nearest bf16, ties to even.

    A rational above the largest finite value by half a step or more
    rounds to infinity, as IEEE 754 round-to-nearest prescribes."""
    if isinstance(q, float):
        if math.isnan(q):
            return QNAN
        if math.isinf(q):
            return POS_INF if q > 0 else NEG_INF
        if q == 0.0:
            return 0x8000 if math.copysign(1.0, q) < 0 else 0
        q = Fraction(q)
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    # exponent of the leading bit: 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                  # below 2^-126 the step stays 2^-133
    step = Fraction(2) ** (e - 7)
    n = a / step
    k = math.floor(n)
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    v = k * step
    if v > BF16_MAX:
        return sign | 0x7F80
    return sign | encode_exact(v)


def encode_exact(v) -> int:
    """Exactly representable non-negative value -> bf16 pattern."""
    v = Fraction(v)
    if v == 0:
        return 0
    if v < Fraction(2) ** -126:
        f = v / Fraction(2) ** -133
        assert f.denominator == 1 and f < 128
        return int(f)
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1
    f = (v / Fraction(2) ** e - 1) * 128
    assert f.denominator == 1, "value not representable in bf16"
    return ((e + 127) << 7) | int(f)


def bits(value) -> int:
    """Pattern of a value that bf16 represents exactly (or 0x.... / nan)."""
    if isinstance(value, str):
        s = value.strip().lower()
        if s.startswith("0x"):
            return int(s, 16)
        if s == "nan":
            return QNAN
        value = Fraction(s)
    v = Fraction(value)
    return (0x8000 if v < 0 else 0) | encode_exact(abs(v))


def ordered(b):
    """Map bf16 patterns to integers whose order is the numeric order,
    with +0 and -0 equal; the ulp distance is the difference."""
    b = np.asarray(b, dtype=np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_diff(a, b) -> np.ndarray:
    return np.abs(ordered(a) - ordered(b))


def nan_mask(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def to_f64(b) -> np.ndarray:
    """bf16 patterns -> float64 (exact)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def from_f64_rne(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 patterns, round to nearest even, one rounding.

    Uses frexp so the rounding happens on the exact binary64 value."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    flat = x.ravel()
    res = out.ravel()
    for i, v in enumerate(flat):
        res[i] = round_rne(float(v)) if (v == 0 or not np.isfinite(v)) \
            else round_rne(Fraction(float(v)))
    return out
