"""Exact rational references used to pin the oracle.

Nothing here shares an algorithm with ``oracle/tsx_oracle.c``: values are
decoded by numpy / bit reinterpretation, and rounding is decided by comparing
exact ``Fraction`` distances to the neighbouring representable values (ties
to the even bit pattern), found by a table search or a library conversion.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

BITS = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32}
MAX_FINITE = {"f16": 0x7BFF, "bf16": 0x7F7F, "f32": 0x7F7FFFFF}
POS_INF = {"f16": 0x7C00, "bf16": 0x7F80, "f32": 0x7F800000}
SIGN = {"f16": 0x8000, "bf16": 0x8000, "f32": 0x80000000}


def decode(bits, dtype: str) -> np.ndarray:
    """Library decode of element bits to float64 (numpy casts; signalling
    NaNs widen quietly)."""
    b = np.asarray(bits)
    with np.errstate(invalid="ignore"):
        if dtype == "f16":
            return b.astype(np.uint16).view(np.float16).astype(np.float64)
        if dtype == "bf16":
            return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        return b.astype(np.uint32).view(np.float32).astype(np.float64)


def frac_of_bits(bits: int, dtype: str) -> Fraction:
    return Fraction(float(decode(np.array([bits]), dtype)[0]))


def _pos_table(dtype: str):
    """All finite non-negative values of a 16-bit format, ascending."""
    bits = np.arange(0, MAX_FINITE[dtype] + 1, dtype=np.uint32)
    return bits, decode(bits, dtype)


_TABLES = {}


def table(dtype: str):
    if dtype not in _TABLES:
        _TABLES[dtype] = _pos_table(dtype)
    return _TABLES[dtype]


def _neighbours_16(az: Fraction, dtype: str):
    bits, vals = table(dtype)
    approx = float(az) if az < Fraction(10) ** 300 else float("inf")
    i = int(np.searchsorted(vals, approx))
    cand = set()
    for j in range(i - 2, i + 3):
        if 0 <= j < len(bits):
            cand.add(int(bits[j]))
    return cand


def _neighbours_32(az: Fraction):
    approx = np.float32(float(az)) if az < Fraction(2) ** 200 else np.float32(np.inf)
    base = int(np.array([approx], dtype=np.float32).view(np.uint32)[0])
    cand = set()
    for j in range(base - 2, base + 3):
        if 0 <= j <= MAX_FINITE["f32"]:
            cand.add(j)
    return cand


def _overflow_threshold(dtype: str) -> Fraction:
    """max finite + half its ulp: at or above this, RN gives infinity."""
    mx = frac_of_bits(MAX_FINITE[dtype], dtype)
    below = frac_of_bits(MAX_FINITE[dtype] - 1, dtype)
    return mx + (mx - below) / 2


def round_exact(z: Fraction, dtype: str, negative_zero: bool = False) -> int:
    """Round-to-nearest-even of the exact rational ``z`` into ``dtype`` bits."""
    sign = SIGN[dtype] if (z < 0 or (z == 0 and negative_zero)) else 0
    az = abs(z)
    if az >= _overflow_threshold(dtype):
        return sign | POS_INF[dtype]
    cand = _neighbours_16(az, dtype) if dtype != "f32" else _neighbours_32(az)
    best = None
    for c in sorted(cand):
        d = abs(frac_of_bits(c, dtype) - az)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    return sign | best[1]
