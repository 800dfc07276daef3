"""Pins for the oracle's decoder, its round-to-nearest-even encoder and its
round-to-odd sum, against library casts and exact rational arithmetic."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import _exact

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rng(seed=1234):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_exhaustive_16bit(dtype):
    bits = np.arange(1 << 16, dtype=np.uint32)
    want = _exact.decode(bits, dtype)
    got = np.array([oracle.value(int(b), dtype) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_f32_random_and_special():
    rng = _rng()
    bits = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, np.array([0, 0x80000000, 1, 0x7F7FFFFF, 0x7F800000, 0xFF800000,
                                           0x7FC00000, 0x00800000, 0x007FFFFF], dtype=np.uint32)])
    want = _exact.decode(bits, "f32")
    got = np.array([oracle.value(int(b), "f32") for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _interesting_doubles(dtype, n=4000, seed=7):
    """Values on, between and exactly halfway between representable values,
    across the subnormal, normal and overflow ranges."""
    rng = _rng(seed)
    if dtype == "f32":
        bits = rng.integers(0, 0x7F800000, size=n, dtype=np.int64).astype(np.uint32)
        nxt = bits + 1
    else:
        bits = rng.integers(0, _exact.MAX_FINITE[dtype], size=n, dtype=np.int64).astype(np.uint32)
        nxt = bits + 1
    lo = _exact.decode(bits, dtype)
    hi = _exact.decode(nxt, dtype)
    mid = (lo + hi) / 2            # exact in binary64 for these formats
    eps = np.abs(hi - lo) * 2.0 ** -20
    vals = np.concatenate([lo, mid, mid + eps, mid - eps, lo + eps, hi - eps,
                           rng.uniform(-1, 1, n) * 10.0 ** rng.uniform(-50, 50, n)])
    sign = rng.integers(0, 2, size=vals.size) * 2 - 1
    extra = [0.0, -0.0, np.inf, -np.inf, 1e300, -1e300, 5e-324, 2.0 ** -1074 * 3]
    return np.concatenate([vals * sign, extra])


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_round_matches_numpy_cast(dtype):
    """numpy's float64 -> float16 / float32 casts round to nearest even."""
    x = _interesting_doubles(dtype)
    np_t = np.float16 if dtype == "f16" else np.float32
    with np.errstate(over="ignore"):
        want = x.astype(np_t).view(np.uint16 if dtype == "f16" else np.uint32).astype(np.int64)
    got = np.array([oracle.round_to(v, dtype) for v in x], dtype=np.int64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_round_matches_exact_nearest_search(dtype):
    """Independent rounding: exact distances to neighbouring values."""
    x = _interesting_doubles(dtype, n=700, seed=11)
    for v in x:
        if not np.isfinite(v):
            continue
        want = _exact.round_exact(Fraction(float(v)), dtype, negative_zero=bool(np.signbit(v)))
        got = oracle.round_to(float(v), dtype)
        assert got == want, (dtype, v, hex(got), hex(want))


def test_round_hand_cases():
    # ties to even, overflow, subnormal boundaries, NaN -> canonical quiet NaN
    assert oracle.round_to(65504.0, "f16") == 0x7BFF
    assert oracle.round_to(65519.99, "f16") == 0x7BFF
    assert oracle.round_to(65520.0, "f16") == 0x7C00          # tie above max -> inf
    assert oracle.round_to(2.0 ** -24, "f16") == 0x0001        # smallest subnormal
    assert oracle.round_to(2.0 ** -25, "f16") == 0x0000        # tie -> even (zero)
    assert oracle.round_to(3 * 2.0 ** -25, "f16") == 0x0002    # tie 1.5 -> 2
    assert oracle.round_to(-2.0 ** -26, "f16") == 0x8000       # rounds to -0
    assert oracle.round_to(1.0 + 2.0 ** -11, "f16") == 0x3C00  # tie -> even
    assert oracle.round_to(1.0 + 3 * 2.0 ** -11, "f16") == 0x3C02
    assert oracle.round_to(1.0 + 2.0 ** -8, "bf16") == 0x3F80
    assert oracle.round_to(1.0 + 3 * 2.0 ** -8, "bf16") == 0x3F82
    assert oracle.round_to(float("nan"), "f16") == 0x7E00
    assert oracle.round_to(float("nan"), "bf16") == 0x7FC0
    assert oracle.round_to(float("nan"), "f32") == 0x7FC00000
    flt_max = 3.4028234663852886e38
    assert oracle.round_to(flt_max, "f32") == 0x7F7FFFFF
    assert oracle.round_to(flt_max + 2.0 ** 103, "f32") == 0x7F800000            # tie above max -> inf
    assert oracle.round_to(np.nextafter(flt_max + 2.0 ** 103, 0), "f32") == 0x7F7FFFFF
    assert oracle.round_to(2.0 ** -149, "f32") == 0x00000001
    assert oracle.round_to(2.0 ** -133, "bf16") == 0x0001


def test_round_odd_sum_definition():
    """x + y rounded to odd: exact if representable, else the odd neighbour
    of the exact sum (checked with exact rationals)."""
    rng = _rng(3)
    xs = rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)
    ys = rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)
    # cancellation-prone pairs and exact cases
    xs = np.concatenate([xs, [1.0, 1.0, 2.0 ** 60, 1e-300, 3.0]])
    ys = np.concatenate([ys, [2.0 ** -60, -1.0, -(2.0 ** 60) + 1, 1e-300, 2.0 ** -53]])
    for x, y in zip(xs, ys):
        s = oracle.add_round_odd(float(x), float(y))
        z = Fraction(float(x)) + Fraction(float(y))
        if Fraction(float(z)) == z:
            assert s == float(z)
            continue
        fs = Fraction(s)
        bits = np.array([s]).view(np.uint64)[0]
        assert bits & 1 == 1, (x, y, s)
        other = np.nextafter(s, np.inf if z > fs else -np.inf)
        lo, hi = sorted([fs, Fraction(float(other))])
        assert lo < z < hi, (x, y, s)


def test_ulp_distance_and_same_value():
    d = oracle.ulp_distance(np.array([0x3C00, 0x3C01, 0x8000, 0x0001, 0x8001, 0x7E00]),
                            np.array([0x3C00, 0x3C00, 0x0000, 0x8001, 0x0001, 0x7E01]), "f16")
    assert list(d) == [0, 1, 0, 2, 2, 0]
    d = oracle.ulp_distance(np.array([0x7E00]), np.array([0x3C00]), "f16")
    assert d[0] > 1 << 40
    assert list(oracle.same_value(np.array([0x7FC00000, 1, 0]), np.array([0x7FC00001, 1, 0x80000000]), "f32")) \
        == [True, True, False]
