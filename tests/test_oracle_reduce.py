"""Pins for the oracle's row reduction: exact rational sums, integer-valued
rows, the decoder against numpy, and the summation error bound against
actual float32 summations in several orders."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import _exact


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_decode_matches_numpy(dtype):
    rng = np.random.default_rng(1)
    top = 1 << (32 if dtype == "f32" else 16)
    bits = rng.integers(0, top, size=5000, dtype=np.uint64).astype(np.uint32 if dtype == "f32" else np.uint16)
    got = oracle.decode(bits, dtype)
    want = _exact.decode(bits, dtype)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("op", ["copy", "sqrt", "mul", "fma"])
def test_rowsum_is_the_exact_sum_rounded_once(op):
    rng = np.random.default_rng(2)
    rows, cols = 6, 300
    n_in = {"copy": 1, "sqrt": 1, "mul": 2, "fma": 3}[op]
    ins = [(np.abs(rng.standard_normal((rows, cols))) * 2.0 ** rng.integers(-20, 20, (rows, cols)))
           .astype(np.float32).view(np.uint32) for _ in range(n_in)]
    sums, abs_sums = oracle.rowsum(op, "f32", *ins)
    x = _exact.decode(oracle.ewise(op, "f32", *ins), "f32").reshape(rows, cols)
    for r in range(rows):
        exact = sum((Fraction(float(v)) for v in x[r]), Fraction(0))
        assert sums[r] == float(exact)
        assert abs_sums[r] == float(sum((abs(Fraction(float(v))) for v in x[r]), Fraction(0)))


def test_rowsum_integer_rows_are_exact():
    a = np.arange(-500, 500, dtype=np.float32).reshape(4, 250)
    sums, _ = oracle.rowsum("copy", "f32", a.view(np.uint32))
    assert list(sums) == [float(v) for v in a.astype(np.float64).sum(axis=1)]


def test_summation_bound_holds_for_float32_orders():
    """Left-to-right, right-to-left, pairwise and strided-lane summation in
    float32 all stay within gamma(n-1) * sum |x| of the exact sum."""
    rng = np.random.default_rng(3)
    for n in (1, 2, 31, 512, 4096):
        x = (rng.standard_normal(n) * 2.0 ** rng.integers(-10, 10, n)).astype(np.float32)
        exact = float(sum((Fraction(float(v)) for v in x), Fraction(0)))
        bound = oracle.summation_error_bound(n, np.array([float(np.abs(x.astype(np.float64)).sum())]))[0]
        orders = []
        s = np.float32(0)
        for v in x:
            s = np.float32(s + v)
        orders.append(s)
        s = np.float32(0)
        for v in x[::-1]:
            s = np.float32(s + v)
        orders.append(s)
        lanes = np.zeros(32, dtype=np.float32)
        for i, v in enumerate(x):
            lanes[i % 32] = np.float32(lanes[i % 32] + v)
        while lanes.size > 1:
            lanes = (lanes[: lanes.size // 2] + lanes[lanes.size // 2:]).astype(np.float32)
        orders.append(lanes[0])
        for got in orders:
            assert abs(float(got) - exact) <= bound * (1 + 1e-12)


def test_summation_bound_closed_form():
    u = 2.0 ** -24
    assert oracle.summation_error_bound(2, np.array([1.0]))[0] == pytest.approx(u / (1 - u), rel=0)
    assert oracle.summation_error_bound(1, np.array([5.0]))[0] == 0.0
