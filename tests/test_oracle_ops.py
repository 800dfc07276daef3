"""Pins for the oracle's elementwise ops.

Each op is checked against something other than the oracle itself: numpy's
IEEE float32 / float16 arithmetic, libm's fmaf, exact rational arithmetic
with round-to-nearest-even decided by exact distances, and mpmath's exp at
200 bits, exhaustively over all 2^16 inputs of the 16-bit types where that
is cheap.
"""

import ctypes
import ctypes.util
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import _exact

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

NPB = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32}


def _rand_bits(dtype, n, seed):
    rng = np.random.default_rng(seed)
    top = 1 << (32 if dtype == "f32" else 16)
    b = rng.integers(0, top, size=n, dtype=np.uint64).astype(NPB[dtype])
    return b


def _finite_bits(dtype, n, seed, max_exp_field=None):
    """Random finite values with magnitudes spread over the whole range."""
    b = _rand_bits(dtype, n, seed)
    vals = _exact.decode(b, dtype)
    return b[np.isfinite(vals)]


def _same(got, want, dtype):
    return np.all(oracle.same_value(got, want, dtype))


# ----------------------------------------------------------------- copy

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_copy_is_bitwise_exhaustive(dtype):
    a = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    assert np.array_equal(oracle.ewise("copy", dtype, a), a)   # NaN payloads kept


def test_copy_is_bitwise_f32():
    a = _rand_bits("f32", 1 << 16, 5)
    assert np.array_equal(oracle.ewise("copy", "f32", a), a)


# ------------------------------------------------------------ fp32 vs numpy

@pytest.mark.parametrize("op", ["add", "mul"])
def test_f32_binary_matches_ieee_single(op):
    a = _rand_bits("f32", 1 << 16, 1)
    b = _rand_bits("f32", 1 << 16, 2)
    # also pairs of close magnitude, where cancellation and ties happen
    a2 = np.random.default_rng(3).standard_normal(1 << 14).astype(np.float32)
    b2 = (a2 * np.float32(-1.0000001)).astype(np.float32)
    a = np.concatenate([a, a2.view(np.uint32)])
    b = np.concatenate([b, b2.view(np.uint32)])
    fa, fb = a.view(np.float32), b.view(np.float32)
    with np.errstate(all="ignore"):
        want = (fa + fb if op == "add" else fa * fb).view(np.uint32)
    got = oracle.ewise(op, "f32", a, b)
    assert _same(got, want, "f32")


def test_f32_sqrt_matches_ieee_single():
    a = _rand_bits("f32", 1 << 17, 4)
    a = np.concatenate([a, np.array([0, 0x80000000, 1, 0x7F800000, 0xFF800000, 0x3F800000, 0x40800000],
                                    dtype=np.uint32)])
    with np.errstate(all="ignore"):
        want = np.sqrt(a.view(np.float32)).view(np.uint32)
    got = oracle.ewise("sqrt", "f32", a)
    assert _same(got, want, "f32")


# ------------------------------------------------------------ fp16 vs numpy

def test_f16_sqrt_matches_numpy_exhaustive():
    a = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(all="ignore"):
        want = np.sqrt(a.view(np.float16)).view(np.uint16)
    assert _same(oracle.ewise("sqrt", "f16", a), want, "f16")


@pytest.mark.parametrize("op", ["add", "mul"])
def test_f16_binary_matches_numpy(op):
    a = _rand_bits("f16", 1 << 17, 6)
    b = _rand_bits("f16", 1 << 17, 7)
    fa, fb = a.view(np.float16), b.view(np.float16)
    with np.errstate(all="ignore"):
        want = (fa + fb if op == "add" else fa * fb).view(np.uint16)
    assert _same(oracle.ewise(op, "f16", a, b), want, "f16")


# ------------------------------------------------ exact rational references

def _sqrt_exact(bits, dtype):
    x = _exact.frac_of_bits(int(bits), dtype)
    if x == 0:
        return int(bits)             # sqrt(+-0) = +-0
    # bracketing candidates around the binary64 estimate
    est = float(np.sqrt(float(x)))
    c0 = _exact.round_exact(Fraction(est), dtype)
    cands = sorted({c0 - 1, c0, c0 + 1} - {-1}, key=lambda c: _exact.frac_of_bits(c, dtype))
    vals = [_exact.frac_of_bits(c, dtype) for c in cands]
    for (cl, vl), (ch, vh) in zip(zip(cands, vals), zip(cands[1:], vals[1:])):
        if vl * vl <= x <= vh * vh:
            m = (vl + vh) / 2
            if x < m * m:
                return cl
            if x > m * m:
                return ch
            return cl if cl % 2 == 0 else ch
    raise AssertionError("no bracket")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_sqrt_16bit_exhaustive_exact(dtype):
    """Correct rounding decided by exact squares, for every non-negative finite input."""
    a = np.arange(0, _exact.MAX_FINITE[dtype] + 1, dtype=np.uint32).astype(np.uint16)
    got = oracle.ewise("sqrt", dtype, a)
    for i in range(a.size):
        want = _sqrt_exact(a[i], dtype)
        assert int(got[i]) == want, (dtype, hex(int(a[i])), hex(int(got[i])), hex(want))
    # negative non-zero inputs give NaN; -0 gives -0
    neg = (a[1:] | np.uint16(0x8000)).astype(np.uint16)
    assert np.all(oracle.is_nan(oracle.ewise("sqrt", dtype, neg), dtype))
    assert int(oracle.ewise("sqrt", dtype, np.array([0x8000], dtype=np.uint16))[0]) == 0x8000


def _exact_op(op, vals):
    if op == "add":
        return vals[0] + vals[1]
    if op == "mul":
        return vals[0] * vals[1]
    return vals[0] * vals[1] + vals[2]


def _check_exact(op, dtype, ops, got):
    vals = [_exact.decode(o, dtype) for o in ops]
    for i in range(got.size):
        xs = [v[i] for v in vals]
        if not all(np.isfinite(xs)):
            continue
        z = _exact_op(op, [Fraction(float(x)) for x in xs])
        neg_zero = False
        if z == 0:
            # exact zero: IEEE sign rules (x + y with both -0, or -0 products)
            with np.errstate(all="ignore"):
                r = (np.float64(xs[0]) + np.float64(xs[1])) if op == "add" else \
                    (np.float64(xs[0]) * np.float64(xs[1])) if op == "mul" else \
                    (np.float64(xs[0]) * np.float64(xs[1]) + np.float64(xs[2]))
            neg_zero = bool(np.signbit(r))
        want = _exact.round_exact(z, dtype, negative_zero=neg_zero)
        assert int(got[i]) == want, (op, dtype, [hex(int(o[i])) for o in ops], hex(int(got[i])), hex(want))


def _moderate_bits(dtype, n, seed):
    """Finite values with exponents near 1, where sums of three operands
    interact (cancellation, ties, carries)."""
    rng = np.random.default_rng(seed)
    if dtype == "f32":
        x = (rng.standard_normal(n) * 2.0 ** rng.integers(-6, 6, n)).astype(np.float32)
        return x.view(np.uint32)
    if dtype == "f16":
        return (rng.standard_normal(n) * 2.0 ** rng.integers(-6, 6, n)).astype(np.float16).view(np.uint16)
    f = (rng.standard_normal(n) * 2.0 ** rng.integers(-6, 6, n)).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("op", ["add", "mul", "fma"])
def test_binary_and_fma_exact(op, dtype):
    n = 4000
    arity = 3 if op == "fma" else 2
    ops = [np.concatenate([_finite_bits(dtype, n, 10 * k + 1)[: n // 2], _moderate_bits(dtype, n // 2, 10 * k + 2)])
           for k in range(arity)]
    m = min(o.size for o in ops)
    ops = [o[:m] for o in ops]
    got = oracle.ewise(op, dtype, *ops)
    _check_exact(op, dtype, ops, got)


def test_fma_hard_cases_f32():
    """a*b lands exactly on a float32 midpoint and c nudges it: naive
    rounding of the binary64 sum to float32 would tie to even instead."""
    cases = []
    # a * b = 1 + 2^-24 (a float32 midpoint), c = +-2^-70 decides the direction
    a = np.float32(1.0 + 2.0 ** -12)
    b = np.float32(1.0 - 2.0 ** -12)      # a*b = 1 - 2^-24 exactly
    for c in (2.0 ** -70, -(2.0 ** -70), 0.0):
        cases.append((a, b, np.float32(c)))
    a = np.float32(1.0 + 2.0 ** -12)
    b = np.float32(1.0 + 2.0 ** -12)      # 1 + 2^-11 + 2^-24
    for c in (2.0 ** -60, -(2.0 ** -60), -1.0, -(1.0 + 2.0 ** -11)):
        cases.append((a, b, np.float32(c)))
    A = np.array([x[0] for x in cases], dtype=np.float32).view(np.uint32)
    B = np.array([x[1] for x in cases], dtype=np.float32).view(np.uint32)
    C = np.array([x[2] for x in cases], dtype=np.float32).view(np.uint32)
    got = oracle.ewise("fma", "f32", A, B, C)
    _check_exact("fma", "f32", [A, B, C], got)


def test_fma_f32_matches_libm_fmaf():
    libm = ctypes.CDLL(ctypes.util.find_library("m"))
    libm.fmaf.restype = ctypes.c_float
    libm.fmaf.argtypes = [ctypes.c_float] * 3
    n = 20000
    a = np.concatenate([_finite_bits("f32", n, 31), _moderate_bits("f32", n, 32)])
    b = np.concatenate([_finite_bits("f32", n, 33), _moderate_bits("f32", n, 34)])
    c = np.concatenate([_finite_bits("f32", n, 35), _moderate_bits("f32", n, 36)])
    m = min(a.size, b.size, c.size)
    a, b, c = a[:m], b[:m], c[:m]
    got = oracle.ewise("fma", "f32", a, b, c)
    fa, fb, fc = a.view(np.float32), b.view(np.float32), c.view(np.float32)
    want = np.array([libm.fmaf(float(x), float(y), float(z)) for x, y, z in zip(fa, fb, fc)],
                    dtype=np.float32).view(np.uint32)
    assert _same(got, want, "f32")


# ------------------------------------------------------------------ exp

def test_exp_special_values():
    for dtype in ("f16", "bf16", "f32"):
        one = oracle.round_to(1.0, dtype)
        inf = oracle.round_to(float("inf"), dtype)
        z = oracle.round_to(0.0, dtype)
        ninf = oracle.round_to(float("-inf"), dtype)
        nz = oracle.round_to(-0.0, dtype)
        nan = oracle.round_to(float("nan"), dtype)
        a = np.array([z, nz, ninf, inf, nan], dtype=NPB[dtype])
        got = oracle.ewise("exp", dtype, a)
        assert list(got[:4]) == [one, one, 0, inf]
        assert oracle.is_nan(got[4:], dtype).all()


def _mp_exp_rounded(x, dtype, mpmath):
    # exp(x) overflows every format above 89 and underflows below -104:
    # the correctly rounded results there are exactly +inf and +0
    if x > 120:
        return _exact.POS_INF[dtype]
    if x < -120:
        return 0
    v = mpmath.exp(mpmath.mpf(float(x)))
    man, ex = v.man_exp
    z = Fraction(int(man)) * (Fraction(2) ** int(ex))
    return _exact.round_exact(z, dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_exp_16bit_exhaustive_vs_mpmath(dtype):
    """Within the 1-ulp bound of the correctly rounded value everywhere."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    a = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = _exact.decode(a, dtype)
    keep = np.isfinite(vals)
    a = a[keep]
    got = oracle.ewise("exp", dtype, a)
    worst = 0
    for x_bits, g in zip(a, got):
        want = _mp_exp_rounded(_exact.decode(np.array([x_bits]), dtype)[0], dtype, mpmath)
        d = int(oracle.ulp_distance(np.array([g]), np.array([want]), dtype)[0])
        worst = max(worst, d)
    assert worst <= oracle.EXP_ULP_BOUND[dtype]


def test_exp_f32_vs_mpmath():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    rng = np.random.default_rng(17)
    x = np.concatenate([rng.uniform(-103, 88.7, 6000), rng.uniform(-1, 1, 2000),
                        rng.uniform(-8, 8, 2000)]).astype(np.float32)
    a = x.view(np.uint32)
    got = oracle.ewise("exp", "f32", a)
    worst = 0
    for xv, g in zip(x, got):
        want = _mp_exp_rounded(float(xv), "f32", mpmath)
        worst = max(worst, int(oracle.ulp_distance(np.array([g]), np.array([want]), "f32")[0]))
    assert worst <= 1   # well inside the 2-ulp bound
