"""CPU oracle for tile-elementwise streaming -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library (``pipelined_elementwise_streaming_gb300``)
never does, and this package never imports the library: the two share no
code.  Inputs come from ``tsx_inputs``, which holds no arithmetic of the
method.

Contents
* ``ewise``: the per-element definitions (C, ``tsx_oracle.c``), evaluated in
  fp64 and rounded once into the element type.
* ``ulp_distance`` / ``same_value``: the comparisons the parity tests use.
* ``ewise_parallel`` / ``count_mismatches``: the same routine and the same
  comparisons, cut into ranges over every host core, for full-size checks.
* ``structure``: the integer plans the pages fix -- the ``[outer, threads,
  vec]`` partition, the box split with its expect_tx bytes, the tensor-map
  arguments and the prologue / main / epilogue schedule.

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (printed values, library routines, exact rational
arithmetic, brute force).  The swizzled shared-memory layout is not modelled
here at all (the pages print no swizzled address): no oracle function stands
for it.  The CUDA path's handling of it is checked end to end instead, by the
copy round trip and by the mixed-load variant, whose directly loaded operand
pairs with the wrong elements unless the swizzle is read correctly.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import structure  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tsx_oracle.c")
_LIB = os.path.join(_HERE, "libtsx_oracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra"]

DTYPE_CODE = {"f16": 0, "bf16": 1, "f32": 2}
OP_CODE = {"copy": 0, "sqrt": 1, "exp": 2, "add": 3, "mul": 4, "fma": 5}
OP_ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}
NP_BITS = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``tsx_oracle.c`` into ``libtsx_oracle.so`` if it is stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.tsxo_value.restype = ctypes.c_double
            L.tsxo_value.argtypes = [ctypes.c_uint32, ctypes.c_int]
            L.tsxo_round.restype = ctypes.c_uint32
            L.tsxo_round.argtypes = [ctypes.c_double, ctypes.c_int]
            L.tsxo_add_round_odd.restype = ctypes.c_double
            L.tsxo_add_round_odd.argtypes = [ctypes.c_double, ctypes.c_double]
            L.tsxo_ewise.restype = ctypes.c_int
            L.tsxo_ewise.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64] + [ctypes.c_void_p] * 4
            L.tsxo_decode.restype = ctypes.c_int
            L.tsxo_decode.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            _lib = L
    return _lib


def _bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """View an array as the element bits the C side expects (contiguous)."""
    want = NP_BITS[dtype]
    x = np.ascontiguousarray(x)
    if x.dtype.itemsize != np.dtype(want).itemsize:
        raise TypeError(f"{dtype} operand has itemsize {x.dtype.itemsize}")
    return x.view(want)


def ewise(op: str, dtype: str, a, b=None, c=None, out=None) -> np.ndarray:
    """out = op(a[, b[, c]]) element by element; returns element bits.

    Operands are numpy arrays of element bits (``float32`` or ``uint32`` for
    fp32, ``uint16`` / ``float16`` for the 16-bit types), all the same shape.
    ``out``, if given, is a contiguous array of that shape and element size
    that receives the result (it is returned viewed as element bits).
    """
    arity = OP_ARITY[op]
    ops = [a, b, c][:arity]
    if any(o is None for o in ops) or any(o is not None for o in [a, b, c][arity:]):
        raise ValueError(f"{op} takes exactly {arity} operand(s)")
    shape = np.shape(a)
    ops = [_bits(o, dtype) for o in ops]
    if any(o.shape != shape for o in ops):
        raise ValueError("operand shapes differ")
    if out is None:
        out = np.empty(shape, dtype=NP_BITS[dtype])
    else:
        if out.shape != shape or not out.flags.c_contiguous:
            raise ValueError("out must be a contiguous array of the operands' shape")
        out = out.view(NP_BITS[dtype])
    ptrs = [o.ctypes.data for o in ops] + [None] * (3 - arity)
    rc = lib().tsxo_ewise(DTYPE_CODE[dtype], OP_CODE[op], int(out.size), *ptrs, out.ctypes.data)
    if rc != 0:
        raise RuntimeError("tsxo_ewise rejected its arguments")
    return out


# --------------------------------------------------------------------------
# Running the oracle on every host core
# --------------------------------------------------------------------------

def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _ranges(n: int, parts: int):
    parts = max(1, min(parts, n)) if n else 1
    return [(k * n // parts, (k + 1) * n // parts) for k in range(parts)]


def ewise_parallel(op: str, dtype: str, a, b=None, c=None, threads: int | None = None, out=None) -> np.ndarray:
    """``ewise`` with the elements cut into contiguous ranges, one call of the
    same C routine per range on a pool of host threads (ctypes releases the
    GIL for the call).  Elements are independent, so the result is the one
    ``ewise`` gives; only the wall time changes."""
    from concurrent.futures import ThreadPoolExecutor

    arity = OP_ARITY[op]
    ops = [_bits(o, dtype).reshape(-1) for o in [a, b, c][:arity] if o is not None]
    if len(ops) != arity:
        raise ValueError(f"{op} takes exactly {arity} operand(s)")
    shape = np.shape(a)
    flat_out = np.empty(ops[0].size, dtype=NP_BITS[dtype]) if out is None else out.view(NP_BITS[dtype]).reshape(-1)
    threads = threads or host_cores()
    # ranges much smaller than the data so that uneven cores still finish together
    parts = max(1, min(4 * threads, ops[0].size // (1 << 16) or 1))

    def one(r):
        s, e = r
        ewise(op, dtype, *[o[s:e] for o in ops], out=flat_out[s:e])

    with ThreadPoolExecutor(max_workers=threads) as pool:
        list(pool.map(one, _ranges(ops[0].size, parts)))
    return flat_out.reshape(shape)


def count_mismatches(op: str, dtype: str, got, want, threads: int | None = None):
    """Compare device bits with the oracle's under the parity rule of ``op``
    (copy bitwise; exp within ``EXP_ULP_BOUND`` ulps; otherwise bit-exact with
    NaN equal to NaN), in ranges on a pool of host threads.  Returns
    ``(mismatches, first mismatching flat index or -1)``."""
    from concurrent.futures import ThreadPoolExecutor

    g = np.asarray(got).reshape(-1).view(NP_BITS[dtype])
    w = np.asarray(want).reshape(-1).view(NP_BITS[dtype])
    if g.size != w.size:
        raise ValueError("sizes differ")
    threads = threads or host_cores()

    def one(r):
        s, e = r
        x, y = g[s:e], w[s:e]
        if op == "copy":
            bad = x != y
        elif op == "exp":
            bad = ulp_distance(x, y, dtype) > EXP_ULP_BOUND[dtype]
        else:
            bad = ~same_value(x, y, dtype)
        idx = np.flatnonzero(bad)
        return int(idx.size), (s + int(idx[0])) if idx.size else -1

    parts = max(1, min(4 * threads, g.size // (1 << 18) or 1))
    with ThreadPoolExecutor(max_workers=threads) as pool:
        res = list(pool.map(one, _ranges(g.size, parts)))
    total = sum(n for n, _ in res)
    first = next((f for n, f in res if n), -1)
    return total, first


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """The exact values (float64) of an array of element bits."""
    b = _bits(bits, dtype)
    out = np.empty(b.shape, dtype=np.float64)
    if lib().tsxo_decode(DTYPE_CODE[dtype], int(b.size), b.ctypes.data, out.ctypes.data) != 0:
        raise RuntimeError("tsxo_decode rejected its arguments")
    return out


def rowsum(op: str, dtype: str, a, b=None, c=None):
    """Row sums of the element-type results x = op(a, b, c) of a [rows, cols]
    problem: the reduction the nvFuser page schedules over staged tiles
    ("Testing Setup", Reduction and InnerPersistent).

    Returns ``(sums, abs_sums)``, float64 arrays of length rows: ``sums[r]``
    is the exact sum of row r rounded once to float64 (``math.fsum``), and
    ``abs_sums[r]`` the exact sum of |x| rounded the same way, which scales
    the error bound of any floating-point summation order.
    """
    import math

    x = decode(ewise(op, dtype, a, b, c), dtype)
    x = x.reshape(x.shape[0], -1)
    sums = np.array([math.fsum(row) for row in x], dtype=np.float64)
    abs_sums = np.array([math.fsum(np.abs(row)) for row in x], dtype=np.float64)
    return sums, abs_sums


def summation_error_bound(n_terms: int, abs_sum: np.ndarray, unit_roundoff: float = 2.0 ** -24) -> np.ndarray:
    """The forward error bound of a sum of n terms in a floating-point format
    with unit roundoff u, in any order of additions: gamma(n-1) * sum |x_i|,
    gamma(k) = k u / (1 - k u) (N. J. Higham, "Accuracy and Stability of
    Numerical Algorithms", 2nd ed., section 4.2)."""
    k = max(0, n_terms - 1)
    gamma = k * unit_roundoff / (1.0 - k * unit_roundoff)
    return gamma * np.asarray(abs_sum, dtype=np.float64)


def value(bits: int, dtype: str) -> float:
    return lib().tsxo_value(int(bits), DTYPE_CODE[dtype])


def round_to(x: float, dtype: str) -> int:
    return int(lib().tsxo_round(float(x), DTYPE_CODE[dtype]))


def add_round_odd(x: float, y: float) -> float:
    return lib().tsxo_add_round_odd(float(x), float(y))


# --------------------------------------------------------------------------
# Comparisons
# --------------------------------------------------------------------------

_SIGN = {"f16": 0x8000, "bf16": 0x8000, "f32": 0x80000000}
_EXP_MASK = {"f16": 0x7C00, "bf16": 0x7F80, "f32": 0x7F800000}
_FRAC_MASK = {"f16": 0x03FF, "bf16": 0x007F, "f32": 0x007FFFFF}


def is_nan(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.asarray(bits).astype(np.int64)
    return ((b & _EXP_MASK[dtype]) == _EXP_MASK[dtype]) & ((b & _FRAC_MASK[dtype]) != 0)


def ordinal(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Map bit patterns to integers that are monotone in the value.

    Adjacent representable values differ by 1; +0 and -0 both map to 0.
    """
    b = np.asarray(bits).astype(np.int64)
    mag = b & (_SIGN[dtype] - 1)
    return np.where((b & _SIGN[dtype]) != 0, -mag, mag)


def ulp_distance(x_bits: np.ndarray, y_bits: np.ndarray, dtype: str) -> np.ndarray:
    """|ord(x) - ord(y)|; 0 where both are NaN, a huge value where one is."""
    x_nan, y_nan = is_nan(x_bits, dtype), is_nan(y_bits, dtype)
    d = np.abs(ordinal(x_bits, dtype) - ordinal(y_bits, dtype))
    d = np.where(x_nan & y_nan, 0, d)
    return np.where(x_nan ^ y_nan, np.iinfo(np.int64).max, d)


def same_value(x_bits: np.ndarray, y_bits: np.ndarray, dtype: str) -> np.ndarray:
    """Bitwise equality, except that any NaN equals any NaN."""
    x = np.asarray(x_bits).astype(np.int64)
    y = np.asarray(y_bits).astype(np.int64)
    both_nan = is_nan(x, dtype) & is_nan(y, dtype)
    return (x == y) | both_nan


# Tolerances the parity tests apply: bit-exact everywhere except exp, which
# is bounded in ulps of the element type against the fp64 reference.
EXP_ULP_BOUND = {"f32": 2, "f16": 1, "bf16": 1}
