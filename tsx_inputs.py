"""Seeded synthetic inputs for the tile-elementwise streaming path.

This module is shared by the tests, the benchmark and the CPU oracle's
callers.  It holds no arithmetic of the method itself (no elementwise op, no
tiling, no pipeline): it only turns a (seed, tensor index, element index)
triple into an input value.

Generator.  Element ``i`` (row-major) of tensor ``t`` (a = 0, b = 1, c = 2)
under seed ``s`` is built from the ``i``-th output of SplitMix64 (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
started from the state ``key(s, t) = mix64(GOLDEN * (256 * s + t + 1))``.
The ``i``-th output of SplitMix64 from state ``k`` is
``mix64(k + GOLDEN * (i + 1))`` with the published finaliser ``mix64``.  Being
counter-based, any element can be regenerated on its own, which the
full-size sampled parity checks use.

Distributions (the pages print no values, so these are the plainest reading
of the workloads' stated distributions):

* uniform[lo, hi): ``u = (z >> 40) * 2**-24`` (24 random bits),
  ``x = lo + (hi - lo) * u`` in double, then rounded to nearest-even into the
  element type; if rounding lands on ``hi`` the largest representable value
  below ``hi`` is taken so the interval stays half-open.  For the
  power-of-two ranges used here ``x`` is exact in fp32.
* N(0, 1): Box-Muller in double from the outputs ``2i`` and ``2i + 1`` of the
  same stream (53-bit uniforms, the first one shifted into (0, 1]), then
  rounded to nearest-even into the element type.

Arrays are returned as numpy arrays holding the element bits: ``float32``
for fp32 and ``uint16`` for fp16 / bf16 (bf16 has no numpy type).
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_CHUNK = 1 << 20

DTYPES = ("f16", "bf16", "f32")
ELEM_SIZE = {"f16": 2, "bf16": 2, "f32": 4}


def _mix64(z: np.ndarray, tmp: np.ndarray | None = None) -> np.ndarray:
    """SplitMix64 output finaliser, in place on a uint64 array (wrapping)."""
    if tmp is None:
        tmp = np.empty_like(z)
    np.right_shift(z, np.uint64(30), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, np.uint64(_M1), out=z)
    np.right_shift(z, np.uint64(27), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, np.uint64(_M2), out=z)
    np.right_shift(z, np.uint64(31), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    return z


def stream_key(seed: int, tensor: int) -> int:
    z = np.array([(GOLDEN * (256 * seed + tensor + 1)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return int(_mix64(z)[0])


def raw64(seed: int, tensor: int, index: np.ndarray) -> np.ndarray:
    """Outputs ``index`` (uint64 array) of the stream for (seed, tensor)."""
    z = np.array(index, dtype=np.uint64, copy=True)
    np.add(z, np.uint64(1), out=z)
    np.multiply(z, np.uint64(GOLDEN), out=z)
    np.add(z, np.uint64(stream_key(seed, tensor)), out=z)
    return _mix64(z)


def _round_f16(x: np.ndarray) -> np.ndarray:
    # numpy's float64 -> float16 cast rounds to nearest even
    return x.astype(np.float16).view(np.uint16)


def _round_bf16(x: np.ndarray) -> np.ndarray:
    # torch's float32 -> bfloat16 cast rounds to nearest even; x is first
    # narrowed to float32 (exact for every range used by the workloads)
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x.astype(np.float32)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _below(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Largest value strictly below the (positive or negative) value ``bits``."""
    if dtype == "f32":
        return np.nextafter(bits, np.float32(-np.inf), dtype=np.float32)
    out = bits.copy()
    neg = (bits & 0x8000) != 0
    is_pz = bits == 0
    out[~neg & ~is_pz] -= 1
    out[neg] += 1
    out[is_pz] = 0x8001  # below +0 is the smallest negative subnormal
    return out


def _to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "f16":
        return _round_f16(x)
    if dtype == "bf16":
        return _round_bf16(x)
    raise ValueError(dtype)


def _bits_value(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return bits.astype(np.float64)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    wide = bits.astype(np.uint32) << np.uint32(16)
    return wide.view(np.float32).astype(np.float64)


def uniform_at(index: np.ndarray, dtype: str, lo: float, hi: float, seed: int, tensor: int) -> np.ndarray:
    """uniform[lo, hi) values at flat ``index`` positions."""
    z = raw64(seed, tensor, index)
    u = (z >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    x = lo + (hi - lo) * u
    out = _to_dtype(x, dtype)
    hit = _bits_value(out, dtype) >= hi
    if hit.any():
        out[hit] = _below(out[hit], dtype)
    return out


def normal_at(index: np.ndarray, dtype: str, seed: int, tensor: int) -> np.ndarray:
    """N(0, 1) values at flat ``index`` positions (Box-Muller)."""
    idx = np.asarray(index, dtype=np.uint64)
    z1 = raw64(seed, tensor, idx * np.uint64(2))
    z2 = raw64(seed, tensor, idx * np.uint64(2) + np.uint64(1))
    u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (z2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return _to_dtype(x, dtype)


def _workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill(out: np.ndarray, fn) -> np.ndarray:
    """Fill the flat array ``out`` chunk by chunk with ``fn(index_chunk)``.

    Chunks are independent (the generator is counter-based), so they are
    filled by a thread pool; numpy releases the GIL inside its loops.
    """
    n = out.shape[0]
    bounds = [(s, min(n, s + _CHUNK)) for s in range(0, n, _CHUNK)]

    def one(b):
        s, e = b
        out[s:e] = fn(np.arange(s, e, dtype=np.uint64))

    if len(bounds) <= 1:
        for b in bounds:
            one(b)
        return out
    with ThreadPoolExecutor(max_workers=_workers()) as pool:
        list(pool.map(one, bounds))
    return out


@dataclass(frozen=True)
class Dist:
    kind: str  # "uniform" | "normal"
    lo: float = 0.0
    hi: float = 1.0

    def at(self, index: np.ndarray, dtype: str, seed: int, tensor: int) -> np.ndarray:
        if self.kind == "uniform":
            return uniform_at(index, dtype, self.lo, self.hi, seed, tensor)
        if self.kind == "normal":
            return normal_at(index, dtype, seed, tensor)
        raise ValueError(self.kind)


def generate(rows: int, cols: int, dtype: str, dist: Dist, seed: int, tensor: int) -> np.ndarray:
    """A full [rows, cols] input tensor (element bits, see module docstring)."""
    np_dtype = np.float32 if dtype == "f32" else np.uint16
    flat = np.empty(rows * cols, dtype=np_dtype)
    _fill(flat, lambda idx: dist.at(idx, dtype, seed, tensor))
    return flat.reshape(rows, cols)


def all_bit_patterns_16() -> np.ndarray:
    """Every 16-bit pattern once, as a [256, 256] uint16 tensor."""
    return np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(256, 256)


# --------------------------------------------------------------------------
# The workloads.  Names say what each one is; sizes are the stated ones.
# --------------------------------------------------------------------------

OP_ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    rows: int
    cols: int
    op: str
    dist: Dist
    seed: int
    box_rows: int
    box_cols: int
    stages: tuple = (2,)
    variant: str = "tma"
    note: str = field(default="", compare=False)
    bench_stages: int = 0     # the stage count the benchmark uses (0: the last stated one)

    @property
    def n_in(self) -> int:
        return OP_ARITY[self.op]

    @property
    def elems(self) -> int:
        return self.rows * self.cols

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes read plus bytes written by one pass: (n_in + 1) * elems * es."""
        return (self.n_in + 1) * self.elems * ELEM_SIZE[self.dtype]

    def with_rows(self, rows: int) -> "Workload":
        """The same workload over its first ``rows`` rows (a smaller case)."""
        from dataclasses import replace

        return replace(self, rows=int(rows))

    @property
    def default_stages(self) -> int:
        return self.bench_stages or self.stages[-1]

    def inputs(self) -> list:
        return [generate(self.rows, self.cols, self.dtype, self.dist, self.seed, t) for t in range(self.n_in)]

    def inputs_range(self, start: int, n: int) -> list:
        """Input values at the flat positions start .. start + n - 1, filled
        chunk by chunk on a thread pool as ``generate`` does."""
        np_dtype = np.float32 if self.dtype == "f32" else np.uint16
        out = []
        for t in range(self.n_in):
            flat = np.empty(n, dtype=np_dtype)
            _fill(flat, lambda idx, t=t: self.dist.at(idx + np.uint64(start), self.dtype, self.seed, t))
            out.append(flat)
        return out

    def inputs_at(self, flat_index: np.ndarray) -> list:
        """Input values at the given flat positions only (for sampled checks)."""
        return [self.dist.at(flat_index, self.dtype, self.seed, t) for t in range(self.n_in)]


WORKLOADS = {
    w.name: w
    for w in (
        Workload("roundtrip_8x256_f16", "f16", 8, 256, "copy", Dist("uniform", -1.0, 1.0), 0, 8, 256, (1,),
                 note="one CTA, one 8x256 fp16 tile through TMA with 128-B swizzle and one mbarrier"),
        Workload("sqrt_500x4096_f32", "f32", 500, 4096, "sqrt", Dist("uniform", 0.0, 4.0), 1, 32, 32, (2,),
                 note="ragged 500-row tail"),
        Workload("sqrt_500x4096_f16_ldgsts", "f16", 500, 4096, "sqrt", Dist("uniform", 0.0, 4.0), 1, 128, 32, (2,),
                 variant="ldgsts", note="the cp.async variant of the same shape"),
        Workload("add_1024x8192_f16", "f16", 1024, 8192, "add", Dist("normal"), 2, 64, 64, (2, 3, 4)),
        Workload("fma_128x1048576_f32", "f32", 128, 1 << 20, "fma", Dist("uniform", -2.0, 2.0), 3, 8, 128, (4,),
                 note="stage tile 8x128 = four 8x32 TMA boxes per operand"),
        Workload("exp_16384x16384_bf16", "bf16", 16384, 16384, "exp", Dist("uniform", -8.0, 8.0), 4, 128, 128, (2, 3, 4),
                 note="128x128 stage tile = two 128x64 TMA boxes", bench_stages=3),
    )
}
