"""Helpers for the GPU tests: host bits <-> CUDA tensors, comparisons."""

from __future__ import annotations

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
NP_BITS = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def to_dev(bits: np.ndarray, dtype: str):
    """Element bits (numpy) -> a CUDA tensor of the element type."""
    arr = np.ascontiguousarray(bits)
    if dtype == "f32":
        t = torch.from_numpy(arr.view(np.float32))
    else:
        t = torch.from_numpy(arr.view(np.int16)).view(TORCH_DTYPE[dtype])
    return t.to("cuda")


def bits_of(t, dtype: str) -> np.ndarray:
    """A tensor's element bits as numpy (uint16 / uint32)."""
    c = t.detach().contiguous().cpu()
    if dtype == "f32":
        return c.numpy().view(np.uint32)
    return c.view(torch.int16).numpy().view(np.uint16)


def compare(op: str, dtype: str, got: np.ndarray, want: np.ndarray, what: str = ""):
    """Bit-exact (copy bitwise; NaN == NaN otherwise), or the exp ulp bound."""
    got = np.asarray(got).reshape(-1)
    want = np.asarray(want).reshape(-1).view(NP_BITS[dtype])
    assert got.shape == want.shape
    if op == "copy":
        bad = np.nonzero(got != want)[0]
    elif op == "exp":
        d = oracle.ulp_distance(got, want, dtype)
        bad = np.nonzero(d > oracle.EXP_ULP_BOUND[dtype])[0]
    else:
        bad = np.nonzero(~oracle.same_value(got, want, dtype))[0]
    if bad.size:
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} of {got.size} elements differ; first at {i}: "
                             f"got {int(got[i]):#x} want {int(want[i]):#x}")


def random_bits(dtype: str, shape, seed: int, finite_fraction: float = 0.7) -> np.ndarray:
    """Random element bits: a mix of arbitrary patterns (NaN, inf,
    subnormals included) and moderate finite values."""
    rng = np.random.default_rng(seed)
    n = int(np.prod(shape))
    top = 1 << (32 if dtype == "f32" else 16)
    raw = rng.integers(0, top, size=n, dtype=np.uint64).astype(NP_BITS[dtype])
    moderate = rng.standard_normal(n) * 2.0 ** rng.integers(-4, 4, n)
    if dtype == "f32":
        mod = moderate.astype(np.float32).view(np.uint32)
    elif dtype == "f16":
        mod = moderate.astype(np.float16).view(np.uint16)
    else:
        mod = (moderate.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    pick = rng.random(n) < finite_fraction
    return np.where(pick, mod, raw).reshape(shape)
