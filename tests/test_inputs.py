"""The seeded input generator: determinism, counter-based access, ranges."""

import numpy as np
import pytest

import tsx_inputs as ti


def test_splitmix64_reference_outputs():
    """SplitMix64 from state 0: the first outputs of the published
    generator (Vigna's reference splitmix64.c seeded with 0)."""
    z = ti.raw64(0, 0, np.arange(3, dtype=np.uint64))  # not state 0: check the finaliser directly
    state = np.array([ti.GOLDEN, 2 * ti.GOLDEN % (1 << 64), 3 * ti.GOLDEN % (1 << 64)], dtype=np.uint64)
    out = ti._mix64(state.copy())
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert z.dtype == np.uint64


def test_deterministic_and_counter_based():
    w = ti.WORKLOADS["sqrt_500x4096_f32"]
    a1 = ti.generate(50, 64, "f32", w.dist, w.seed, 0)
    a2 = ti.generate(50, 64, "f32", w.dist, w.seed, 0)
    assert np.array_equal(a1, a2)
    idx = np.array([0, 7, 1234, 50 * 64 - 1], dtype=np.uint64)
    assert np.array_equal(a1.reshape(-1)[idx.astype(np.int64)], w.dist.at(idx, "f32", w.seed, 0))
    b = ti.generate(50, 64, "f32", w.dist, w.seed, 1)
    assert not np.array_equal(a1, b)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("lo,hi", [(-1.0, 1.0), (0.0, 4.0), (-2.0, 2.0), (-8.0, 8.0)])
def test_uniform_range_half_open(dtype, lo, hi):
    x = ti.generate(64, 1024, dtype, ti.Dist("uniform", lo, hi), 9, 0)
    v = ti._bits_value(x.reshape(-1), dtype)
    assert v.min() >= lo and v.max() < hi
    assert abs(v.mean() - (lo + hi) / 2) < 0.02 * (hi - lo)


def test_uniform_clamp_below_hi():
    # 16-bit rounding of values just under hi lands on hi; the clamp moves it below
    idx = np.arange(1 << 16, dtype=np.uint64)
    x = ti.uniform_at(idx, "bf16", -8.0, 8.0, 4, 0)
    assert ti._bits_value(x, "bf16").max() < 8.0


def test_normal_moments():
    x = ti.generate(256, 1024, "f16", ti.Dist("normal"), 2, 0)
    v = ti._bits_value(x.reshape(-1), "f16")
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


def test_workload_table():
    w = ti.WORKLOADS["fma_128x1048576_f32"]
    assert w.n_in == 3 and w.algorithmic_bytes == 4 * 128 * (1 << 20) * 4
    w = ti.WORKLOADS["exp_16384x16384_bf16"]
    assert w.algorithmic_bytes == 2 * 16384 * 16384 * 2
