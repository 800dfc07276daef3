"""The stated workloads at their full sizes, in the launch configuration the
benchmark times, against the oracle: in full where the oracle takes seconds,
on sampled elements (plus every element of the ragged edges) otherwise."""

import numpy as np
import pytest

import oracle
import tsx_inputs as ti
from tests import _gpu
from tests._gpu import bits_of, compare, to_dev, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _run(tsx, w, ins, stages, variant=None):
    with tsx.Plan(w.dtype, w.rows, w.cols, box=(w.box_rows, w.box_cols), stages=stages,
                  variant=variant or w.variant) as plan:
        out = plan.ewise(w.op, *[to_dev(x, w.dtype) for x in ins])
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    return bits_of(out, w.dtype)


@pytest.mark.parametrize("name", ["sqrt_500x4096_f32", "sqrt_500x4096_f16_ldgsts", "add_1024x8192_f16"])
def test_workload_full_compare(tsx, name):
    w = ti.WORKLOADS[name]
    ins = w.inputs()
    want = oracle.ewise(w.op, w.dtype, *ins)
    for stages in w.stages:
        compare(w.op, w.dtype, _run(tsx, w, ins, stages), want, f"{name} S={stages}")


def test_sqrt_500x4096_f32_all_variants(tsx):
    w = ti.WORKLOADS["sqrt_500x4096_f32"]
    ins = w.inputs()
    want = oracle.ewise(w.op, w.dtype, *ins)
    for variant in ("tma_rank3", "ldgsts", "sync"):
        compare(w.op, w.dtype, _run(tsx, w, ins, 2, variant), want, f"{variant}")


def _sample_index(w, n=1 << 20, seed=0):
    """Random positions plus every element of the first and last tile rows
    and of the last tile column."""
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, w.elems, size=n, dtype=np.int64)]
    r_last = (w.rows - 1) // w.box_rows * w.box_rows
    for r0, r1 in ((0, min(w.rows, w.box_rows)), (r_last, w.rows)):
        idx.append(np.arange(r0 * w.cols, r1 * w.cols, dtype=np.int64))
    c_last = (w.cols - 1) // w.box_cols * w.box_cols
    rows = np.arange(w.rows, dtype=np.int64)[:, None]
    idx.append((rows * w.cols + np.arange(c_last, w.cols, dtype=np.int64)[None, :]).reshape(-1))
    return np.unique(np.concatenate(idx))


@pytest.mark.parametrize("name", ["fma_128x1048576_f32", "exp_16384x16384_bf16"])
def test_workload_sampled_compare(tsx, name):
    w = ti.WORKLOADS[name]
    ins = w.inputs()
    idx = _sample_index(w)
    want = oracle.ewise(w.op, w.dtype, *[x.reshape(-1)[idx] for x in ins])
    # the sampled inputs are the generator's values at those positions
    regen = w.inputs_at(idx.astype(np.uint64))
    for x, r in zip(ins, regen):
        assert np.array_equal(x.reshape(-1)[idx], r)
    for stages in w.stages:
        got = _run(tsx, w, ins, stages).reshape(-1)[idx]
        compare(w.op, w.dtype, got, want, f"{name} S={stages}")
