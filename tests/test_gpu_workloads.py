"""The stated workloads at their full sizes, in the launch configuration the
benchmark times, against the oracle, every element of every output."""

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


@pytest.mark.parametrize("name", ["fma_128x1048576_f32", "exp_16384x16384_bf16"])
def test_workload_full_compare_at_full_size(tsx, name):
    """Every element of the two largest workloads, at every stated stage
    count, in the benchmark's launch configuration, against the oracle (run
    over every host core; the comparison too)."""
    w = ti.WORKLOADS[name]
    ins = w.inputs()
    want = oracle.ewise_parallel(w.op, w.dtype, *ins)
    dev = [to_dev(x, w.dtype) for x in ins]
    for stages in w.stages:
        with tsx.Plan(w.dtype, w.rows, w.cols, box=(w.box_rows, w.box_cols), stages=stages,
                      variant=w.variant) as plan:
            out = torch.zeros_like(dev[0])
            plan.ewise(w.op, *dev, out=out)
            torch.cuda.synchronize()
            assert plan.status() == tsx.TSX_OK
        bad, first = oracle.count_mismatches(w.op, w.dtype, bits_of(out, w.dtype), want)
        assert bad == 0, f"{name} S={stages}: {bad} of {w.elems} elements differ, first at {first}"
        del out
