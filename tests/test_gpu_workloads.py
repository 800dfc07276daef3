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


_INPUTS = {}


def _full_inputs(w):
    """The workload's input tensors (seeded per tensor index, so an op of
    arity n takes the first n), generated once per module."""
    have = _INPUTS.get(w.name, [])
    if len(have) < w.n_in:
        have = w.inputs()
        _INPUTS[w.name] = have
    return have[: w.n_in]


@pytest.mark.parametrize("name,op,box,stages,variant", [
    ("exp_16384x16384_bf16", "exp", (64, 128), 2, "tma"),        # two-stage ring: 4 CTAs of 128 threads
    ("exp_16384x16384_bf16", "add", (32, 128), 2, "tma"),        # two-stage ring: 3 CTAs of 160
    ("exp_16384x16384_bf16", "exp", (64, 64), 4, "tma"),         # small sqrt / exp stages
    ("exp_16384x16384_bf16", "mul", (64, 128), 4, "tma_mixed"),  # mixed add / mul: 1 CTA of 256
    ("fma_128x1048576_f32", "fma", (8, 128), 2, "tma"),          # two-stage ring: 6 CTAs of 64
    ("fma_128x1048576_f32", "add", (8, 128), 4, "tma"),          # add / mul on a long stream
    ("fma_128x1048576_f32", "fma", (8, 128), 6, "tma_mixed"),    # mixed fma: every CTA that fits
])
def test_planner_launch_shapes_at_full_size(tsx, name, op, box, stages, variant):
    """The launch shapes the planner's rules choose on long streams, on the
    full-size inputs, every element against the oracle."""
    from dataclasses import replace

    w = replace(ti.WORKLOADS[name], op=op, box_rows=box[0], box_cols=box[1])
    ins = _full_inputs(w)
    want = oracle.ewise_parallel(op, w.dtype, *ins)
    dev = [to_dev(x, w.dtype) for x in ins]
    with tsx.Plan(w.dtype, w.rows, w.cols, box=box, stages=stages, variant=variant) as plan:
        out = torch.zeros_like(dev[0])
        plan.ewise(op, *dev, out=out)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
        info = plan.info(op)
    bad, first = oracle.count_mismatches(op, w.dtype, bits_of(out, w.dtype), want)
    assert bad == 0, f"{name} {op} {box} S={stages} {variant} ({info['ctas_per_sm']} CTAs of " \
                     f"{info['threads']}): {bad} of {w.elems} elements differ, first at {first}"
