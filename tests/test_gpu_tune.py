"""tsx_plan_tune: the op's candidate launch shapes timed on the caller's
operands, the fastest kept for the plan's later calls.  The shape never
changes a result, so every test checks the tuned output and a later call
against the oracle, and that the launch kept is one of the candidates."""

import zlib

import pytest

import oracle
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu

ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _inputs(dtype, op, rows, cols, tag):
    seed = zlib.crc32(f"tune/{dtype}/{op}/{rows}/{cols}/{tag}".encode())
    return [random_bits(dtype, (rows, cols), seed + k) for k in range(ARITY[op])]


def _candidates():
    shapes = set()
    for ctas in range(1, 9):
        for total in (256, 512):
            shapes.add((ctas, max(32, total // ctas // 32 * 32)))
    return shapes


@pytest.mark.parametrize("dtype,rows,cols,box,stages,variant,op", [
    ("bf16", 2048, 4096, (32, 128), 3, "tma", "exp"),
    ("f32", 64, 1 << 17, (8, 128), 4, "tma", "fma"),
    ("f16", 1000, 3008, (16, 64), 2, "tma_rank3", "add"),
    ("f32", 257, 8200, (8, 128), 6, "tma_mixed", "mul"),
    ("bf16", 513, 8192, (64, 64), 3, "tma", "copy"),
    ("f32", 300, 4096, (16, 64), 2, "ldgsts", "sqrt"),
    ("f32", 70, 8192, (8, 512), 2, "tma_promoted", "exp"),
])
def test_tune_keeps_a_candidate_and_exact_results(tsx, dtype, rows, cols, box, stages, variant, op):
    ins = _inputs(dtype, op, rows, cols, "main")
    want = oracle.ewise(op, dtype, *ins)
    dev = [to_dev(x, dtype) for x in ins]
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant) as plan:
        planner = plan.info(op)
        out = torch.empty_like(dev[0])
        out.view(torch.uint8).fill_(0xA5)
        chosen = plan.tune(op, *dev, out=out, launches=3)
        torch.cuda.synchronize()
        compare(op, dtype, bits_of(out, dtype), want, f"tuned output {variant} {op}")
        shape = (chosen["ctas_per_sm"], chosen["threads"])
        assert shape == (planner["ctas_per_sm"], planner["threads"]) or shape[1] in {t for _, t in _candidates()}
        after = plan.info(op)
        assert (after["ctas_per_sm"], after["threads"], after["grid"]) == (chosen["ctas_per_sm"], chosen["threads"],
                                                                          chosen["grid"])
        again = torch.empty_like(dev[0])
        again.view(torch.uint8).fill_(0x5A)
        plan.ewise(op, *dev, out=again)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare(op, dtype, bits_of(again, dtype), want, f"call after tuning {variant} {op}")


def test_tune_rejects_aliasing_and_accumulate(tsx):
    rows, cols = 64, 4096
    a, b = (to_dev(x, "f32") for x in _inputs("f32", "add", rows, cols, "alias"))
    with tsx.Plan("f32", rows, cols, box=(8, 128), stages=3) as plan:
        with pytest.raises(tsx.TsxError) as e:
            plan.tune("add", a, b, out=a)
        assert e.value.code == tsx.TSX_ERR_INVALID
        with pytest.raises(tsx.TsxError) as e:
            plan.tune(tsx.OPS["add"] | tsx.TSX_ACCUMULATE, a, b, out=torch.zeros_like(a))
        assert e.value.code == tsx.TSX_ERR_INVALID
        with pytest.raises(tsx.TsxError) as e:
            plan.tune("add", a, None, out=torch.zeros_like(a))   # add needs b
        assert e.value.code == tsx.TSX_ERR_INVALID


def test_tune_keeps_a_forced_shape(tsx):
    rows, cols = 128, 8192
    ins = _inputs("bf16", "exp", rows, cols, "forced")
    with tsx.Plan("bf16", rows, cols, box=(32, 128), stages=3, tuning={"threads": 96, "ctas_per_sm": 2}) as plan:
        before = plan.info("exp")
        chosen = plan.tune("exp", to_dev(ins[0], "bf16"))
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    assert (chosen["threads"], chosen["ctas_per_sm"]) == (before["threads"], before["ctas_per_sm"]) == (96, 2)
    # a forced store side is kept while the shape is tuned
    with tsx.Plan("bf16", rows, cols, box=(32, 128), stages=3, tuning={"store_warps": 2, "store_lag": 0}) as plan:
        chosen = plan.tune("exp", to_dev(ins[0], "bf16"), launches=2)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    assert (chosen["store_warps"], chosen["store_lag"]) == (2, 0)


def test_tuned_launch_in_a_cuda_graph(tsx):
    """Calls after tuning only launch, so they can be captured and replayed."""
    rows, cols = 256, 8192
    ins = _inputs("f32", "fma", rows, cols, "graph")
    want = oracle.ewise("fma", "f32", *ins)
    dev = [to_dev(x, "f32") for x in ins]
    with tsx.Plan("f32", rows, cols, box=(8, 128), stages=4) as plan:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            out = torch.empty_like(dev[0])
            plan.tune("fma", *dev, out=out, launches=2, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.ewise("fma", *dev, out=out)
        out.view(torch.uint8).fill_(0xA5)
        g.replay()
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("fma", "f32", bits_of(out, "f32"), want, "replayed after tuning")


def test_tune_on_an_empty_tensor(tsx):
    with tsx.Plan("f16", 0, 256, box=(8, 64), stages=2) as plan:
        a = torch.empty((0, 256), dtype=torch.float16, device="cuda")
        plan.tune("sqrt", a, out=torch.empty_like(a))
