"""The tuning knobs (tsx_tuning, given at plan creation) change launch
shapes and timing only, never results: every setting is checked against the
oracle on ragged shapes, and the store lag also against the schedule model
through the traced kernel."""

import zlib

import pytest

import oracle
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch
from tests.test_gpu_schedule_trace import _check_all

pytestmark = pytest.mark.gpu

ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}
CASES = [("f32", "fma", 77, 1000, (8, 128)), ("bf16", "exp", 130, 2056, (32, 64)), ("f16", "add", 33, 520, (16, 256))]


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _run(tsx, dtype, op, rows, cols, box, stages, variant="tma", tuning=None):
    seed = zlib.crc32(f"knob/{dtype}/{op}/{rows}/{cols}/{box}/{stages}/{variant}".encode())
    ins = [random_bits(dtype, (rows, cols), seed + k) for k in range(ARITY[op])]
    want = oracle.ewise(op, dtype, *ins)
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant, tuning=tuning) as plan:
        out = plan.ewise(op, *[to_dev(x, dtype) for x in ins])
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
        info = plan.info(op)
    compare(op, dtype, bits_of(out, dtype), want, f"{variant} {dtype} {op} box {box} S={stages}")
    return info


@pytest.mark.parametrize("knob,values", [
    ("store_lag", [0, 1, 2, 3]),
    ("store_warps", [1, 2]),
    ("role_wait", [1, 2]),
    ("l2_promotion", [0, 1, 2, 3]),
    ("store_split", [1, 2]),
    ("threads", [32, 96, 256, 960]),
    ("ctas_per_sm", [1, 2, 3]),
])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_knobs_leave_results_unchanged(tsx, knob, values, case):
    dtype, op, rows, cols, box = CASES[case]
    for v in values:
        for variant in ("tma", "tma_rank3"):
            for stages in (2, 4):
                try:
                    q = tsx.query(dtype, rows, cols, box, stages, variant, op, tuning={knob: v})
                except tsx.TsxError:
                    continue
                info = _run(tsx, dtype, op, rows, cols, box, stages, variant, tuning={knob: v})
                if knob == "threads":
                    assert info["threads"] == q["threads"] == v
                if knob == "ctas_per_sm":
                    assert info["ctas_per_sm"] <= v
                if knob in ("store_lag", "store_warps", "role_wait"):
                    assert info[knob] == q[knob] == v
                if knob == "store_split":
                    assert info["compute_groups"] == q["compute_groups"] <= v
                if knob == "l2_promotion":
                    assert info["l2_promotion"] == q["l2_promotion"] == v


@pytest.mark.parametrize("lag", [0, 2, 3])
@pytest.mark.parametrize("stages", [2, 4])
def test_store_lag_follows_the_schedule_model(tsx, lag, stages):
    """With a forced store lag one store warp releases tile i - lag (lag
    capped at S - 1) after tile i's stores; the trace must still satisfy the
    model (two store warps and the copy's dynamic order:
    test_gpu_schedule_trace.py)."""
    tiles = 1000
    rows, cols = 8 * tiles, 32
    a, b = random_bits("f32", (rows, cols), lag), random_bits("f32", (rows, cols), lag + 1)
    with tsx.Plan("f32", rows, cols, box=(8, 32), stages=stages, tuning={"store_lag": lag, "ctas_per_sm": 1,
                                                                                  "store_warps": 1}) as plan:
        plan.enable_trace(256)
        out = plan.ewise("add", to_dev(a, "f32"), to_dev(b, "f32"))
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
        trace = plan.trace()
    compare("add", "f32", bits_of(out, "f32"), oracle.ewise("add", "f32", a, b), "traced add")
    _check_all(trace, tiles, stages, min(lag, stages - 1), "add", 1, 1, 0)


@pytest.mark.parametrize("dtype,rows,cols,box,stages,op,shape", [
    ("f32", 128, 1 << 20, (8, 128), 4, "fma", (5, 64)),     # every CTA the registers leave
    ("f32", 128, 1 << 20, (8, 128), 6, "fma", (4, 64)),     # every CTA shared memory leaves
    ("f32", 128, 1 << 20, (8, 128), 8, "fma", (3, 64)),
    ("f32", 128, 1 << 20, (8, 128), 6, "add", (4, 64)),     # 96 KB of 24 KB rings
    ("bf16", 16384, 16384, (64, 64), 6, "add", (2, 128)),   # 96 KB of 48 KB rings
    ("bf16", 16384, 16384, (64, 128), 4, "mul", (1, 256)),  # 1.5 rounds down
])
def test_mixed_variant_launch_shape(tsx, dtype, rows, cols, box, stages, op, shape):
    """The mixed variant's default launch: compute threads that just hold b a
    tile ahead; fma keeps every CTA that fits, add and mul enough for about
    96 KB of stages per SM.  The same defaults on a ragged shape match the
    oracle."""
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant="tma_mixed") as plan:
        info = plan.info(op)
    assert (info["ctas_per_sm"], info["threads"]) == shape
    _run(tsx, dtype, op, 3 * box[0] + 5, 7 * box[1] + 8, box, stages, "tma_mixed")


@pytest.mark.parametrize("dtype,rows,cols,box,op,shape", [
    ("bf16", 16384, 16384, (128, 128), "exp", (2, 256)),   # 128 KB of 64 KB rings
    ("bf16", 16384, 16384, (64, 128), "exp", (4, 128)),    # 128 KB of 32 KB rings
    ("bf16", 16384, 16384, (128, 128), "copy", (2, 128)),  # 96 KB of 64 KB rings: 1.5 rounds up
    ("bf16", 16384, 16384, (32, 128), "add", (3, 160)),    # 96 KB of 32 KB rings
    ("f32", 128, 1 << 20, (8, 128), "fma", (6, 64)),       # 144 KB of 24 KB rings
    ("f32", 128, 1 << 20, (8, 128), "add", (6, 64)),       # 96 KB of 16 KB rings
])
def test_two_stage_ring_launch_shape(tsx, dtype, rows, cols, box, op, shape):
    """Two-stage rings on long streams: CTAs for the op's target of stage
    bytes per SM, sharing 512 compute threads (256 for copy).  The same
    launch shape on a ragged shape (too few tiles for the rule, so given as
    knobs) matches the oracle."""
    with tsx.Plan(dtype, rows, cols, box=box, stages=2) as plan:
        info = plan.info(op)
    assert (info["ctas_per_sm"], info["threads"]) == shape
    _run(tsx, dtype, op, 3 * box[0] + 5, 7 * box[1] + 8, box, 2,
         tuning={"ctas_per_sm": shape[0], "threads": shape[1]})
