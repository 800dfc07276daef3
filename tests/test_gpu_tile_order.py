"""The dynamic tile order of the TMA copy: a launch's CTAs claim tiles from
a counter that the launch's last CTA zeroes again, one counter per stream a
plan launches on.  Results must not depend on it: every test poisons the
outputs between launches, so that a tile left out (a counter not zeroed,
two launches sharing a counter) shows as a mismatch against the input."""

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
    seed = zlib.crc32(f"order/{dtype}/{op}/{rows}/{cols}/{tag}".encode())
    return [random_bits(dtype, (rows, cols), seed + k) for k in range(ARITY[op])]


def _poison(t):
    t.view(torch.uint8).fill_(0xA5)


@pytest.mark.parametrize("share", [100, 30])
@pytest.mark.parametrize("dtype,rows,cols,box,stages", [
    ("bf16", 1000, 3000, (32, 64), 2),
    ("f32", 77, 5000, (8, 128), 4),
    ("f16", 513, 1024, (16, 256), 3),
    ("f32", 9, 40, (8, 32), 1),        # 4 tiles: fewer tiles than CTAs
])
def test_repeated_launches_on_one_stream(tsx, dtype, rows, cols, box, stages, share):
    """Back-to-back copies by one plan on one stream (each with its own
    inputs), then another op on the same plan, then copies again."""
    op = "copy"
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, tuning={"tile_order": 2, "dynamic_share": share}) as plan:
        assert plan.info(op)["tile_order"] == 2
        runs = []
        for j in range(5):
            ins = _inputs(dtype, op, rows, cols, j)
            out = torch.empty((rows, cols), dtype=_gpu.TORCH_DTYPE[dtype], device="cuda")
            _poison(out)
            plan.ewise(op, *[to_dev(x, dtype) for x in ins], out=out)
            runs.append((ins, out))
        other = "sqrt"
        ins2 = _inputs(dtype, other, rows, cols, "other")
        out2 = torch.empty((rows, cols), dtype=_gpu.TORCH_DTYPE[dtype], device="cuda")
        _poison(out2)
        plan.ewise(other, *[to_dev(x, dtype) for x in ins2], out=out2)
        for j in range(5, 8):
            ins = _inputs(dtype, op, rows, cols, j)
            out = torch.empty((rows, cols), dtype=_gpu.TORCH_DTYPE[dtype], device="cuda")
            _poison(out)
            plan.ewise(op, *[to_dev(x, dtype) for x in ins], out=out)
            runs.append((ins, out))
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    for j, (ins, out) in enumerate(runs):
        compare(op, dtype, bits_of(out, dtype), oracle.ewise(op, dtype, *ins), f"launch {j}")
    compare(other, dtype, bits_of(out2, dtype), oracle.ewise(other, dtype, *ins2), f"then {other}")


def test_streams_sharing_a_plan(tsx):
    """Three streams launch one plan in turn without waiting for one
    another: each stream's launches take their own counter."""
    dtype, op, rows, cols = "f32", "copy", 300, 4096
    streams = [torch.cuda.Stream() for _ in range(3)]
    torch.cuda.synchronize()
    runs = []
    with tsx.Plan(dtype, rows, cols, box=(16, 128), stages=3, tuning={"tile_order": 2}) as plan:
        for j in range(12):
            s = streams[j % 3]
            ins = _inputs(dtype, op, rows, cols, j)
            with torch.cuda.stream(s):
                dev = [to_dev(x, dtype) for x in ins]
                out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
                _poison(out)
                plan.ewise(op, *dev, out=out, stream=s)
            runs.append((ins, out, dev))
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    for j, (ins, out, _) in enumerate(runs):
        compare(op, dtype, bits_of(out, dtype), oracle.ewise(op, dtype, *ins), f"stream {j % 3} launch {j}")


def test_more_streams_than_counters(tsx):
    """Past the plan's counter slots, launches on further streams take the
    static order; all results still match."""
    dtype, op, rows, cols = "bf16", "copy", 64, 2048
    ins = _inputs(dtype, op, rows, cols, "many")
    dev = [to_dev(x, dtype) for x in ins]
    want = oracle.ewise(op, dtype, *ins)
    outs = []
    with tsx.Plan(dtype, rows, cols, box=(16, 64), stages=2, tuning={"tile_order": 2}) as plan:
        for j in range(70):
            s = torch.cuda.Stream()
            out = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
            _poison(out)
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                plan.ewise(op, *dev, out=out, stream=s)
            outs.append(out)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    for j, out in enumerate(outs):
        compare(op, dtype, bits_of(out, dtype), want, f"stream {j}")


@pytest.mark.parametrize("variant", ["tma", "tma_rank3", "tma_promoted"])
def test_static_and_dynamic_orders_agree(tsx, variant):
    """Both orders copy every element on a ragged shape; the other ops take
    the static order whatever the knob says."""
    rows, cols = 515, 1096
    box = (16, 512) if variant == "tma_promoted" else (32, 64)
    for op in ARITY:
        ins = _inputs("f16", op, rows, cols, "agree")
        want = oracle.ewise(op, "f16", *ins)
        for order in (1, 2):
            try:
                plan = tsx.Plan("f16", rows, cols, box=box, stages=3, variant=variant,
                                tuning={"tile_order": order})
            except tsx.TsxError:
                pytest.skip(f"{variant} declines box {box}")
            with plan:
                assert plan.info(op)["tile_order"] == (order if op == "copy" else 1)
                out = plan.ewise(op, *[to_dev(x, "f16") for x in ins])
                torch.cuda.synchronize()
                assert plan.status() == tsx.TSX_OK
            compare(op, "f16", bits_of(out, "f16"), want, f"{variant} {op} order {order}")


def test_copy_accumulate_keeps_the_static_order(tsx):
    rows, cols = 200, 4096
    a = random_bits("f32", (rows, cols), 5, finite_fraction=1.0)
    with tsx.Plan("f32", rows, cols, box=(8, 128), stages=3, tuning={"tile_order": 2}) as plan:
        assert plan.info("copy")["tile_order"] == 2
        d = to_dev(a, "f32")
        out = d.clone()
        plan.ewise("copy", d, out=out, accumulate=True)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("add", "f32", bits_of(out, "f32"), oracle.ewise("add", "f32", a, a), "copy accumulated")


def test_planner_takes_the_dynamic_order_for_long_copies(tsx):
    """By default a copy launch takes the dynamic order only with at least
    16 tiles per CTA (the launch's grid decides; no tensors needed)."""
    with tsx.Plan("bf16", 16384, 16384, box=(128, 128), stages=3) as plan:
        info = plan.info("copy")
        assert info["tiles"] >= 16 * info["grid"] and info["tile_order"] == 2
        assert plan.info("exp")["tile_order"] == 1
    with tsx.Plan("f16", 1024, 8192, box=(64, 64), stages=3) as plan:
        info = plan.info("copy")
        assert info["tiles"] < 16 * info["grid"] and info["tile_order"] == 1
    with tsx.Plan("f16", 1024, 8192, box=(64, 64), stages=3, tuning={"tile_order": 2}) as plan:
        assert plan.info("copy")["tile_order"] == 2


def test_dynamic_order_copy_in_a_cuda_graph(tsx):
    """A launch captured into a graph takes the static order (a graph may be
    replayed on any stream, so no per-stream counter applies); replays copy
    every element, and direct launches on the capturing stream still use
    their counter."""
    rows, cols = 300, 4096
    ins = _inputs("f32", "copy", rows, cols, "graph")
    want = oracle.ewise("copy", "f32", *ins)
    d = to_dev(ins[0], "f32")
    out = torch.empty_like(d)
    with tsx.Plan("f32", rows, cols, box=(16, 128), stages=3, tuning={"tile_order": 2}) as plan:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            plan.ewise("copy", d, out=out, stream=s)   # first call: sets up the launch
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.ewise("copy", d, out=out)
        for _ in range(3):
            _poison(out)
            g.replay()
            torch.cuda.synchronize()
            compare("copy", "f32", bits_of(out, "f32"), want, "replayed copy")
        _poison(out)
        with torch.cuda.stream(s):
            plan.ewise("copy", d, out=out, stream=s)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("copy", "f32", bits_of(out, "f32"), want, "direct copy after the graph")
