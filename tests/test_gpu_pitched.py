"""Pitched rows: [rows, cols] views whose rows start `pitch` elements apart
(the tensor-map strides of TVM docs "copy_async -> tma", "Algorithm" step
3).  Every variant computes the oracle's result on the view and leaves the
padding between rows untouched."""

import zlib

import numpy as np
import pytest

import oracle
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu

SENTINEL = {"f32": 0x7FBADBAD, "f16": 0x7DAD, "bf16": 0x7FAD}
ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _pitched(bits, dtype, pitch):
    """A device [rows, pitch] buffer holding `bits` in its first cols
    columns and sentinels in the rest, and the [rows, cols] view."""
    rows, cols = bits.shape
    full = np.full((rows, pitch), SENTINEL[dtype], dtype=bits.dtype)
    full[:, :cols] = bits
    buf = to_dev(full, dtype)
    return buf, buf[:, :cols]


def _padding_intact(buf, dtype, cols):
    b = bits_of(buf, dtype)
    return bool(np.all(b[:, cols:] == SENTINEL[dtype]))


CASES = {"f32": (45, 100, 108, (8, 32)), "f16": (33, 200, 216, (16, 64)), "bf16": (70, 128, 192, (32, 128))}


@pytest.mark.parametrize("variant", ["tma", "tma_rank3", "tma_mixed", "ldgsts", "sync"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("op", ["add", "fma", "exp"])
def test_pitched_ewise(tsx, variant, dtype, op):
    rows, cols, pitch, box = CASES[dtype]
    try:
        tsx.query(dtype, rows, cols, box, 3, variant, op, pitch=pitch)
    except tsx.TsxError:
        pytest.skip("declined on the host (rank 3 needs whole atoms per row)")
    seed = zlib.crc32(f"pitch/{variant}/{dtype}/{op}".encode())
    ins = [random_bits(dtype, (rows, cols), seed + k) for k in range(ARITY[op])]
    want = oracle.ewise(op, dtype, *ins)
    views = [_pitched(x, dtype, pitch) for x in ins]
    obuf, out = _pitched(np.zeros((rows, cols), dtype=ins[0].dtype), dtype, pitch)
    with tsx.Plan(dtype, rows, cols, box=box, stages=3, variant=variant, pitch=pitch) as plan:
        plan.ewise(op, *[v for _, v in views], out=out)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare(op, dtype, bits_of(out, dtype), want, f"{variant} {dtype} {op}")
    assert _padding_intact(obuf, dtype, cols)
    for (buf, _), x in zip(views, ins):
        assert np.array_equal(bits_of(buf, dtype)[:, :cols], x) and _padding_intact(buf, dtype, cols)


def test_pitched_accumulate_and_row_sums(tsx):
    dtype, rows, cols, pitch, box = "f32", 45, 100, 108, (8, 32)
    a = random_bits(dtype, (rows, cols), 7, finite_fraction=1.0)
    o0 = random_bits(dtype, (rows, cols), 8, finite_fraction=1.0)
    _, va = _pitched(a, dtype, pitch)
    obuf, out = _pitched(o0, dtype, pitch)
    with tsx.Plan(dtype, rows, cols, box=box, stages=3, pitch=pitch) as plan:
        plan.ewise("copy", va, out=out, accumulate=True)
        sums = plan.reduce_rows("copy", va)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("add", dtype, bits_of(out, dtype), oracle.ewise("add", dtype, a, o0), "accumulate")
    assert _padding_intact(obuf, dtype, cols)
    exact, abs_sums = oracle.rowsum("copy", dtype, a)
    err = np.abs(sums.cpu().numpy().astype(np.float64) - exact)
    assert np.all(err <= oracle.summation_error_bound(cols, abs_sums) * (1 + 1e-9) + 1e-30)


def test_pitched_view_must_match_the_plan(tsx):
    rows, cols, pitch = 16, 64, 96
    buf = torch.zeros(rows, pitch, device="cuda")
    with tsx.Plan("f32", rows, cols, box=(8, 32), stages=2, pitch=pitch) as plan:
        with pytest.raises(tsx.TsxError):
            plan.ewise("copy", torch.zeros(rows, cols, device="cuda"), out=buf[:, :cols])   # dense input
        out = plan.ewise("copy", buf[:, :cols])          # out allocated with the plan's pitch
        assert out.stride(0) == pitch


@pytest.mark.parametrize("variant", ["tma", "tma_rank3"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pitched_row_sums(tsx, variant, dtype):
    """Row sums over a pitched view: the padding (NaN sentinels) must not
    leak into any sum; integer-valued rows make the sums exact."""
    rows, cols, pitch, box = {"f32": (45, 96, 128, (8, 32)), "bf16": (70, 128, 192, (32, 64))}[dtype]
    rng = np.random.default_rng(rows + cols)
    vals = rng.integers(-8, 8, (rows, cols)).astype(np.float32)
    if dtype == "f32":
        bits = vals.view(np.uint32)
    else:
        bits = (vals.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    buf, view = _pitched(bits, dtype, pitch)
    try:
        plan = tsx.Plan(dtype, rows, cols, box=box, stages=3, variant=variant, pitch=pitch)
    except tsx.TsxError:
        pytest.skip("declined on the host")
    with plan:
        got = plan.reduce_rows("copy", view).cpu().numpy().astype(np.float64)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    assert np.array_equal(got, vals.astype(np.float64).sum(axis=1))


@pytest.mark.parametrize("variant", ["tma", "tma_rank3"])
@pytest.mark.parametrize("op,tuning", [("copy", {"tile_order": 2}), ("copy", {"tile_order": 2, "dynamic_share": 30}),
                                       ("exp", {"store_split": 2}), ("fma", {"store_split": 2})])
def test_pitched_with_the_tile_order_and_split_knobs(tsx, variant, op, tuning):
    """The copy's dynamic tile order and the split stores on pitched rows:
    tile coordinates and box groups address the rows by the pitch."""
    dtype, rows, cols, pitch, box = "bf16", 70, 128, 192, (32, 128)
    try:
        q = tsx.query(dtype, rows, cols, box, 3, variant, op, pitch=pitch, tuning=tuning)
    except tsx.TsxError:
        pytest.skip("declined on the host")
    seed = zlib.crc32(f"pitch-knob/{variant}/{op}/{sorted(tuning.items())}".encode())
    ins = [random_bits(dtype, (rows, cols), seed + k) for k in range(ARITY[op])]
    want = oracle.ewise(op, dtype, *ins)
    views = [_pitched(x, dtype, pitch) for x in ins]
    obuf, out = _pitched(np.zeros((rows, cols), dtype=ins[0].dtype), dtype, pitch)
    with tsx.Plan(dtype, rows, cols, box=box, stages=3, variant=variant, pitch=pitch, tuning=tuning) as plan:
        info = plan.info(op)
        if "tile_order" in tuning:
            assert info["tile_order"] == 2
        if "store_split" in tuning:
            assert info["compute_groups"] == q["compute_groups"]
        plan.ewise(op, *[v for _, v in views], out=out)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare(op, dtype, bits_of(out, dtype), want, f"{variant} {op} {tuning}")
    assert _padding_intact(obuf, dtype, cols)
