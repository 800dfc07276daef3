"""Row sums over staged tiles (tsx_reduce_rows) against the oracle: within
the summation bound gamma(cols - 1) * sum |x| of the exact sum (plus the exp
bound where the terms themselves carry it), exact for integer-valued rows
(also when bands are cut between CTAs), repeatable bit for bit, and blind to
the zero-filled columns of ragged tiles."""

import zlib

import numpy as np
import pytest

import oracle
from tests import _gpu
from tests._gpu import to_dev, torch

pytestmark = pytest.mark.gpu

OPS = ["copy", "sqrt", "exp", "add", "mul", "fma"]
ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}
PRECISION = {"f16": 11, "bf16": 8, "f32": 24}


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _values(dtype, shape, seed, lo=-2.0, hi=2.0):
    rng = np.random.default_rng(seed)
    x = rng.uniform(lo, hi, int(np.prod(shape)))
    if dtype == "f32":
        return x.astype(np.float32).view(np.uint32).reshape(shape)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16).reshape(shape)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16).reshape(shape)


def _rowsum(tsx, dtype, rows, cols, box, stages, variant, op, ins, tuning=None):
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant, tuning=tuning) as plan:
        out = plan.reduce_rows(op, *[to_dev(x, dtype) for x in ins])
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    return out.cpu().numpy().astype(np.float64)


def _check(got, op, dtype, ins, cols, what):
    sums, abs_sums = oracle.rowsum(op, dtype, *ins)
    bound = oracle.summation_error_bound(cols, abs_sums)
    if op == "exp":
        # every term may be off by the exp bound in ulps of the element type
        bound = bound + abs_sums * oracle.EXP_ULP_BOUND[dtype] * 2.0 ** (1 - PRECISION[dtype])
    err = np.abs(got - sums)
    bad = np.nonzero(err > bound * (1 + 1e-9) + 1e-30)[0]
    assert bad.size == 0, f"{what}: row {bad[0]}: got {got[bad[0]]!r} want {sums[bad[0]]!r} bound {bound[bad[0]]!r}"


SHAPES = [(37, 700, (8, 128)), (5, 64, (4, 64)), (130, 1024, (16, 256)), (64, 2048, (32, 64))]


@pytest.mark.parametrize("variant", ["tma", "tma_rank3"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("op", OPS)
def test_rowsum_within_the_summation_bound(tsx, variant, dtype, op):
    n = 0
    for rows, cols, box in SHAPES:
        es = 4 if dtype == "f32" else 2
        if (cols * es) % 16:
            continue
        try:
            tsx.query(dtype, rows, cols, box, 3, variant, op)
        except tsx.TsxError:
            continue
        seed = zlib.crc32(f"rowsum/{variant}/{dtype}/{op}/{rows}/{cols}".encode())
        lo = 0.0 if op == "sqrt" else -2.0
        ins = [_values(dtype, (rows, cols), seed + k, lo=lo) for k in range(ARITY[op])]
        got = _rowsum(tsx, dtype, rows, cols, box, 3, variant, op, ins)
        _check(got, op, dtype, ins, cols, f"{variant} {dtype} {op} [{rows},{cols}] box {box}")
        n += 1
    assert n >= 2


def test_rowsum_integer_rows_are_exact(tsx):
    """Small integers: every partial sum is exact in fp32, so the result is
    the exact sum whatever the order -- no element is missed or doubled."""
    rows, cols = 45, 1000
    rng = np.random.default_rng(4)
    a = rng.integers(-64, 64, (rows, cols)).astype(np.float32)
    for box, stages in (((8, 128), 3), ((16, 64), 2), ((1, 256), 4)):
        got = _rowsum(tsx, "f32", rows, cols, box, stages, "tma", "copy", [a.view(np.uint32)])
        assert np.array_equal(got, a.astype(np.float64).sum(axis=1)), box


@pytest.mark.parametrize("rows,cols,box,ctas_per_sm", [
    (3, 65536, (1, 256), 0),       # 768 tiles: each band cut between about 256 CTAs
    (300, 4096, (1, 256), 0),      # 4800 tiles: ranges of several tiles end mid-band
    (300, 4096, (1, 256), 1),      # the same with one CTA per SM: other cut points
    (37, 5000, (8, 64), 2),        # ragged rows and columns, 8-row bands cut
    (1, 1 << 20, (1, 512), 0),     # one row over every CTA
])
def test_rowsum_bands_cut_between_ctas_are_exact(tsx, rows, cols, box, ctas_per_sm):
    """Integer-valued rows, so any lost or doubled share shows: the tile
    ranges of consecutive CTAs cut bands at many points, and the shares of a
    cut band are combined by its last arriving CTA."""
    rng = np.random.default_rng(rows * 7 + cols)
    a = rng.integers(-64, 64, (rows, cols)).astype(np.float32)
    want = a.astype(np.float64).sum(axis=1)
    for stages in (2, 4):
        got = _rowsum(tsx, "f32", rows, cols, box, stages, "tma", "copy", [a.view(np.uint32)],
                      tuning={"ctas_per_sm": ctas_per_sm})
        assert np.array_equal(got, want), (box, stages, np.nonzero(got != want)[0][:5])


def test_rowsum_cut_bands_repeat_bit_for_bit(tsx):
    rows, cols = 5, 300000
    a = _values("f16", (rows, cols), 8)
    with tsx.Plan("f16", rows, cols, box=(1, 256), stages=3) as plan:
        da = to_dev(a, "f16")
        runs = [plan.reduce_rows("exp", da).cpu().numpy().view(np.uint32) for _ in range(4)]
        assert plan.status() == tsx.TSX_OK
    for r in runs[1:]:
        assert np.array_equal(runs[0], r)
    _check(runs[0].view(np.float32).astype(np.float64), "exp", "f16", [a], cols, "cut bands")


def test_rowsum_ignores_the_padding_of_ragged_tiles(tsx):
    """exp of the zero fill would add 1 per padded element; the true sums
    here are tiny, so any leak shows."""
    rows, cols = 19, 200   # 200 = 3 * 64 + 8: the last column tile is mostly padding
    a = np.full((rows, cols), -30.0, dtype=np.float32)
    got = _rowsum(tsx, "f32", rows, cols, (8, 64), 2, "tma", "exp", [a.view(np.uint32)])
    assert np.all(got < 1e-8) and np.all(got > 0)


def test_rowsum_repeats_bit_for_bit(tsx):
    rows, cols = 64, 4096
    a = _values("bf16", (rows, cols), 5)
    with tsx.Plan("bf16", rows, cols, box=(8, 128), stages=4) as plan:
        da = to_dev(a, "bf16")
        r1 = plan.reduce_rows("exp", da).cpu().numpy()
        r2 = plan.reduce_rows("exp", da).cpu().numpy()
    assert np.array_equal(r1.view(np.uint32), r2.view(np.uint32))


def test_rowsum_edges_and_declines(tsx):
    with tsx.Plan("f32", 7, 0, box=(8, 32), stages=2) as plan:
        out = torch.full((7,), 3.0, device="cuda")
        plan.reduce_rows("copy", torch.empty(7, 0, device="cuda"), out=out)
        torch.cuda.synchronize()
        assert torch.all(out == 0)
    a = torch.rand(16, 64, device="cuda")
    for variant in ("ldgsts", "sync", "tma_mixed"):
        with tsx.Plan("f32", 16, 64, box=(8, 32), stages=2, variant=variant) as plan:
            with pytest.raises(tsx.TsxError) as ei:
                plan.reduce_rows("copy", a)
            assert ei.value.code == tsx.TSX_ERR_UNSUPPORTED
    with tsx.Plan("f32", 16, 64, box=(8, 32), stages=2) as plan:
        out = torch.empty(16, device="cuda")
        rc = tsx.tsx_reduce_rows(plan.handle, tsx.OPS["copy"] | tsx.TSX_ACCUMULATE, a.data_ptr(), None, None,
                                 out.data_ptr(), 0)
        assert rc == tsx.TSX_ERR_INVALID


def test_rowsum_launch_info(tsx):
    """TSX_ROW_SUMS asks tsx_plan_get_info for the row reduction's launch;
    the other entry points reject the flag."""
    with tsx.Plan("bf16", 300, 4096, box=(8, 128), stages=3) as plan:
        ew, rs = plan.info("exp"), plan.info("exp", row_sums=True)
        assert rs["block_threads"] == rs["threads"] + 32   # compute warps + the producer
        assert ew["block_threads"] == ew["threads"] + 64   # + producer and store warps
        assert 0 < rs["grid"] <= rs["tiles"] and rs["grid"] <= rs["ctas_per_sm"] * rs["sm_count"]
        a = torch.zeros(300, 4096, dtype=torch.bfloat16, device="cuda")
        out = torch.empty_like(a)
        s = torch.cuda.current_stream().cuda_stream
        assert tsx.tsx_ewise(plan.handle, tsx.OPS["exp"] | tsx.TSX_ROW_SUMS, a.data_ptr(), None, None,
                             out.data_ptr(), s) == tsx.TSX_ERR_INVALID
        sums = torch.empty(300, device="cuda")
        assert tsx.tsx_reduce_rows(plan.handle, tsx.OPS["exp"] | tsx.TSX_ROW_SUMS, a.data_ptr(), None, None,
                                   sums.data_ptr(), s) == tsx.TSX_ERR_INVALID
    with tsx.Plan("f32", 16, 64, box=(8, 32), stages=2, variant="sync") as plan:
        with pytest.raises(tsx.TsxError) as ei:
            plan.info("copy", row_sums=True)
        assert ei.value.code == tsx.TSX_ERR_UNSUPPORTED


def test_rowsum_wait_timeout_is_reported(tsx):
    """The producer is told to skip one tile's loads: the compute warps'
    bounded wait gives up, TSX_ERR_TIMEOUT is recorded, and the GPU stays
    usable."""
    rows, cols = 64, 1024
    a = _values("f32", (rows, cols), 6)
    bad = tsx.Plan("f32", rows, cols, box=(8, 128), stages=3, tuning={"timeout_ms": 50})
    bad.set_fault_tile(9)
    da = to_dev(a, "f32")
    try:
        bad.reduce_rows("copy", da)
        torch.cuda.synchronize()
        assert bad.status() == tsx.TSX_ERR_TIMEOUT
    finally:
        bad.close()
    got = _rowsum(tsx, "f32", rows, cols, (8, 128), 3, "tma", "copy", [a])
    _check(got, "copy", "f32", [a], cols, "after the timeout")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_rowsum_exp_meets_every_16bit_input(tsx, dtype):
    """The row reduction evaluates exp its own way (halving and squaring), so
    it is checked on every 16-bit input: row r is bit pattern r followed by
    seven -inf.  exp(-inf) = 0 adds nothing, so the row sum is the reduction's
    exp of pattern r rounded into the element type and widened exactly; it
    must be within the exp bound of the oracle's (NaN for NaN)."""
    rows, cols = 1 << 16, 8
    neg_inf = 0xFC00 if dtype == "f16" else 0xFF80
    a = np.full((rows, cols), neg_inf, dtype=np.uint16)
    a[:, 0] = np.arange(rows, dtype=np.uint32).astype(np.uint16)
    for box, stages in (((256, 8), 2), ((64, 8), 3)):
        got = _rowsum(tsx, dtype, rows, cols, box, stages, "tma", "exp", [a]).astype(np.float32)
        nan = np.isnan(got)
        fin = got[~nan]
        if dtype == "bf16":
            bits = (got.view(np.uint32) >> 16).astype(np.uint16)
            assert np.array_equal((bits[~nan].astype(np.uint32) << 16), fin.view(np.uint32)), "not a widened bf16"
            bits[nan] = 0x7FC0
        else:
            h = got.astype(np.float16)
            assert np.array_equal(h[~nan].astype(np.float32).view(np.uint32), fin.view(np.uint32)), \
                "not a widened fp16"
            bits = h.view(np.uint16).copy()
            bits[nan] = 0x7E00
        want = oracle.ewise("exp", dtype, a[:, 0])
        d = oracle.ulp_distance(bits, want, dtype)
        bad = np.flatnonzero(d > oracle.EXP_ULP_BOUND[dtype])
        assert bad.size == 0, f"box {box}: {bad.size} inputs off, first {int(a[bad[0], 0]):#06x}"


def test_rowsum_launch_shape(tsx):
    """fp32 row sums take enough CTAs for about 128 KB of stages per SM (96
    KB for sqrt and exp; three to six) of 384 threads in all; 16-bit ones
    about 768 threads per SM over every CTA that fits."""
    with tsx.Plan("f32", 128, 1 << 20, box=(8, 128), stages=4) as plan:
        fma = plan.info("fma", row_sums=True)      # 12 KB stages: three CTAs
        add = plan.info("add", row_sums=True)      # 8 KB stages: four
        copy = plan.info("copy", row_sums=True)    # 4 KB stages: eight wanted, six at most
        exp = plan.info("exp", row_sums=True)      # 4 KB stages, 96 KB: six
    assert (fma["ctas_per_sm"], fma["threads"]) == (3, 128)
    assert (add["ctas_per_sm"], add["threads"]) == (4, 96)
    assert (copy["ctas_per_sm"], copy["threads"]) == (6, 64)
    assert (exp["ctas_per_sm"], exp["threads"]) == (6, 64)
    with tsx.Plan("f32", 128, 1 << 20, box=(8, 256), stages=6) as plan:
        big = plan.info("fma", row_sums=True)      # 144 KB of stages: the one CTA that fits
    assert (big["ctas_per_sm"], big["threads"]) == (1, 192)
    with tsx.Plan("bf16", 16384, 16384, box=(32, 256), stages=2) as plan:
        h = plan.info("exp", row_sums=True)
    assert h["ctas_per_sm"] * h["threads"] <= 768 and h["ctas_per_sm"] >= 3
