"""TMA reduce-store (TSX_ACCUMULATE): out = out + op(a, b, c), the sum added
by the TMA unit in global memory ("copy_async -> tma", table under "How
inputs change the algorithm": s2g with a reduce op).  The expected value is
the oracle's add of the oracle's op result and the initial out."""

import zlib

import numpy as np
import pytest

import oracle
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu

OPS = ["copy", "sqrt", "exp", "add", "mul", "fma"]
ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _moderate(dtype, shape, seed, positive=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(int(np.prod(shape))) * 2.0 ** rng.integers(-6, 6, int(np.prod(shape)))
    if positive:
        x = np.abs(x)
    if dtype == "f32":
        return x.astype(np.float32).view(np.uint32).reshape(shape)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16).reshape(shape)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16).reshape(shape)


def _run_acc(tsx, dtype, rows, cols, box, stages, variant, op, ins, out0):
    d_out = to_dev(out0, dtype)
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant) as plan:
        plan.ewise(op, *[to_dev(x, dtype) for x in ins], out=d_out, accumulate=True)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    return bits_of(d_out, dtype)


SHAPES = [(37, 384, (8, 128)), (130, 256, (64, 64)), (5, 64, (16, 32))]


@pytest.mark.parametrize("variant", ["tma", "tma_rank3"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("op", OPS)
def test_accumulate_matches_oracle(tsx, variant, dtype, op):
    n = 0
    for rows, cols, box in SHAPES:
        try:
            tsx.query(dtype, rows, cols, box, 3, variant, op)
        except tsx.TsxError:
            continue
        seed = zlib.crc32(f"acc/{variant}/{dtype}/{op}/{rows}".encode())
        ins = [_moderate(dtype, (rows, cols), seed + k, positive=(op == "sqrt")) for k in range(ARITY[op])]
        out0 = _moderate(dtype, (rows, cols), seed + 7, positive=(op == "exp"))
        got = _run_acc(tsx, dtype, rows, cols, box, 3, variant, op, ins, out0)
        want = oracle.ewise("add", dtype, oracle.ewise(op, dtype, *ins), out0)
        if op == "exp":
            # exp is within its bound of the exact value and both addends are
            # non-negative, so the rounded sum is within one ulp more
            d = oracle.ulp_distance(got.reshape(-1), want.reshape(-1), dtype)
            assert int(d.max()) <= oracle.EXP_ULP_BOUND[dtype] + 1
        else:
            compare(op, dtype, got, want, f"{variant} {dtype} {op} [{rows},{cols}]")
        n += 1
    assert n >= 2


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_accumulate_special_values(tsx, dtype):
    """Arbitrary bit patterns (NaN, infinities, subnormals, signed zeros) in
    both the op result and the value accumulated into."""
    rows, cols = 64, 256
    a = random_bits(dtype, (rows, cols), 501, finite_fraction=0.3)
    out0 = random_bits(dtype, (rows, cols), 502, finite_fraction=0.3)
    got = _run_acc(tsx, dtype, rows, cols, (16, 64), 2, "tma", "copy", [a], out0)
    want = oracle.ewise("add", dtype, a, out0)
    compare("add", dtype, got, want, f"{dtype} special values")


def test_accumulate_into_an_input(tsx):
    """out is a: out = out + sqrt(out)."""
    dtype, rows, cols = "f32", 40, 512
    a = _moderate(dtype, (rows, cols), 9, positive=True)
    d = to_dev(a, dtype)
    with tsx.Plan(dtype, rows, cols, box=(8, 128), stages=4) as plan:
        plan.ewise("sqrt", d, out=d, accumulate=True)
        torch.cuda.synchronize()
    want = oracle.ewise("add", dtype, oracle.ewise("sqrt", dtype, a), a)
    compare("add", dtype, bits_of(d, dtype), want, "out is a")


def test_accumulate_declines_outside_the_tma_variants(tsx):
    a = torch.rand(16, 64, device="cuda")
    for variant in ("ldgsts", "sync", "tma_mixed"):
        with tsx.Plan("f32", 16, 64, box=(8, 32), stages=2, variant=variant) as plan:
            with pytest.raises(tsx.TsxError) as ei:
                plan.ewise("copy", a, out=a.clone(), accumulate=True)
            assert ei.value.code == tsx.TSX_ERR_UNSUPPORTED
