"""Seeded random plans against the oracle: dtype, shape (ragged in both
dimensions), box, stage count, variant and op drawn at random, every plan
the host accepts run once and compared element by element (bit-exact, or
the exp ulp bound).  Shapes stay small so the whole sweep takes seconds."""

import numpy as np
import pytest

import oracle
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu

ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}
VARIANTS = ["tma", "tma_rank3", "tma_mixed", "tma_promoted", "ldgsts", "sync"]
ES = {"f16": 2, "bf16": 2, "f32": 4}


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _draw(rng):
    dtype = ["f16", "bf16", "f32"][rng.integers(3)]
    es = ES[dtype]
    unit = 16 // es                                   # elements per 16 bytes
    cols = int(unit * rng.integers(1, 160))           # rows a whole number of 16-byte units
    rows = int(rng.integers(1, 300))
    box_cols = int(unit * 2 ** rng.integers(0, 5))    # 16 .. 256 bytes of elements
    box_cols = min(box_cols, 256)
    box_rows = int(rng.choice([1, 2, 3, 5, 8, 16, 32, 64, 100, 256]))
    stages = int(rng.integers(1, 5))
    variant = VARIANTS[rng.integers(len(VARIANTS))]
    op = list(ARITY)[rng.integers(len(ARITY))]
    return dtype, rows, cols, (box_rows, box_cols), stages, variant, op


@pytest.mark.parametrize("seed", range(8))
def test_random_plans_match_the_oracle(tsx, seed):
    rng = np.random.default_rng(1000 + seed)
    ran = 0
    for _ in range(40):
        dtype, rows, cols, box, stages, variant, op = _draw(rng)
        try:
            tsx.query(dtype, rows, cols, box, stages, variant, op)
        except tsx.TsxError:
            continue
        ins = [random_bits(dtype, (rows, cols), int(rng.integers(1 << 30))) for _ in range(ARITY[op])]
        want = oracle.ewise(op, dtype, *ins)
        with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant) as plan:
            dev = [to_dev(x, dtype) for x in ins]
            out = plan.ewise(op, *dev)
            torch.cuda.synchronize()
            assert plan.status() == tsx.TSX_OK
        compare(op, dtype, bits_of(out, dtype), want,
                f"{variant} {dtype} {op} [{rows},{cols}] box {box} S={stages}")
        ran += 1
    assert ran >= 10, ran
