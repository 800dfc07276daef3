"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element, on small ragged shapes over every variant, op, dtype and stage
count (bit-exact; exp within its ulp bound)."""

import itertools
import zlib

import numpy as np
import pytest

import oracle
import tsx_inputs as ti
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


def run_and_check(tsx, dtype, rows, cols, box, stages, variant, op, seed, ins=None):
    if ins is None:
        ins = [random_bits(dtype, (rows, cols), seed + 101 * k) for k in range(ARITY[op])]
    want = oracle.ewise(op, dtype, *ins)
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant) as plan:
        out = plan.ewise(op, *[to_dev(x, dtype) for x in ins])
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare(op, dtype, bits_of(out, dtype), want,
            f"{variant} {op} {dtype} [{rows},{cols}] box {box} S={stages}")


# shapes with ragged row and column tails, single tiles, single rows; every
# one keeps the row pitch a multiple of 16 bytes for the TMA variants
SHAPES = {
    "f32": [(1, 64, (8, 32)), (7, 96, (8, 32)), (33, 160, (16, 64)), (100, 256, (32, 128)), (5, 8, (4, 8)),
            (300, 64, (300, 32))],
    "f16": [(1, 64, (8, 64)), (7, 136, (8, 64)), (33, 200, (16, 128)), (100, 256, (64, 64)), (5, 8, (4, 8)),
            (130, 128, (130, 64))],
    "bf16": [(1, 64, (8, 64)), (9, 72, (8, 64)), (65, 192, (64, 128)), (100, 256, (32, 256)), (5, 8, (4, 8)),
             (260, 64, (260, 64))],
}


@pytest.mark.parametrize("variant", ["tma", "tma_rank3", "tma_mixed", "tma_promoted", "ldgsts", "sync"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("op", OPS)
def test_parity_small_shapes(tsx, variant, dtype, op):
    n = 0
    for (rows, cols, box), stages in itertools.product(SHAPES[dtype], (1, 2, 3, 4)):
        try:
            tsx.query(dtype, rows, cols, box, stages, variant, op)
        except tsx.TsxError as e:
            # declined on the host: stages that do not fit in shared memory,
            # or (rank 3) atoms that are not whole / 1024-byte aligned
            assert e.code == tsx.TSX_ERR_UNSUPPORTED
            continue
        seed = zlib.crc32(f"{variant}/{dtype}/{op}/{rows}/{cols}/{stages}".encode())
        run_and_check(tsx, dtype, rows, cols, box, stages, variant, op, seed=seed)
        n += 1
    assert n >= 8


@pytest.mark.parametrize("variant", ["tma", "tma_mixed"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_every_swizzle_mode(tsx, variant, dtype):
    """Inner boxes of 16, 32, 48, 64, 128 bytes and rows of several 128-byte
    atoms: every swizzle mode of the tensor map (none, 32, 64, 128 bytes).
    In the mixed variant b is read from global memory at the positions the
    staged vectors hold, so a wrong reading of the swizzle pairs the wrong
    elements and fails here."""
    es = 4 if dtype == "f32" else 2
    n = 0
    for row_bytes in (16, 32, 48, 64, 128, 256, 384):
        box_cols = row_bytes // es
        for box_rows, rows in ((8, 45), (3, 10), (16, 33)):
            cols = 3 * box_cols + (16 // es if box_cols > 16 // es else 0)
            for op in ("add", "fma"):
                run_and_check(tsx, dtype, rows, cols, (box_rows, box_cols), 3, variant, op,
                              seed=zlib.crc32(f"swz/{variant}/{dtype}/{row_bytes}/{box_rows}/{op}".encode()))
                n += 1
    assert n == 42


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_promoted_wide_tiles(tsx, dtype):
    """Tile rows wider than 256 elements in one box: the tensor map counts
    in 4- or 8-byte elements (element-type promotion), with ragged column
    and row tails."""
    es = 4 if dtype == "f32" else 2
    n = 0
    for box_cols in (256, 512, 768, 1024):
        for rows, cols, box_rows in ((45, 2 * box_cols + 8 * (8 // es), 8), (30, box_cols, 8)):
            try:
                q = tsx.query(dtype, rows, cols, (box_rows, box_cols), 3, "tma_promoted", "fma")
            except tsx.TsxError:
                continue
            assert q["tma_elem_bytes"] >= es
            for op in ("fma", "exp"):
                run_and_check(tsx, dtype, rows, cols, (box_rows, box_cols), 3, "tma_promoted", op,
                              seed=zlib.crc32(f"promo/{dtype}/{box_cols}/{rows}/{op}".encode()))
            n += 1
    assert n >= 4


@pytest.mark.parametrize("stages", [1, 2, 3, 5, 8])
def test_many_tiles_per_cta(tsx, stages):
    """More tiles than CTAs, so every CTA cycles through its stages many
    times (parity flips), with a ragged last row tile."""
    rows, cols = 1000, 2048
    for variant, op in (("tma", "fma"), ("tma", "copy"), ("ldgsts", "add"), ("tma_rank3", "mul"), ("tma_mixed", "fma")):
        run_and_check(tsx, "f32", rows, cols, (8, 128), stages, variant, op, seed=stages)


def test_all_16bit_patterns_every_unary_op(tsx):
    """Every fp16 / bf16 bit pattern through copy, sqrt and exp."""
    a = ti.all_bit_patterns_16()
    for dtype, op, variant in itertools.product(("f16", "bf16"), ("copy", "sqrt", "exp"), ("tma", "ldgsts")):
        run_and_check(tsx, dtype, 256, 256, (64, 64), 3, variant, op, 0, ins=[a])


@pytest.mark.parametrize("variant", ["tma", "tma_rank3"])
def test_roundtrip_8x256_f16(tsx, variant):
    """One CTA, one 8x256 fp16 tile, one mbarrier, TMA in and out: the tile
    comes back bit for bit (TVM "copy_async -> tma", Demonstration program)."""
    w = ti.WORKLOADS["roundtrip_8x256_f16"]
    a = w.inputs()[0]
    with tsx.Plan("f16", 8, 256, box=(8, 256), stages=1, variant=variant) as plan:
        info = plan.info("copy")
        assert info["grid"] == 1 and info["tiles"] == 1
        assert info["loads_per_operand"] == (1 if variant == "tma_rank3" else 4)
        out = plan.ewise("copy", to_dev(a, "f16"))
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    assert np.array_equal(bits_of(out, "f16"), a)


def test_empty_tensors_are_a_no_op(tsx):
    for rows, cols in ((0, 64), (16, 0), (0, 0)):
        with tsx.Plan("f32", rows, cols, box=(8, 32), stages=2) as plan:
            a = torch.empty(rows, cols, device="cuda")
            out = torch.full((rows, cols), 7.0, device="cuda")
            plan.ewise("sqrt", a, out=out)
            torch.cuda.synchronize()
            assert plan.status() == tsx.TSX_OK
