"""The calls are stream-ordered and capturable: once a plan has made its
first call of an op (which sets up the launch), later calls can be captured
into a CUDA graph and replayed, with the same results as direct calls."""

import numpy as np
import pytest

import oracle
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


@pytest.mark.parametrize("variant", ["tma", "tma_rank3", "tma_mixed", "ldgsts", "sync"])
def test_ewise_in_a_cuda_graph(tsx, variant):
    rows, cols = 77, 1024
    a, b, c = (random_bits("f32", (rows, cols), 40 + k) for k in range(3))
    want_fma = oracle.ewise("fma", "f32", a, b, c)
    want_mul = oracle.ewise("mul", "f32", a, b)
    da, db, dc = to_dev(a, "f32"), to_dev(b, "f32"), to_dev(c, "f32")
    o1, o2 = torch.zeros_like(da), torch.zeros_like(da)
    with tsx.Plan("f32", rows, cols, box=(8, 128), stages=3, variant=variant) as plan:
        plan.ewise("fma", da, db, dc, out=o1)     # first calls: set up the launches
        plan.ewise("mul", da, db, out=o2)
        torch.cuda.synchronize()
        o1.zero_()
        o2.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.ewise("fma", da, db, dc, out=o1)
            plan.ewise("mul", da, db, out=o2)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("fma", "f32", bits_of(o1, "f32"), want_fma, f"{variant} fma replayed")
    compare("mul", "f32", bits_of(o2, "f32"), want_mul, f"{variant} mul replayed")


def test_row_sums_in_a_cuda_graph(tsx):
    rows, cols = 45, 5000
    rng = np.random.default_rng(9)
    a = rng.integers(-64, 64, (rows, cols)).astype(np.float32)
    da = to_dev(a.view(np.uint32), "f32")
    out = torch.zeros(rows, device="cuda")
    with tsx.Plan("f32", rows, cols, box=(1, 256), stages=3) as plan:
        plan.reduce_rows("copy", da, out=out)
        torch.cuda.synchronize()
        out.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.reduce_rows("copy", da, out=out)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    assert np.array_equal(out.cpu().numpy().astype(np.float64), a.astype(np.float64).sum(axis=1))
