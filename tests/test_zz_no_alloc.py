"""tsx_ewise_noalloc, the allocation-free entry point.

Some callers of this library cannot allocate device memory: plugins that
may only use what their host engine hands them, frameworks whose pooling
allocator has reserved the device memory, latency-critical loops that
cannot pay for the synchronisation cudaMalloc / cudaFree may cause.  For
them tsx_ewise_noalloc runs the same kernel as tsx_ewise without a plan,
keeping the kernel's device status word in a static device array instead of
allocating it.  This test calls it through the C ABI twice in a row and
checks each result against tsx_ewise through a plan and against the CPU
oracle, with the tolerance the parity tests use (bit-exact; exp within its
ulp bound).  A timeout planted on the host (the producer skips one tile's
loads) must come back through status_out, and the next clean call must
report TSX_OK with the right result.  It lives in a file of its own that
pytest collects last.
"""

import ctypes

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


def _noalloc(tsx, dtype, rows, cols, box, stages, variant, op, ins, out, status):
    ptrs = [t.data_ptr() for t in ins] + [None] * (3 - len(ins))
    stream = torch.cuda.current_stream().cuda_stream
    return tsx.tsx_ewise_noalloc(tsx.DTYPES[dtype], rows, cols, box[0], box[1], stages, tsx.VARIANTS[variant],
                                 tsx.OPS[op], *ptrs, out.data_ptr(), stream,
                                 ctypes.byref(status) if status is not None else None)


@pytest.mark.parametrize("dtype,rows,cols,box,stages,variant,op", [
    ("f32", 203, 640, (8, 128), 4, "tma", "fma"),
    ("bf16", 300, 1024, (128, 128), 3, "tma", "exp"),
    ("bf16", 300, 1024, (128, 128), 2, "tma", "exp"),     # two-stage ring: two store warps, capped CTAs
    ("f16", 77, 512, (16, 256), 2, "tma_rank3", "add"),
])
def test_noalloc_matches_tsx_ewise_on_two_calls_in_a_row(tsx, dtype, rows, cols, box, stages, variant, op):
    n_in = tsx.ARITY[op]
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant) as plan:
        for call in range(2):
            host = [random_bits(dtype, (rows, cols), 1000 * call + k) for k in range(n_in)]
            ins = [to_dev(x, dtype) for x in host]
            want = plan.ewise(op, *ins)
            out = torch.full_like(ins[0], 0)
            status = ctypes.c_int(-99)
            rc = _noalloc(tsx, dtype, rows, cols, box, stages, variant, op, ins, out, status)
            assert rc == tsx.TSX_OK, tsx.tsx_last_error()
            assert status.value == tsx.TSX_OK
            torch.cuda.synchronize()
            got = bits_of(out, dtype)
            compare(op, dtype, got, bits_of(want, dtype), f"call {call} against tsx_ewise")
            compare(op, dtype, got, oracle.ewise(op, dtype, *host), f"call {call} against the oracle")


def test_noalloc_reports_a_timeout_and_recovers(tsx):
    """The fault is made on the host: the producer announces tile 3's bytes
    but issues no load, so the bounded wait on that stage runs out after
    50 ms.  The status word must say TSX_ERR_TIMEOUT; the next call, with the
    hook cleared, starts from a cleared word and reports TSX_OK."""
    rows, cols, box = 96, 512, (8, 128)
    host = random_bits("f32", (rows, cols), 11)
    a = to_dev(host, "f32")
    out = torch.zeros_like(a)
    status = ctypes.c_int(-99)
    tsx.tsx_debug_noalloc_set_fault(3, 50)
    try:
        rc = _noalloc(tsx, "f32", rows, cols, box, 3, "tma", "sqrt", [a], out, status)
    finally:
        tsx.tsx_debug_noalloc_set_fault(-1, 0)
    assert rc == tsx.TSX_OK, tsx.tsx_last_error()
    assert status.value == tsx.TSX_ERR_TIMEOUT
    status.value = -99
    rc = _noalloc(tsx, "f32", rows, cols, box, 3, "tma", "sqrt", [a], out, status)
    assert rc == tsx.TSX_OK and status.value == tsx.TSX_OK
    torch.cuda.synchronize()
    compare("sqrt", "f32", bits_of(out, "f32"), oracle.ewise("sqrt", "f32", host), "after the timeout")


def test_noalloc_without_status_and_its_errors(tsx):
    rows, cols = 64, 256
    a = to_dev(random_bits("f32", (rows, cols), 7), "f32")
    out = torch.empty_like(a)
    assert _noalloc(tsx, "f32", rows, cols, (8, 64), 2, "tma", "sqrt", [a], out, None) == tsx.TSX_OK
    torch.cuda.synchronize()
    with tsx.Plan("f32", rows, cols, box=(8, 64), stages=2) as plan:
        want = plan.ewise("sqrt", a)
        torch.cuda.synchronize()
    assert np.array_equal(bits_of(out, "f32"), bits_of(want, "f32"))
    # only the TMA kernel is offered
    rc = _noalloc(tsx, "f32", rows, cols, (8, 64), 2, "ldgsts", "sqrt", [a], out, None)
    assert rc == tsx.TSX_ERR_INVALID and "TMA" in tsx.tsx_last_error()
    # a call turned away before its launch leaves status_out alone
    status = ctypes.c_int(-99)
    rc = _noalloc(tsx, "f32", rows, cols, (8, 64), 2, "tma", "add", [a], out, status)
    assert rc == tsx.TSX_ERR_INVALID and status.value == -99
    # the same declines as a plan would give
    rc = _noalloc(tsx, "f32", rows, cols, (8, 40), 2, "tma", "sqrt", [a], out, None)
    assert rc == tsx.TSX_ERR_UNSUPPORTED and "128-byte atoms" in tsx.tsx_last_error()
    # an empty tensor is a no-op
    empty = torch.empty(0, cols, device="cuda")
    assert _noalloc(tsx, "f32", 0, cols, (8, 64), 2, "tma", "sqrt", [empty], empty, None) == tsx.TSX_OK
