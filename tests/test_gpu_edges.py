"""GPU edge cases: bounds (canaries), untouched inputs, aliasing, pointer
alignment, argument errors, many buffers through one plan, side streams,
and a device-side wait that is made to run out (the fault is planted on the
host: the producer is told to skip one tile's loads, so a barrier that
nothing completes times out; nothing faults)."""

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


SENTINEL = {"f32": 0x7FBADBAD, "f16": 0x7DAD, "bf16": 0x7FAD}


def _embedded(bits, dtype, pad):
    """A device buffer [pad | bits | pad] with sentinel pads, and the view of
    the middle part."""
    flat = np.concatenate([np.full(pad, SENTINEL[dtype], dtype=bits.dtype), bits.reshape(-1),
                           np.full(pad, SENTINEL[dtype], dtype=bits.dtype)])
    buf = to_dev(flat, dtype)
    return buf, buf[pad:pad + bits.size].view(bits.shape)


@pytest.mark.parametrize("variant", ["tma", "tma_rank3", "tma_mixed", "tma_promoted", "ldgsts", "sync"])
def test_canaries_and_inputs_untouched(tsx, variant):
    dtype, rows, cols, box = "f32", 77, 320, (16, 64)
    ins = [random_bits(dtype, (rows, cols), 40 + k) for k in range(3)]
    want = oracle.ewise("fma", dtype, *ins)
    dev_ins = [to_dev(x, dtype) for x in ins]
    pad = 4096
    buf, out = _embedded(np.zeros((rows, cols), dtype=np.uint32), dtype, pad)
    with tsx.Plan(dtype, rows, cols, box=box, stages=3, variant=variant) as plan:
        plan.ewise("fma", *dev_ins, out=out)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    b = bits_of(buf, dtype)
    assert np.all(b[:pad] == SENTINEL[dtype]) and np.all(b[-pad:] == SENTINEL[dtype])
    compare("fma", dtype, b[pad:-pad], want, variant)
    for x, d in zip(ins, dev_ins):
        assert np.array_equal(bits_of(d, dtype), x)


@pytest.mark.parametrize("variant", ["tma", "tma_mixed", "ldgsts"])
@pytest.mark.parametrize("alias", ["a", "b", "c"])
def test_out_may_alias_an_input(tsx, variant, alias):
    dtype, rows, cols = "bf16", 130, 256
    ins = [random_bits(dtype, (rows, cols), 60 + k) for k in range(3)]
    want = oracle.ewise("fma", dtype, *ins)
    d = [to_dev(x, dtype) for x in ins]
    out = d["abc".index(alias)]
    with tsx.Plan(dtype, rows, cols, box=(32, 128), stages=2, variant=variant) as plan:
        plan.ewise("fma", *d, out=out)
        torch.cuda.synchronize()
    compare("fma", dtype, bits_of(out, dtype), want, f"out is {alias}")


def _offset_view(bits, dtype, offset_elems):
    es = 4 if dtype == "f32" else 2
    flat = np.concatenate([np.zeros(offset_elems, dtype=bits.dtype), bits.reshape(-1)])
    buf = to_dev(flat, dtype)
    view = buf[offset_elems:]
    assert view.data_ptr() % 16 == (offset_elems * es) % 16
    return buf, view.view(bits.shape)


def test_tma_rejects_unaligned_base(tsx):
    dtype, rows, cols = "f32", 16, 64
    a = random_bits(dtype, (rows, cols), 1)
    _, va = _offset_view(a, dtype, 1)          # 4-byte aligned only
    out = torch.empty(rows, cols, device="cuda")
    with tsx.Plan(dtype, rows, cols, box=(8, 32), stages=2) as plan:
        with pytest.raises(tsx.TsxError) as ei:
            plan.ewise("copy", va, out=out)
        assert ei.value.code == tsx.TSX_ERR_ALIGN


@pytest.mark.parametrize("variant", ["ldgsts", "sync"])
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_copy_variants_narrow_to_pointer_alignment(tsx, variant, offset):
    """cp.async falls back to 8- and 4-byte copies on 8- and 4-byte aligned
    bases (TVM "copy_async -> ldgsts", table under "How inputs change the
    algorithm") and still computes the exact result."""
    dtype, rows, cols = "f32", 45, 96
    ins = [random_bits(dtype, (rows, cols), 80 + k) for k in range(2)]
    want = oracle.ewise("add", dtype, *ins)
    keep = []
    views = []
    for x in ins:
        buf, v = _offset_view(x, dtype, offset)
        keep.append(buf)
        views.append(v)
    obuf, out = _offset_view(np.zeros((rows, cols), dtype=np.uint32), dtype, offset)
    with tsx.Plan(dtype, rows, cols, box=(16, 32), stages=3, variant=variant) as plan:
        plan.ewise("add", *views, out=out)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("add", dtype, bits_of(out, dtype), want, f"offset {offset}")


def test_f16_two_byte_aligned_base_is_rejected(tsx):
    dtype, rows, cols = "f16", 8, 64
    a = random_bits(dtype, (rows, cols), 3)
    _, va = _offset_view(a, dtype, 1)   # 2-byte aligned
    out = torch.empty(rows, cols, device="cuda", dtype=torch.float16)
    with tsx.Plan(dtype, rows, cols, box=(8, 64), stages=2, variant="ldgsts") as plan:
        with pytest.raises(tsx.TsxError) as ei:
            plan.ewise("copy", va, out=out)
        assert ei.value.code == tsx.TSX_ERR_ALIGN


def test_operand_count_is_checked(tsx):
    a = torch.rand(16, 64, device="cuda")
    with tsx.Plan("f32", 16, 64, box=(8, 32), stages=2) as plan:
        pa = a.data_ptr()
        for op, args in (("add", (pa, None, None)), ("copy", (pa, pa, None)), ("fma", (pa, pa, None)),
                         ("sqrt", (pa, None, pa))):
            with pytest.raises(tsx.TsxError) as ei:
                plan.ewise_ptr(op, *args, out=pa)
            assert ei.value.code == tsx.TSX_ERR_INVALID
        with pytest.raises(tsx.TsxError) as ei:
            plan.ewise_ptr("copy", None, None, None, out=pa)
        assert ei.value.code == tsx.TSX_ERR_INVALID
        with pytest.raises(tsx.TsxError):
            plan.ewise_ptr(7, pa, None, None, out=pa)


def test_many_buffers_through_one_plan(tsx):
    """More distinct pointers than the tensor-map cache holds."""
    dtype, rows, cols = "f16", 40, 128
    with tsx.Plan(dtype, rows, cols, box=(16, 64), stages=2) as plan:
        for k in range(20):
            a = random_bits(dtype, (rows, cols), 200 + k)
            want = oracle.ewise("sqrt", dtype, a)
            out = plan.ewise("sqrt", to_dev(a, dtype))
            torch.cuda.synchronize()
            compare("sqrt", dtype, bits_of(out, dtype), want, f"buffer {k}")


def test_side_stream(tsx):
    dtype, rows, cols = "f32", 300, 512
    a = random_bits(dtype, (rows, cols), 9)
    want = oracle.ewise("exp", dtype, a)
    s = torch.cuda.Stream()
    da = to_dev(a, dtype)
    torch.cuda.synchronize()
    with tsx.Plan(dtype, rows, cols, box=(32, 128), stages=3) as plan:
        with torch.cuda.stream(s):
            out = plan.ewise("exp", da)
        s.synchronize()
        compare("exp", dtype, bits_of(out, dtype), want, "side stream")


def test_plan_info_launch(tsx):
    with tsx.Plan("bf16", 16384, 16384, box=(128, 128), stages=4) as plan:
        info = plan.info("exp")
        assert info["sm_count"] > 0 and info["ctas_per_sm"] >= 1
        assert info["grid"] == min(info["tiles"], info["sm_count"] * info["ctas_per_sm"])
        assert info["smem_bytes"] <= 232448


def test_wait_timeout_is_reported_and_the_context_survives(tsx):
    """The producer skips the loads of one tile (but announces its bytes), so
    that stage's barrier never completes: the bounded wait gives up, the
    kernel records TSX_ERR_TIMEOUT and returns, and the GPU stays usable."""
    dtype, rows, cols = "f32", 256, 1024
    a = random_bits(dtype, (rows, cols), 5, finite_fraction=1.0)
    bad = tsx.Plan(dtype, rows, cols, box=(8, 128), stages=3, tuning={"timeout_ms": 50})
    bad.set_fault_tile(5)
    bad_checked = tsx.Plan(dtype, rows, cols, box=(8, 128), stages=3, tuning={"timeout_ms": 50, "checked": 1})
    bad_checked.set_fault_tile(5)
    da = to_dev(a, dtype)
    try:
        bad.ewise("sqrt", da)
        torch.cuda.synchronize()
        assert bad.status() == tsx.TSX_ERR_TIMEOUT
        assert bad.status() == tsx.TSX_OK        # reading clears it
        with pytest.raises(tsx.TsxError) as ei:
            bad_checked.ewise("sqrt", da)
        assert ei.value.code == tsx.TSX_ERR_TIMEOUT
    finally:
        bad.close()
        bad_checked.close()
    # the context is intact: a normal plan gives the exact result
    want = oracle.ewise("sqrt", dtype, a)
    with tsx.Plan(dtype, rows, cols, box=(8, 128), stages=3) as plan:
        out = plan.ewise("sqrt", da)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("sqrt", dtype, bits_of(out, dtype), want, "after the timeout")
