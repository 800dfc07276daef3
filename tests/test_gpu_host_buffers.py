"""Host buffers: the cp.async and synchronous variants run on page-locked
host memory that the device addresses directly (inputs read and the result
written over the host link, no staging copies).  Results must equal the
oracle's exactly as on device memory, and the plan's status stays clean."""

import zlib

import numpy as np
import pytest

import oracle
from tests import _gpu
from tests._gpu import compare, random_bits, torch

pytestmark = pytest.mark.gpu

ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _pinned(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).pin_memory()


@pytest.mark.parametrize("variant", ["ldgsts", "sync"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("op", ["copy", "sqrt", "exp", "add", "fma"])
def test_host_buffers_match_the_oracle(tsx, variant, dtype, op):
    rows, cols, box = 37, 1000, (8, 128)
    seed = zlib.crc32(f"host/{variant}/{dtype}/{op}".encode())
    ins = [random_bits(dtype, (rows, cols), seed + k) for k in range(ARITY[op])]
    want = oracle.ewise(op, dtype, *ins)
    hosts = [_pinned(x) for x in ins]
    out = _pinned(np.zeros((rows, cols), dtype=ins[0].dtype))
    ptrs = [h.data_ptr() for h in hosts] + [None] * (3 - len(hosts))
    with tsx.Plan(dtype, rows, cols, box=box, stages=3, variant=variant) as plan:
        plan.ewise_ptr(op, ptrs[0], ptrs[1], ptrs[2], out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare(op, dtype, out.numpy(), want, f"{variant} {dtype} {op} on host buffers")


def test_host_and_device_buffers_mix(tsx):
    """Inputs on the host, result on the device, and the reverse."""
    rows, cols = 64, 4096
    a, b = random_bits("f32", (rows, cols), 11), random_bits("f32", (rows, cols), 12)
    want = oracle.ewise("mul", "f32", a, b)
    ha, hb = _pinned(a), _pinned(b)
    da, db = ha.cuda(), hb.cuda()
    dout = torch.empty(rows, cols, dtype=torch.int32, device="cuda")
    hout = _pinned(np.zeros((rows, cols), dtype=np.uint32))
    s = torch.cuda.current_stream().cuda_stream
    with tsx.Plan("f32", rows, cols, box=(16, 256), stages=2, variant="ldgsts") as plan:
        plan.ewise_ptr("mul", ha.data_ptr(), hb.data_ptr(), None, dout.data_ptr(), s)
        plan.ewise_ptr("mul", da.data_ptr(), db.data_ptr(), None, hout.data_ptr(), s)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    compare("mul", "f32", dout.cpu().numpy().view(np.uint32), want, "host in, device out")
    compare("mul", "f32", hout.numpy(), want, "device in, host out")
