"""Host-side logic of bench.py: the reference (CPU oracle) arm's JSON line
and its rank handling, the oracle check of the device output, the timing
aggregation over ranks (world size 2, gloo, on CPU) and the clock-sample
parser."""

import json
import multiprocessing as mp
import os
import socket

import pytest

import bench


def test_reference_arm_json_line(capsys):
    rc = bench.main(["--impl", "reference", "--steps", "3", "--warmup", "1", "--workload", "sqrt_500x4096_f32"])
    assert rc == 0
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "sqrt_500x4096_f32"


def test_reference_arm_other_ranks_print_nothing(capsys, monkeypatch):
    """Under torchrun only rank 0 runs and prints the reference arm; the
    other ranks exit 0 without work."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    rc = bench.main(["--impl", "reference", "--steps", "3", "--warmup", "1", "--workload", "sqrt_500x4096_f32"])
    assert rc == 0
    assert capsys.readouterr().out.strip() == ""


def test_parity_leg_flags_a_differing_element():
    """The CPU-baseline leg's check of the device output: an output equal to
    the oracle's has no mismatch, one flipped bit is one mismatch."""
    import numpy as np

    import oracle

    w = bench.ti.WORKLOADS["fma_128x1048576_f32"].with_rows(1)
    band = bench.oracle_band_rows(w)
    idx = np.arange(0, band * w.cols, dtype=np.uint64)
    head = np.asarray(oracle.ewise(w.op, w.dtype, *w.inputs_at(idx))).view(np.int32).reshape(band, w.cols)
    assert bench.cpu_baseline(w, 0.2, head)[1]["mismatches"] == 0
    head[0, 7] ^= 1
    assert bench.cpu_baseline(w, 0.2, head)[1]["mismatches"] == 1


def test_cpu_baseline_is_bounded():
    w = bench.ti.WORKLOADS["fma_128x1048576_f32"]
    nbytes, spent, rows, cores = bench.cpu_time_oracle(w, 0.05, max_rows=8)
    assert 1 <= rows <= 8 and cores == 1 and nbytes == rows * w.cols * 16


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    td = bench.init_dist(world, "gloo")
    seconds = 1.0 + rank          # rank 1 is the slow one
    units = 10.0 * (rank + 1)
    q.put((rank, bench.aggregate(td, seconds, units)))
    bench.barrier(td)
    td.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 30.0)   # max of seconds, sum of units


def test_clock_sampler_parses_samples():
    s = bench.ClockSampler(0)

    class P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = P()
    s.lines = [(1.0, "0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (2.0, "0, 1900, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active"),
               (9.0, "0, 300, 2070, 90.0, 0x0, Active, Not Active, Not Active, Not Active")]
    import time as _t

    orig = _t.sleep
    _t.sleep = lambda x: None
    try:
        c = s.stop(0.5, 5.0)
    finally:
        _t.sleep = orig
    assert c["samples"] == 2 and c["sm_mhz"] == pytest.approx(1932.5) and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
