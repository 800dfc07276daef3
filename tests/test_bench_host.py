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


def test_reference_arm_reports_its_cores(capsys):
    """The reference arm times the oracle on every host core and names the
    count, with a single-thread figure beside it."""
    import oracle

    rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1", "--workload", "add_1024x8192_f16"])
    assert rc == 0
    d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    cb = d["cpu_baseline"]
    assert cb["cores"] == oracle.host_cores() >= 1
    assert cb["single_core"]["cores"] == 1 and cb["single_core"]["value"] > 0


def test_parity_leg_flags_a_differing_element():
    """The CPU-baseline leg's check of the whole device output: an output
    equal to the oracle's has no mismatch, one flipped bit is one mismatch,
    and its position is reported."""
    import numpy as np

    w = bench.ti.WORKLOADS["fma_128x1048576_f32"].with_rows(2)
    ins = w.inputs()
    base, parity = bench.cpu_baseline(w, ins, None, 0.1)
    assert parity is None and base["cores"] >= 1 and base["single_core"]["value"] > 0
    import oracle

    dev = np.asarray(oracle.ewise(w.op, w.dtype, *ins)).view(np.uint32).copy()
    assert bench.cpu_baseline(w, ins, dev, 0.1)[1]["mismatches"] == 0
    dev[1, 7] ^= 1
    p = bench.cpu_baseline(w, ins, dev, 0.1)[1]
    assert p["mismatches"] == 1 and p["elements"] == w.elems
    assert p["first_mismatch_flat_index"] == w.cols + 7


def test_parity_record_uses_the_exp_bound():
    import numpy as np

    import oracle

    w = bench.ti.WORKLOADS["exp_16384x16384_bf16"].with_rows(4)
    ins = w.inputs()
    want = oracle.ewise(w.op, w.dtype, *ins)
    got = want.copy().reshape(-1)
    got[3] += 1          # one ulp: within the bf16 bound
    assert bench.parity_record(w, got, want, 2)["mismatches"] == 0
    got[5] += 2          # two ulps: outside
    rec = bench.parity_record(w, got, want, 2)
    assert rec["mismatches"] == 1 and rec["first_mismatch_flat_index"] == 5 and rec["rule"] == "within 1 ulp"


def test_single_core_oracle_timing_is_bounded():
    w = bench.ti.WORKLOADS["fma_128x1048576_f32"].with_rows(8)
    ins = w.inputs()
    nbytes, spent, elems = bench.oracle_single_core(w, ins, 0.01, band_elems=1 << 18)
    assert 1 <= elems < w.elems and nbytes == elems * 16 and spent > 0


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


def test_clock_summary():
    """Median SM clock and the throttle reasons of the samples in a region."""
    samples = [(1965.0, 0x0), (1900.0, 0x4), (2070.0, 0x1)]
    c = bench.summarise_clocks(samples, 2070.0)
    assert c["samples"] == 3 and c["sm_mhz"] == 1965.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]   # idle (0x1) is not a throttle reason
    c = bench.summarise_clocks([(1200.0, 0x8 | 0x40)], 2070.0)
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.summarise_clocks([], None)["sm_mhz"] is None


def test_clock_sampler_regions_without_nvml():
    """Without NVML (no GPU here) the sampler says so instead of failing."""
    s = bench.ClockSampler(0).start()
    s.stop()
    r = s.region(0.0, 1e12)
    assert r["samples"] == 0 or r["sm_mhz"] is not None


def test_recorded_traffic_per_stage(tmp_path, monkeypatch):
    """The roofline's traffic comes from a committed profile summary only
    while its kernel-source hash matches, per stage count."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = bench.source_digest()
    (prof / "tma_ewise_w.md").write_text(
        f"- kernel_sources_sha256_16: `{digest}`\n- variant: `tma`\n"
        "- dram_bytes_per_launch[S=2]: `100`\n- dram_bytes_per_launch[S=3]: `200`\n")
    (prof / "tma_ewise_old.md").write_text(
        "- kernel_sources_sha256_16: `0000000000000000`\n- variant: `tma`\n- stages: `4`\n"
        "- dram_bytes_per_launch: `300`\n")
    (prof / "tma_ewise_one.md").write_text(
        f"- kernel_sources_sha256_16: `{digest}`\n- variant: `tma`\n- stages: `4`\n"
        "- dram_bytes_per_launch: `400`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: digest)
    assert bench.recorded_traffic("w", "tma", 2) == 100.0
    assert bench.recorded_traffic("w", "tma", 3) == 200.0
    assert bench.recorded_traffic("w", "tma", 4) is None
    assert bench.recorded_traffic("w", "tma_rank3", 2) is None
    assert bench.recorded_traffic("old", "tma", 4) is None        # taken on other kernel sources
    assert bench.recorded_traffic("one", "tma", 4) == 400.0
    assert bench.recorded_traffic("missing", "tma", 4) is None
