"""Benchmark of tile-elementwise streaming on GB300.

One step = one ``tsx_ewise`` call: the whole path (tile loads through the
S-stage mbarrier ring, the shared-memory elementwise stage, the TMA stores)
over the workload's tensors.  Default workload: fp32 fma over three
[128, 1048576] tensors (box 8x128 = four 8x32 TMA loads per operand, 4
stages), the largest stated configuration (2 GiB moved per step).

Prints one JSON line (rank 0).  Metric: HBM GB/s = (n_in + 1) * rows * cols *
element size / device time, i.e. algorithmic bytes read plus written.

    python bench.py [--steps K] [--warmup W] [--workload NAME] [--stages S]
                    [--variant tma|tma_rank3|ldgsts|sync] [--impl reference]

``--impl reference`` times the CPU oracle (the only reference there is) on
bounded samples of the same workload, one sample per step.  Under torchrun
with N > 1 every rank runs an independent replica (the path has no exchange
step); only timing is reduced across ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import tsx_inputs as ti  # noqa: E402

METRIC = "pipelined tile-ewise HBM GB/s (read+write) and % of GB300 peak/memcpy ceiling"
DEFAULT_WORKLOAD = "fma_128x1048576_f32"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
DTYPE_NAME = {"f32": "f32", "f16": "f16", "bf16": "bf16"}
KERNEL_SOURCES = ["pipelined_elementwise_streaming_gb300/csrc/k_tma.cu",
                  "pipelined_elementwise_streaming_gb300/csrc/tsx_tma_common.cuh",
                  "pipelined_elementwise_streaming_gb300/csrc/tsx_device.cuh",
                  "pipelined_elementwise_streaming_gb300/csrc/tsx_internal.h"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(ti.WORKLOADS))
    p.add_argument("--stages", type=int, default=None,
                   help="default: the workload's benchmark stage count (one of its stated ones)")
    p.add_argument("--rows", type=int, default=None,
                   help="run the workload over its first ROWS rows only (a smaller case, e.g. for profiling)")
    p.add_argument("--variant", default=None, help="default: the workload's variant")
    p.add_argument("--box", type=int, nargs=2, default=None, metavar=("ROWS", "COLS"),
                   help="stage tile other than the workload's (row sums run one CTA per band of ROWS rows)")
    p.add_argument("--op", default=None, choices=["copy", "sqrt", "exp", "add", "mul", "fma"],
                   help="op other than the workload's (same shape, dtype and value distribution)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--mode", default="ewise", choices=["ewise", "accumulate", "rowsum"],
                   help="ewise: out = op(...); accumulate: out += op(...) by TMA reduce-store; "
                        "rowsum: fp32 row sums of op(...)")
    p.add_argument("--sweep", action="store_true",
                   help="tuning sweep instead of the benchmark: time the workload's op over candidate boxes, stage "
                        "counts and thread counts (the plans the host accepts), check each result against the "
                        "workload's own plan bit for bit, and print one JSON line per candidate, fastest first")
    p.add_argument("--tune", action="append", default=[], metavar="KNOB=VALUE",
                   help="launch knob of the timed plan (threads, ctas_per_sm, store_lag, store_warps, l2_promotion); "
                        "repeatable")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-second", action="store_true",
                   help="skip the second stated bar (bf16 exp over [16384, 16384] at stages 2, 3 and 4), which the "
                        "default run times after the headline workload")
    p.add_argument("--cpu-seconds", type=float, default=5.0,
                   help="budget of the single-thread oracle timing")
    return p.parse_args(argv)


# ------------------------------------------------------------------ ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as td

    if world > 1 and not td.is_initialized():
        td.init_process_group(backend=backend)
    return td if world > 1 else None


def aggregate(td, seconds: float, units: float):
    """(max seconds over ranks, sum of units over ranks)."""
    if td is None:
        return seconds, units
    import torch

    dev = "cuda" if td.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    td.all_reduce(u, op=td.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(td):
    if td is not None:
        td.barrier()


# ----------------------------------------------------------------- helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def git_revision():
    """The checkout's commit, or None where the tree is not a git checkout."""
    import subprocess

    try:
        r = subprocess.run(["git", "-C", ROOT, "rev-parse", "--short=12", "HEAD"], capture_output=True, text=True,
                           timeout=10)
    except (OSError, subprocess.SubprocessError):
        return None
    return r.stdout.strip() or None if r.returncode == 0 else None


def source_digest() -> str:
    import hashlib

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, variant: str, stages: int):
    """DRAM bytes per launch from the committed ncu summary of this kernel
    and workload (``dram_bytes_per_launch[S=<stages>]``, or
    ``dram_bytes_per_launch`` with a matching ``stages``), if it was taken on
    the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"tma_ewise_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_sources_sha256_16") != source_digest() or fields.get("variant") != variant:
        return None
    value = fields.get(f"dram_bytes_per_launch[S={stages}]")
    if value is None and fields.get("stages") == str(stages):
        value = fields.get("dram_bytes_per_launch")
    try:
        return float(value) if value is not None else None
    except ValueError:
        return None


class ClockSampler:
    """SM clock and clock-event reasons of this process's GPU while timed
    regions run, read on a background thread about every half millisecond
    through NVML's read-only queries (nvmlDeviceGetClockInfo,
    nvmlDeviceGetCurrentClocksEventReasons).  Nothing is set.  Samples keep
    their host time, so each timed region takes its own (``region``)."""

    # nvmlClocksEventReason* bits that matter for a timing
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    PERIOD_S = 0.0005

    def __init__(self, device_index: int, uuid: str | None = None):
        self.device_index = device_index
        self.uuid = uuid
        self.samples = []          # (host time, sm MHz, reason bits)
        self.sm_max = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open(self):
        import ctypes

        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError as e:
            self.error = f"NVML unavailable: {e}"
            return False
        if nv.nvmlInit_v2() != 0:
            self.error = "nvmlInit failed"
            return False
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            u = self.uuid if self.uuid.startswith("GPU-") else "GPU-" + self.uuid
            ok = nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.device_index), ctypes.byref(h)) == 0
        if not ok:
            self.error = "no NVML handle for the device"
            return False
        self._nvml, self._handle = nv, h
        mhz = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mhz)) == 0:   # NVML_CLOCK_SM
            self.sm_max = float(mhz.value)
        self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        return True

    def _read_one(self):
        import ctypes

        mhz = ctypes.c_uint()
        bits = ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._handle, ctypes.c_int(1), ctypes.byref(mhz)) != 0:
            return None
        if self._reasons_fn is None or self._reasons_fn(self._handle, ctypes.byref(bits)) != 0:
            bits.value = 0
        return float(mhz.value), int(bits.value)

    def _run(self):
        while not self._stop.is_set():
            r = self._read_one()
            if r is not None:
                self.samples.append((time.monotonic(), r[0], r[1]))
            time.sleep(self.PERIOD_S)

    def start(self):
        if self._open():
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        if self._nvml is not None:
            self._nvml.nvmlShutdown()
            self._nvml = None

    def region(self, t0: float, t1: float) -> dict:
        """Summary of the samples taken between host times t0 and t1."""
        if self.error:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.error], "samples": 0, "source": "nvml"}
        return summarise_clocks([(f, b) for t, f, b in list(self.samples) if t0 <= t <= t1], self.sm_max)


def summarise_clocks(samples, sm_max) -> dict:
    """Median SM MHz and the union of the throttle reasons over (MHz, reason
    bits) samples."""
    reasons = sorted({name for _, bits in samples for bit, name in ClockSampler.REASONS.items() if bits & bit})
    mhz = [f for f, _ in samples]
    return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": sm_max, "reasons": reasons,
            "samples": len(mhz), "source": "nvml"}


# --------------------------------------------------------------- our path

def to_host_tensors(w, torch, ins=None):
    """The workload's inputs (element bits; generated unless given) as pinned
    host tensors of the element type."""
    out = []
    for bits in (w.inputs() if ins is None else ins):
        if w.dtype == "f32":
            t = torch.from_numpy(bits.view(np.float32))
        else:
            t = torch.from_numpy(bits.view(np.int16)).view(torch.float16 if w.dtype == "f16" else torch.bfloat16)
        out.append(t.pin_memory())
    return out


def memcpy_ceiling(torch, nbytes=1 << 30, reps=20):
    """Device-to-device copy GB/s (read + write counted), median of reps."""
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    src.fill_(1)
    for _ in range(3):
        dst.copy_(src)
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src)
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    del src, dst
    return 2 * nbytes / statistics.median(times) / 1e9


def step_bytes(w, mode: str) -> int:
    """Algorithmic bytes of one step: every input read once, plus the output
    written (ewise), read and written (accumulate), or one fp32 per row
    (rowsum)."""
    es = ti.ELEM_SIZE[w.dtype]
    if mode == "accumulate":
        return (w.n_in + 2) * w.elems * es
    if mode == "rowsum":
        return w.n_in * w.elems * es + 4 * w.rows
    return w.algorithmic_bytes


def time_steps(torch, tsx, w, plan, mode, dev_in, out, row_sums, K, W, sampler):
    """W untimed then K timed steps of one plan on the current stream, each
    bracketed by CUDA events on that stream.  Inputs larger than L2 run back
    to back; smaller ones get an L2 flush before every step and only the
    kernels are counted.  Returns the timing record."""
    nbytes = step_bytes(w, mode)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    ptrs = [t.data_ptr() for t in dev_in] + [None] * (3 - len(dev_in))
    po = out.data_ptr()
    small = nbytes < 2 * L2_BYTES   # inputs of twice the L2 or more stream through it without reuse
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if small else None
    op_code = tsx.OPS[w.op] | (tsx.TSX_ACCUMULATE if mode == "accumulate" else 0)

    def step():
        if mode == "rowsum":
            rc = tsx.tsx_reduce_rows(plan.handle, op_code, ptrs[0], ptrs[1], ptrs[2], row_sums.data_ptr(), sh)
            if rc != tsx.TSX_OK:
                raise tsx.TsxError(rc, tsx.tsx_last_error())
        else:
            plan.ewise_ptr(op_code, ptrs[0], ptrs[1], ptrs[2], po, sh)

    for _ in range(W):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    if plan.status() != tsx.TSX_OK:
        raise RuntimeError("device-side wait gave up during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    region0, region1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_wall0 = time.monotonic()
    region0.record(stream)
    for k in range(K):
        if flush is not None:
            flush.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    region1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.monotonic()
    if plan.status() != tsx.TSX_OK:
        raise RuntimeError("device-side wait gave up in the timed region")
    launch_s = [a.elapsed_time(b) / 1e3 for a, b in ev]
    kernel_total = sum(launch_s)
    region_s = region0.elapsed_time(region1) / 1e3
    return {"nbytes": nbytes, "small": small, "launch_s": launch_s, "kernel_total": kernel_total,
            "step_s": kernel_total if small else region_s, "K": K,
            "clocks": sampler.region(t_wall0, t_wall1) if sampler else None}


def roofline_of(t, peak, peak_kind, traffic, kernel):
    avg_launch = t["kernel_total"] / t["K"]
    achieved = t["nbytes"] / avg_launch / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
            "traffic": traffic, "kernel": kernel, "median_launch_ms": round(statistics.median(t["launch_s"]) * 1e3, 5)}


def device_bits(torch, t):
    """A CUDA tensor's element bits as a host numpy array."""
    if t.element_size() == 2:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


# The second stated bar: bf16 exp over [16384, 16384] (box 128x128 as two
# 128x64 loads), timed at each of its stated stage counts after the headline.
SECOND_WORKLOAD = "exp_16384x16384_bf16"


def run_second(args, torch, tsx, sampler, peak, peak_kind):
    """The second bar workload at every stated stage count: its own timing,
    roofline and memcpy ceiling, and its output kept for the oracle check."""
    w = ti.WORKLOADS[SECOND_WORKLOAD]
    ins = w.inputs()
    dev_in = [h.to("cuda") for h in to_host_tensors(w, torch, ins)]
    out = torch.zeros_like(dev_in[0])
    ceiling = memcpy_ceiling(torch)
    per_stage = {}
    outputs = {}
    for S in w.stages:
        plan = tsx.Plan(w.dtype, w.rows, w.cols, box=(w.box_rows, w.box_cols), stages=S, variant=w.variant)
        info = plan.info(w.op)
        out.zero_()
        t = time_steps(torch, tsx, w, plan, "ewise", dev_in, out, None, args.steps, args.warmup, sampler)
        plan.close()
        value = t["nbytes"] * t["K"] / t["step_s"] / 1e9
        outputs[S] = device_bits(torch, out)
        per_stage[str(S)] = {
            "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(t["step_s"] / t["K"] * 1e3, 5),
            "steps": t["K"], "gpu_launches": t["K"], "frac_of_memcpy_ceiling": round(value / ceiling, 4),
            "threads": info["threads"], "grid": info["grid"], "ctas_per_sm": info["ctas_per_sm"],
            "roofline": roofline_of(t, peak, peak_kind, recorded_traffic(w.name, w.variant, S),
                                    f"tma_ewise<{w.dtype},{w.op}>"),
            "clocks": t["clocks"],
        }
    del dev_in, out
    torch.cuda.empty_cache()
    return {"workload": w.name, "op": w.op, "dtype": w.dtype, "rows": w.rows, "cols": w.cols,
            "box": [w.box_rows, w.box_cols], "loads_per_operand": 2, "variant": w.variant,
            "algorithmic_bytes_per_step": w.algorithmic_bytes, "memcpy_ceiling_gbs": round(ceiling, 1),
            "l2": f"inputs larger than L2 ({w.algorithmic_bytes >> 20} MiB moved per step vs 129 MiB L2), "
                  "steps back to back",
            "stages": per_stage}, (ins, outputs)


def run_ours(args, w, stages, variant):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    td = init_dist(world, "nccl")
    import pipelined_elementwise_streaming_gb300 as tsx

    ins = w.inputs()
    host = to_host_tensors(w, torch, ins)
    dev_in = [h.to("cuda", non_blocking=False) for h in host]
    out = torch.zeros_like(dev_in[0])
    row_sums = torch.empty(w.rows, dtype=torch.float32, device="cuda")
    mode = args.mode
    tuning = {k: int(v) for k, v in (t.split("=", 1) for t in args.tune)} or None
    plan = tsx.Plan(w.dtype, w.rows, w.cols, box=(w.box_rows, w.box_cols), stages=stages, variant=variant,
                    tuning=tuning)
    info = plan.info(w.op, row_sums=mode == "rowsum")
    peak, peak_kind = measured_peak()
    sampler = None
    if rank == 0:
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(local).uuid)
        except Exception:
            pass
        sampler = ClockSampler(local, uuid).start()

    ceiling = memcpy_ceiling(torch)
    barrier(td)
    t = time_steps(torch, tsx, w, plan, mode, dev_in, out, row_sums, args.steps, args.warmup, sampler)
    barrier(td)
    nbytes, K = t["nbytes"], t["K"]
    max_s, total_bytes = aggregate(td, t["step_s"], float(nbytes) * K)
    value = total_bytes / max_s / 1e9

    # end to end: pinned host inputs in, host result out, every step
    E = max(1, args.e2e_steps)
    if mode == "ewise":
        e2e_s, h2d, d2h, bands = run_e2e(torch, tsx, w, stages, variant, host, dev_in, out, E, td)
        e2e_bytes = float(nbytes) * E
        e2e_s, e2e_bytes = aggregate(td, e2e_s, e2e_bytes)
        staged = {"value": round(e2e_bytes / e2e_s / 1e9, 2), "unit": "GB/s", "steps": E,
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "method": f"{bands} row bands per step through tsx_ewise ({variant}); each band's H2D copies "
                            "(two alternating copy streams), kernel and D2H copy overlap the neighbouring bands', "
                            "also across consecutive steps (a band is reloaded once its kernel has read it)"}
        zc_s, h2d, d2h = run_e2e_host(torch, tsx, w, stages, host, out, E, td)
        zc_s, zc_bytes = aggregate(td, zc_s, float(nbytes) * E)
        direct = {"value": round(zc_bytes / zc_s / 1e9, 2), "unit": "GB/s", "steps": E,
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "method": f"tsx_ewise ({HOST_VARIANT}) on the pinned host buffers themselves: the kernel reads "
                            "the inputs and writes the result over the host link, no staging copies"}
        best, other = (direct, staged) if direct["value"] >= staged["value"] else (staged, direct)
        e2e = dict(best, alternative=other)
    else:
        e2e = {"value": None, "unit": "GB/s", "note": f"the end-to-end leg runs in ewise mode only, not {mode}"}
    plan.close()
    # the whole device result of the timed steps, for the oracle check in the
    # CPU-baseline leg (ewise mode: out holds op(inputs) exactly once)
    result_bits = device_bits(torch, out) if mode == "ewise" else None
    del dev_in, out, host
    torch.cuda.empty_cache()

    second, second_out = None, None
    if (rank == 0 and not args.no_second and mode == "ewise" and w.name == DEFAULT_WORKLOAD and args.rows is None
            and args.box is None and args.op is None):
        second, second_out = run_second(args, torch, tsx, sampler, peak, peak_kind)
    if sampler:
        sampler.stop()

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(t["step_s"] / K * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE_NAME[w.dtype],
        "data": "synthetic (seeded SplitMix64 inputs, the workload's stated distribution)",
        "config": {
            "workload": w.name + ("" if args.rows is None else f" (first {w.rows} rows)"), "op": w.op, "rows": w.rows,
            "cols": w.cols, "box": [w.box_rows, w.box_cols],
            "stages": stages, "variant": variant, "threads": info["threads"], "grid": info["grid"],
            "store_lag": info["store_lag"], "tuning": tuning,
            "ctas_per_sm": info["ctas_per_sm"], "loads_per_operand": info["loads_per_operand"],
            "mode": mode, "algorithmic_bytes_per_step": nbytes,
            "l2": "L2 flushed between timed steps (kernel time only)" if t["small"]
                  else f"inputs larger than L2 ({nbytes >> 20} MiB moved per step vs 129 MiB L2), "
                       "steps back to back",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "kernel_sources_sha256_16": source_digest(),
            "git": git_revision(),
        },
        "memcpy_ceiling_gbs": round(ceiling, 1),
        "frac_of_memcpy_ceiling": round(value / world / ceiling, 4),
        "clocks": t["clocks"],
        "e2e": e2e,
        "gpu_launches": K,
        "roofline": roofline_of(t, peak, peak_kind,
                                recorded_traffic(w.name, variant, stages) if mode == "ewise" else None,
                                f"tma_rowsum<{w.dtype},{w.op}>" if mode == "rowsum" else
                                f"tma_ewise<{w.dtype},{w.op}>" if variant.startswith("tma") else f"{variant}_ewise"),
    }
    if second is not None:
        result["workloads"] = {second["workload"]: second}
    result["_check"] = (ins, result_bits) if result_bits is not None else None
    result["_second_out"] = second_out
    return result, td, rank


HOST_VARIANT = "ldgsts"


def run_e2e_host(torch, tsx, w, stages, host, dev_out, steps, td):
    """Time `steps` end-to-end steps on host buffers with no staging copies:
    the inputs stay in pinned host memory and the kernel writes the result
    straight into pinned host memory, both over the host link (the device
    addresses pinned host memory directly).  Each step is one tsx_ewise call
    of the cp.async variant.  The result must equal the device path's
    `dev_out` bit for bit.  Returns (seconds, h2d bytes, d2h bytes per step)."""
    host_out = torch.empty(dev_out.shape, dtype=dev_out.dtype, pin_memory=True)
    plan = tsx.Plan(w.dtype, w.rows, w.cols, box=(w.box_rows, w.box_cols), stages=stages, variant=HOST_VARIANT)
    ptrs = [h.data_ptr() for h in host] + [None] * (3 - len(host))
    stream = torch.cuda.Stream()

    def step():
        plan.ewise_ptr(w.op, ptrs[0], ptrs[1], ptrs[2], host_out.data_ptr(), stream.cuda_stream)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    barrier(td)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    seconds = start.elapsed_time(stop) / 1e3
    ok = plan.status() == tsx.TSX_OK
    plan.close()
    if not ok:
        raise RuntimeError("device-side wait gave up in the host-buffer steps")
    if not torch.equal(host_out.view(torch.uint8), dev_out.cpu().view(torch.uint8)):
        raise RuntimeError("the host-buffer result differs from the device path's")
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = host_out.numel() * host_out.element_size()
    return seconds, h2d, d2h


def run_e2e(torch, tsx, w, stages, variant, host, dev_in, out, steps, td, band_bytes=64 << 20):
    """Time `steps` end-to-end steps: every step copies all inputs from
    pinned host memory to the device, runs the path, and copies the result
    back to pinned host memory.  A step is cut into row bands so that the
    copies of one band overlap the kernels and copies of the others: band i's
    uploads go on copy stream i % 2, its kernel on the compute stream once
    they are done, its download on the download stream once the kernel is
    done.  Consecutive steps overlap too: band i of the next step is
    uploaded once this step's kernel of band i has read its inputs, and
    computed once this step's download of band i has read its result.

    Returns (seconds, h2d bytes per step, d2h bytes per step, bands)."""
    es = ti.ELEM_SIZE[w.dtype]
    row_bytes = w.cols * es * (w.n_in + 1)
    rows_per_band = max(w.box_rows, (band_bytes // max(1, row_bytes)) // w.box_rows * w.box_rows)
    rows_per_band = min(rows_per_band, w.rows)
    bounds = [(r, min(w.rows, r + rows_per_band)) for r in range(0, w.rows, rows_per_band)]
    plans = {}
    for r0, r1 in bounds:
        if r1 - r0 not in plans:
            plans[r1 - r0] = tsx.Plan(w.dtype, r1 - r0, w.cols, box=(w.box_rows, w.box_cols), stages=stages,
                                      variant=variant)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    up = [torch.cuda.Stream(), torch.cuda.Stream()]
    compute, down = torch.cuda.Stream(), torch.cuda.Stream()
    # per band: the previous step's kernel (inputs read) and download (result read)
    read_in = [None] * len(bounds)
    read_out = [None] * len(bounds)

    def one_step():
        done = None
        for i, (r0, r1) in enumerate(bounds):
            s_up = up[i % 2]
            if read_in[i] is not None:
                s_up.wait_event(read_in[i])
            with torch.cuda.stream(s_up):
                for h, d in zip(host, dev_in):
                    d[r0:r1].copy_(h[r0:r1], non_blocking=True)
                loaded = torch.cuda.Event()
                loaded.record(s_up)
            compute.wait_event(loaded)
            if read_out[i] is not None:
                compute.wait_event(read_out[i])
            p = plans[r1 - r0]
            ptrs = [d[r0:r1].data_ptr() for d in dev_in] + [None] * (3 - len(dev_in))
            p.ewise_ptr(w.op, ptrs[0], ptrs[1], ptrs[2], out[r0:r1].data_ptr(), compute.cuda_stream)
            computed = torch.cuda.Event()
            computed.record(compute)
            read_in[i] = computed
            down.wait_event(computed)
            with torch.cuda.stream(down):
                host_out[r0:r1].copy_(out[r0:r1], non_blocking=True)
            done = torch.cuda.Event()
            done.record(down)
            read_out[i] = done
        return done

    for _ in range(2):
        one_step()
    torch.cuda.synchronize()
    barrier(td)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(up[0])
    for st in (up[1], compute, down):
        st.wait_event(start)
    for _ in range(steps):
        one_step()
    stop.record(down)
    torch.cuda.synchronize()
    seconds = start.elapsed_time(stop) / 1e3
    for p in plans.values():
        if p.status() != tsx.TSX_OK:
            raise RuntimeError("device-side wait gave up in the end-to-end steps")
        p.close()
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = host_out.numel() * host_out.element_size()
    return seconds, h2d, d2h, len(bounds)


# ------------------------------------------------------------ the oracle

def oracle_single_core(w, ins, seconds_budget, band_elems=1 << 22):
    """The oracle on one host thread over leading bands of the workload's
    inputs until the budget is spent.  Returns (bytes, seconds, elements)."""
    import oracle

    flat = [x.reshape(-1) for x in ins]
    n, spent, done = flat[0].size, 0.0, 0
    while done < n and spent < seconds_budget:
        e = min(n, done + band_elems)
        t0 = time.perf_counter()
        oracle.ewise(w.op, w.dtype, *[x[done:e] for x in flat])
        spent += time.perf_counter() - t0
        done = e
    return (w.n_in + 1) * done * ti.ELEM_SIZE[w.dtype], spent, done


def oracle_check(w, ins, device_out, cores):
    """The oracle over the whole workload on every host core, timed, and the
    device output compared with it element by element under the parity rule
    (bit-exact; exp within its ulp bound).  Returns (oracle seconds, oracle
    bits, parity record)."""
    import oracle

    t0 = time.perf_counter()
    want = oracle.ewise_parallel(w.op, w.dtype, *ins, threads=cores)
    seconds = time.perf_counter() - t0
    parity = None
    if device_out is not None:
        parity = parity_record(w, device_out, want, cores)
    return seconds, want, parity


def parity_record(w, device_out, want, cores):
    import oracle

    bad, first = oracle.count_mismatches(w.op, w.dtype, device_out, want, cores)
    rule = (f"within {oracle.EXP_ULP_BOUND[w.dtype]} ulp" if w.op == "exp" else
            "bitwise" if w.op == "copy" else "bit-exact")
    rec = {"elements": int(np.asarray(device_out).size), "mismatches": bad, "rule": rule, "against": "oracle",
           "rows": f"all {w.rows} rows of the timed steps' output"}
    if bad:
        rec["first_mismatch_flat_index"] = first
    return rec


def cpu_baseline(w, ins, device_out, seconds, cores=None):
    """The oracle's throughput on the host (all cores over the whole workload,
    and one core over a bounded sample) and, with the device output, the
    element-by-element check of all of it against the oracle's."""
    import oracle

    cores = cores or oracle.host_cores()
    oracle.build()
    all_s, _, parity = oracle_check(w, ins, device_out, cores)
    nbytes = w.algorithmic_bytes
    one_bytes, one_s, one_elems = oracle_single_core(w, ins, seconds)
    base = {"value": round(nbytes / all_s / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"all {w.elems} elements of {w.name}, C oracle cut into element ranges over {cores} host "
                      f"threads, {all_s:.2f} s wall",
            "single_core": {"value": round(one_bytes / one_s / 1e9, 4), "unit": "GB/s", "cores": 1,
                            "sample": f"the first {one_elems} elements of {w.name}, one thread, {one_s:.1f} s"}}
    return base, parity


def second_checks(args, second, second_data, cores):
    """Oracle timing and full parity of the second bar workload's outputs."""
    w = ti.WORKLOADS[second["workload"]]
    ins, outputs = second_data
    all_s, want, _ = oracle_check(w, ins, None, cores)
    second["cpu_baseline"] = {"value": round(w.algorithmic_bytes / all_s / 1e9, 4), "unit": "GB/s", "cores": cores,
                              "kind": "oracle",
                              "sample": f"all {w.elems} elements, C oracle over {cores} host threads, {all_s:.2f} s"}
    for S, bits in outputs.items():
        second["stages"][str(S)]["parity"] = parity_record(w, bits, want, cores)


SWEEP_BOXES = [(8, 128), (16, 128), (32, 128), (64, 128), (128, 128), (8, 256), (32, 256), (64, 64), (128, 64),
               (256, 64), (16, 512), (64, 512)]
# row sums: wide, short tiles as well (a band's rows are summed by one CTA
# wherever its tile range allows)
SWEEP_BOXES_ROWSUM = [(1, 1024), (2, 1024), (4, 512), (4, 1024), (8, 256), (8, 512), (8, 1024), (16, 256),
                      (16, 512), (32, 128), (32, 256), (64, 128), (128, 128), (128, 64), (256, 64)]


def run_sweep(args, w, stages, variant):
    """Time every accepted (box, stages, threads) candidate of the workload's
    op and variant.  Elementwise: each candidate's output must equal the
    workload's own plan's output bit for bit.  Row sums (--mode rowsum): the
    order of additions depends on the plan, so each candidate's sums must lie
    within the summation error bound of the workload plan's, taken from the
    device's own sums of |x| scale (a sanity check; the tests hold every plan
    to the oracle).  Returns the result lines, fastest first."""
    import torch

    import pipelined_elementwise_streaming_gb300 as tsx

    torch.cuda.set_device(0)
    rowsum = args.mode == "rowsum"
    dev_in = [h.to("cuda") for h in to_host_tensors(w, torch)]
    ptrs = [t.data_ptr() for t in dev_in] + [None] * (3 - len(dev_in))
    ref = torch.zeros(w.rows, dtype=torch.float32, device="cuda") if rowsum else torch.zeros_like(dev_in[0])
    out = torch.zeros_like(ref)
    s = torch.cuda.current_stream().cuda_stream

    def launch(plan, dst):
        if rowsum:
            rc = tsx.tsx_reduce_rows(plan.handle, tsx.OPS[w.op], ptrs[0], ptrs[1], ptrs[2], dst.data_ptr(), s)
            if rc != tsx.TSX_OK:
                raise tsx.TsxError(rc, tsx.tsx_last_error())
        else:
            plan.ewise_ptr(w.op, ptrs[0], ptrs[1], ptrs[2], dst.data_ptr(), s)

    with tsx.Plan(w.dtype, w.rows, w.cols, box=(w.box_rows, w.box_cols), stages=stages, variant=variant) as p:
        launch(p, ref)
    torch.cuda.synchronize()
    if rowsum:
        # tolerance: twice the summation bound gamma(cols) * sum |x| of any
        # order, with x = op(...) from the elementwise path
        with tsx.Plan(w.dtype, w.rows, w.cols, box=(w.box_rows, w.box_cols), stages=stages, variant=variant) as p:
            x = torch.empty_like(dev_in[0])
            p.ewise_ptr(w.op, ptrs[0], ptrs[1], ptrs[2], x.data_ptr(), s)
        abs_sum = x.float().abs().sum(dim=1)
        del x
        tol = abs_sum * (2.0 * w.cols * 2.0 ** -24) + 1e-30
    nbytes = step_bytes(w, args.mode)
    K = max(20, min(args.steps, 200))
    lines = []
    seen = set()
    boxes = SWEEP_BOXES_ROWSUM if rowsum else SWEEP_BOXES
    for box in boxes:
        for st in (2, 3, 4, 6, 8):
            for threads in (None, 128, 256, 512):
                tuning = None if threads is None else {"threads": threads}
                try:
                    plan = tsx.Plan(w.dtype, w.rows, w.cols, box=box, stages=st, variant=variant, tuning=tuning)
                    info = plan.info(w.op, row_sums=rowsum)
                except tsx.TsxError:
                    continue
                key = (box, st, info["threads"])
                if key in seen:
                    plan.close()
                    continue
                seen.add(key)
                out.zero_()
                for _ in range(3):
                    launch(plan, out)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(K):
                    launch(plan, out)
                e1.record()
                torch.cuda.synchronize()
                if rowsum:
                    ok = plan.status() == tsx.TSX_OK and bool(((out - ref).abs() <= tol).all())
                else:
                    ok = plan.status() == tsx.TSX_OK and torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
                plan.close()
                sec = e0.elapsed_time(e1) / 1e3 / K
                lines.append({"sweep": w.name, "mode": args.mode, "op": w.op, "variant": variant, "box": list(box),
                              "stages": st, "threads": info["threads"], "grid": info["grid"],
                              "ctas_per_sm": info["ctas_per_sm"], "gbs": round(nbytes / sec / 1e9, 1),
                              "same_as_workload_plan": bool(ok)})
    lines.sort(key=lambda d: -d["gbs"])
    return lines


def run_reference(args, w, stages, variant):
    """The reference arm: the oracle, as it stands, on the host's cores.  Each
    step is one bounded contiguous sample of the workload at a random offset,
    cut into element ranges over every host core; one more sample is timed on
    a single thread for scale."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle

    K, W = args.steps, args.warmup
    cores = oracle.host_cores()
    oracle.build()
    probe = np.arange(0, min(w.elems, 1 << 16), dtype=np.uint64)
    ins = w.inputs_at(probe)
    t0 = time.perf_counter()
    oracle.ewise(w.op, w.dtype, *ins)
    per_elem = (time.perf_counter() - t0) / probe.size
    # about 1 s of single-thread oracle work per step (input generation comes
    # on top), at most 2^24 elements: the whole run stays within a few minutes
    n = int(max(1024, min(w.elems, 1 << 24, 1.0 / max(per_elem, 1e-10))))
    # up to 16 samples at random offsets, generated before the timing and
    # taken in turn (generating a fresh sample for each of thousands of steps
    # took longer than the oracle itself)
    rng = np.random.default_rng(0)
    pool = [w.inputs_range(int(rng.integers(0, max(1, w.elems - n))), n) for _ in range(min(W + K, 16))]
    total_bytes, total_s = 0, 0.0
    for k in range(W + K):
        x = pool[k % len(pool)]
        t0 = time.perf_counter()
        oracle.ewise_parallel(w.op, w.dtype, *x, threads=cores)
        dt = time.perf_counter() - t0
        if k >= W:
            total_s += dt
            total_bytes += (w.n_in + 1) * n * ti.ELEM_SIZE[w.dtype]
    value = total_bytes / total_s / 1e9
    t0 = time.perf_counter()
    oracle.ewise(w.op, w.dtype, *x)
    one = (w.n_in + 1) * n * ti.ELEM_SIZE[w.dtype] / (time.perf_counter() - t0) / 1e9
    sample = (f"{n} contiguous elements of {w.name} per step ({len(pool)} samples at random offsets, taken in "
              f"turn), C oracle cut into element ranges over {cores} host threads")
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(total_s / K * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[w.dtype], "data": "synthetic",
        "config": {"workload": w.name, "op": w.op, "rows": w.rows, "cols": w.cols,
                   "box": [w.box_rows, w.box_cols], "stages": stages, "variant": variant},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "single_core": {"value": round(one, 4), "unit": "GB/s", "cores": 1,
                                         "sample": f"one more sample of {n} elements on one thread"}},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    w = ti.WORKLOADS[args.workload]
    if args.rows is not None:
        w = w.with_rows(args.rows)
    if args.box is not None:
        from dataclasses import replace

        w = replace(w, box_rows=args.box[0], box_cols=args.box[1])
    if args.op is not None:
        from dataclasses import replace

        w = replace(w, op=args.op)
    stages = args.stages if args.stages is not None else w.default_stages
    variant = args.variant or w.variant
    if args.sweep:
        for line in run_sweep(args, w, stages, variant):
            print(json.dumps(line), flush=True)
        return 0
    if args.impl == "reference":
        res = run_reference(args, w, stages, variant)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    res, td, rank = run_ours(args, w, stages, variant)
    check = res.pop("_check", None)
    second_data = res.pop("_second_out", None)
    if rank == 0:
        if not args.no_cpu_baseline:
            import oracle

            cores = oracle.host_cores()
            if check is not None:
                ins, device_out = check
            else:
                ins, device_out = w.inputs(), None
            res["cpu_baseline"], parity = cpu_baseline(w, ins, device_out, args.cpu_seconds, cores)
            if parity is not None:
                res["parity"] = parity
            if second_data is not None:
                second_checks(args, res["workloads"][SECOND_WORKLOAD], second_data, cores)
        print(json.dumps(res), flush=True)
    barrier(td)
    if td is not None:
        td.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
