"""Python binding of libtsx: tile-elementwise streaming on GB300.

Argument marshalling only: every step of the path runs in the CUDA library
``libtsx.so`` (built from ``csrc/`` by ``_build.py``).  There is no Python or
CPU fallback; importing this module fails loudly when the library is absent.

The C functions are exposed under their own names (``tsx_plan_create``,
``tsx_ewise``, ``tsx_plan_destroy``, ``tsx_plan_status``, ``tsx_last_error``,
``tsx_plan_query``, ``tsx_plan_get_info``, ...) with plain-integer arguments;
``Plan`` wraps them for torch tensors::

    plan = Plan("bf16", rows, cols, box=(128, 128), stages=4, variant="tma")
    plan.ewise("exp", a, out=out)          # a, out: CUDA tensors, [rows, cols]

PyTorch only supplies device memory and the current stream.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtsx.so")

DTYPES = {"f16": 0, "bf16": 1, "f32": 2}
VARIANTS = {"tma": 0, "ldgsts": 1, "sync": 2, "tma_rank3": 3, "tma_mixed": 4, "tma_promoted": 5}
OPS = {"copy": 0, "sqrt": 1, "exp": 2, "add": 3, "mul": 4, "fma": 5}
TSX_ACCUMULATE = 0x100   # OR into an op: out += op(a, b, c) by TMA reduce-store
TSX_ROW_SUMS = 0x200     # OR into an op for tsx_plan_get_info: the launch of tsx_reduce_rows
ARITY = {"copy": 1, "sqrt": 1, "exp": 1, "add": 2, "mul": 2, "fma": 3}
STATUS = {0: "TSX_OK", -1: "TSX_ERR_INVALID", -2: "TSX_ERR_UNSUPPORTED", -3: "TSX_ERR_ALIGN",
          -4: "TSX_ERR_CUDA", -5: "TSX_ERR_TIMEOUT", -6: "TSX_ERR_NOMEM"}
TSX_OK, TSX_ERR_INVALID, TSX_ERR_UNSUPPORTED, TSX_ERR_ALIGN, TSX_ERR_CUDA, TSX_ERR_TIMEOUT, TSX_ERR_NOMEM = \
    0, -1, -2, -3, -4, -5, -6


class TsxError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code


class tsx_plan_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("dtype", "variant", "op", "n_in", "elem_size",
                                               "box_rows", "box_cols", "stages")] + \
               [(n, ctypes.c_int64) for n in ("rows", "cols", "tiles", "tiles_r", "tiles_c")] + \
               [(n, ctypes.c_int32) for n in ("inner_elems", "inner_bytes", "atoms", "rows_per_load",
                                               "row_chunks", "loads_per_operand", "bytes_per_load",
                                               "tx_bytes", "rank")] + \
               [("global_dim", ctypes.c_uint64 * 5), ("global_stride_bytes", ctypes.c_uint64 * 4),
                ("box_dim", ctypes.c_uint32 * 5), ("element_strides", ctypes.c_uint32 * 5)] + \
               [(n, ctypes.c_int32) for n in ("interleave", "swizzle", "l2_promotion", "oob_fill",
                                               "threads", "vec", "outer", "copy_vec_bytes",
                                               "slot_bytes", "stage_bytes", "smem_bytes",
                                               "ctas_per_sm", "grid", "sm_count", "block_threads")] + \
               [("pitch", ctypes.c_int64), ("tma_elem_bytes", ctypes.c_int32), ("store_lag", ctypes.c_int32),
                ("timeout_ms", ctypes.c_int32), ("store_warps", ctypes.c_int32), ("role_wait", ctypes.c_int32),
                ("b_prefetch", ctypes.c_int32), ("tile_order", ctypes.c_int32),
                ("dynamic_share", ctypes.c_int32), ("compute_groups", ctypes.c_int32)]

    def as_dict(self) -> dict:
        d = {}
        for name, _ in self._fields_:
            v = getattr(self, name)
            d[name] = list(v) if hasattr(v, "__len__") else int(v)
        return d


class tsx_tuning(ctypes.Structure):
    """Launch knobs of a plan (include/tsx.h); see ``tuning()``."""
    _fields_ = [(n, ctypes.c_int32) for n in ("threads", "ctas_per_sm", "store_lag", "l2_promotion", "timeout_ms",
                                               "checked", "store_warps", "role_wait", "b_prefetch",
                                               "tile_order", "dynamic_share", "store_split")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                          "(libtsx is the only implementation; there is no fallback)")
    L = ctypes.CDLL(LIB_PATH)
    L.tsx_plan_create.restype = ctypes.c_void_p
    L.tsx_plan_create.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int]
    L.tsx_ewise.restype = ctypes.c_int
    L.tsx_ewise.argtypes = [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5
    L.tsx_plan_create_pitched.restype = ctypes.c_void_p
    L.tsx_plan_create_pitched.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.tsx_plan_create_tuned.restype = ctypes.c_void_p
    L.tsx_plan_create_tuned.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(tsx_tuning)]
    L.tsx_plan_query_tuned.restype = ctypes.c_int
    L.tsx_plan_query_tuned.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(tsx_tuning),
                                       ctypes.c_int, ctypes.POINTER(tsx_plan_info)]
    L.tsx_tuning_defaults.restype = None
    L.tsx_tuning_defaults.argtypes = [ctypes.POINTER(tsx_tuning)]
    L.tsx_plan_query_pitched.restype = ctypes.c_int
    L.tsx_plan_query_pitched.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(tsx_plan_info)]
    L.tsx_plan_destroy.restype = None
    L.tsx_plan_destroy.argtypes = [ctypes.c_void_p]
    L.tsx_plan_status.restype = ctypes.c_int
    L.tsx_plan_status.argtypes = [ctypes.c_void_p]
    L.tsx_last_error.restype = ctypes.c_char_p
    L.tsx_last_error.argtypes = []
    L.tsx_plan_query.restype = ctypes.c_int
    L.tsx_plan_query.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(tsx_plan_info)]
    L.tsx_plan_get_info.restype = ctypes.c_int
    L.tsx_plan_get_info.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(tsx_plan_info)]
    L.tsx_reduce_rows.restype = ctypes.c_int
    L.tsx_reduce_rows.argtypes = [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5
    L.tsx_plan_tune.restype = ctypes.c_int
    L.tsx_plan_tune.argtypes = [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5 + \
                               [ctypes.c_int32, ctypes.POINTER(tsx_plan_info)]
    L.tsx_ewise_noalloc.restype = ctypes.c_int
    L.tsx_ewise_noalloc.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5 + \
                                   [ctypes.POINTER(ctypes.c_int)]
    L.tsx_debug_plan_enable_trace.restype = ctypes.c_int
    L.tsx_debug_plan_enable_trace.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    L.tsx_debug_plan_set_fault_tile.restype = ctypes.c_int
    L.tsx_debug_plan_set_fault_tile.argtypes = [ctypes.c_void_p, ctypes.c_int64]
    L.tsx_debug_noalloc_set_fault.restype = None
    L.tsx_debug_noalloc_set_fault.argtypes = [ctypes.c_int64, ctypes.c_int32]
    L.tsx_debug_stage_image.restype = ctypes.c_int
    L.tsx_debug_stage_image.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p]
    L.tsx_debug_trace.restype = ctypes.c_int
    L.tsx_debug_trace.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                  ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    return L


lib = _load()

# The C entry points under their own names (plain integers / addresses).
tsx_plan_create = lib.tsx_plan_create
tsx_plan_create_pitched = lib.tsx_plan_create_pitched
tsx_plan_create_tuned = lib.tsx_plan_create_tuned
tsx_plan_query_tuned = lib.tsx_plan_query_tuned
tsx_tuning_defaults = lib.tsx_tuning_defaults
tsx_plan_query_pitched = lib.tsx_plan_query_pitched
tsx_ewise = lib.tsx_ewise
tsx_plan_destroy = lib.tsx_plan_destroy
tsx_plan_status = lib.tsx_plan_status
tsx_plan_query = lib.tsx_plan_query
tsx_plan_get_info = lib.tsx_plan_get_info
tsx_reduce_rows = lib.tsx_reduce_rows
tsx_plan_tune = lib.tsx_plan_tune
# The plan-free, allocation-free form of tsx_ewise (device status word in a
# static device array; see include/tsx.h for who needs it and its limits).
tsx_ewise_noalloc = lib.tsx_ewise_noalloc
# Test hooks (include/tsx_debug.h): the schedule trace of traced launches and
# the host-planted load skip that makes a bounded device-side wait run out.
tsx_debug_trace = lib.tsx_debug_trace
tsx_debug_plan_enable_trace = lib.tsx_debug_plan_enable_trace
tsx_debug_plan_set_fault_tile = lib.tsx_debug_plan_set_fault_tile
tsx_debug_noalloc_set_fault = lib.tsx_debug_noalloc_set_fault
tsx_debug_stage_image = lib.tsx_debug_stage_image


def tsx_last_error() -> str:
    return lib.tsx_last_error().decode()


def _code(table: dict, key) -> int:
    return table[key] if isinstance(key, str) else int(key)


def tuning(**knobs) -> tsx_tuning:
    """A tsx_tuning with the planner's choices, except the knobs given
    (threads, ctas_per_sm, store_lag, l2_promotion, timeout_ms, checked, store_warps, role_wait,
    b_prefetch, tile_order, dynamic_share, store_split)."""
    t = tsx_tuning()
    tsx_tuning_defaults(ctypes.byref(t))
    for k, v in knobs.items():
        if k not in dict(tsx_tuning._fields_):
            raise TypeError(f"unknown tuning knob {k!r}")
        setattr(t, k, int(v))
    return t


def _tuning_ref(t):
    if t is None:
        return None
    return ctypes.byref(t if isinstance(t, tsx_tuning) else tuning(**t))


def query(dtype, rows, cols, box, stages, variant="tma", op="copy", pitch=None, tuning=None) -> dict:
    """The plan and launch shape the library would use (host only, no GPU).
    ``tuning``: a dict of knobs or a tsx_tuning (None: the planner's)."""
    info = tsx_plan_info()
    rc = tsx_plan_query_tuned(_code(DTYPES, dtype), rows, cols, cols if pitch is None else pitch, box[0], box[1],
                              stages, _code(VARIANTS, variant), _tuning_ref(tuning), _code(OPS, op),
                              ctypes.byref(info))
    if rc != TSX_OK:
        raise TsxError(rc, tsx_last_error())
    return info.as_dict()


_TORCH_DTYPE_NAME = {"torch.float16": "f16", "torch.bfloat16": "bf16", "torch.float32": "f32"}


class Plan:
    """A tsx plan bound to the current CUDA device."""

    def __init__(self, dtype: str, rows: int, cols: int, box=(32, 32), stages: int = 2, variant: str = "tma",
                 pitch: int | None = None, tuning=None):
        self.dtype, self.rows, self.cols = dtype, int(rows), int(cols)
        self.pitch = self.cols if pitch is None else int(pitch)
        self.box, self.stages, self.variant = (int(box[0]), int(box[1])), int(stages), variant
        h = tsx_plan_create_tuned(_code(DTYPES, dtype), self.rows, self.cols, self.pitch, self.box[0], self.box[1],
                                  self.stages, _code(VARIANTS, variant), _tuning_ref(tuning))
        if not h:
            raise TsxError(TSX_ERR_UNSUPPORTED, tsx_last_error())
        self.handle = h

    def _check(self, t, name):
        if t is None:
            return None
        if not t.is_cuda:
            raise TsxError(TSX_ERR_INVALID, f"{name} must be a CUDA tensor")
        if _TORCH_DTYPE_NAME.get(str(t.dtype)) != self.dtype:
            raise TsxError(TSX_ERR_INVALID, f"{name} has dtype {t.dtype}, the plan is {self.dtype}")
        if self.pitch == self.cols:
            if t.numel() != self.rows * self.cols or not t.is_contiguous():
                raise TsxError(TSX_ERR_INVALID, f"{name} must be a contiguous [{self.rows}, {self.cols}] tensor")
        elif (tuple(t.shape) != (self.rows, self.cols) or t.stride(-1) != 1
              or (self.rows > 1 and t.stride(0) != self.pitch)):
            raise TsxError(TSX_ERR_INVALID, f"{name} must be a [{self.rows}, {self.cols}] view with row stride "
                                            f"{self.pitch}")
        return t.data_ptr()

    def ewise_ptr(self, op, a: int, b: int | None, c: int | None, out: int, stream: int = 0) -> None:
        """tsx_ewise on raw device addresses (an int stream handle)."""
        rc = tsx_ewise(self.handle, _code(OPS, op), a, b, c, out, stream)
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())

    def ewise(self, op: str, a, b=None, c=None, out=None, stream=None, accumulate: bool = False):
        """out = op(a[, b[, c]]) on the current (or given) torch CUDA stream;
        with accumulate, out += op(...) (out must then be given)."""
        import torch

        if out is None:
            if accumulate:
                raise TsxError(TSX_ERR_INVALID, "accumulate needs an out tensor to add into")
            if self.pitch == self.cols:
                out = torch.empty_like(a)
            else:
                out = torch.empty(self.rows, self.pitch, dtype=a.dtype, device=a.device)[:, : self.cols]
        pa, pb, pc, po = (self._check(a, "a"), self._check(b, "b"), self._check(c, "c"), self._check(out, "out"))
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        code = _code(OPS, op) | (TSX_ACCUMULATE if accumulate else 0)
        self.ewise_ptr(code, pa, pb, pc, po, s.cuda_stream)
        return out

    def reduce_rows(self, op: str, a, b=None, c=None, out=None, stream=None):
        """fp32 row sums of op(a[, b[, c]]) over the plan's [rows, cols]."""
        import torch

        if out is None:
            out = torch.empty(self.rows, dtype=torch.float32, device=a.device)
        if out.dtype != torch.float32 or not out.is_cuda or out.numel() != self.rows:
            raise TsxError(TSX_ERR_INVALID, f"out must be a CUDA float32 tensor of {self.rows} elements")
        pa, pb, pc = self._check(a, "a"), self._check(b, "b"), self._check(c, "c")
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        rc = tsx_reduce_rows(self.handle, _code(OPS, op), pa, pb, pc, out.data_ptr(), s.cuda_stream)
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())
        return out

    def tune(self, op: str, a, b=None, c=None, out=None, launches: int = 10, stream=None) -> dict:
        """Time the op's candidate launch shapes on these operands and keep
        the fastest for the plan's later calls of `op` (tsx_plan_tune; out
        must not alias an input and ends holding op(a, b, c)).  Returns the
        launch kept, as info() gives it."""
        import torch

        if out is None:
            out = torch.empty_like(a) if self.pitch == self.cols else \
                torch.empty(self.rows, self.pitch, dtype=a.dtype, device=a.device)[:, : self.cols]
        pa, pb, pc, po = (self._check(a, "a"), self._check(b, "b"), self._check(c, "c"), self._check(out, "out"))
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        info = tsx_plan_info()
        rc = tsx_plan_tune(self.handle, _code(OPS, op), pa, pb, pc, po, s.cuda_stream, int(launches),
                           ctypes.byref(info))
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())
        return info.as_dict()

    def status(self) -> int:
        """Device-side status since the last call (reads and clears it)."""
        return tsx_plan_status(self.handle)

    def enable_trace(self, events_per_cta: int) -> None:
        """Test hook: later launches record their schedule (0: off)."""
        rc = tsx_debug_plan_enable_trace(self.handle, int(events_per_cta))
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())

    def set_fault_tile(self, tile: int) -> None:
        """Test hook: later launches skip the loads of `tile` (-1: none)."""
        rc = tsx_debug_plan_set_fault_tile(self.handle, int(tile))
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())

    def stage_image(self, a, tile: int):
        """Test hook: the raw shared-memory bytes of tile `tile` of `a` as the
        plan's TMA loads stage it (uint8 CUDA tensor of slot_bytes)."""
        import torch

        info = self.info("copy")
        img = torch.zeros(info["slot_bytes"], dtype=torch.uint8, device=a.device)
        s = torch.cuda.current_stream(a.device)
        rc = tsx_debug_stage_image(self.handle, self._check(a, "a"), int(tile), img.data_ptr(), s.cuda_stream)
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())
        return img

    def trace(self):
        """The schedule trace of the plan's last traced launch (after
        ``enable_trace``): uint32 [grid, events per CTA, 4]."""
        import numpy as np

        grid, per = ctypes.c_int32(), ctypes.c_int32()
        rc = tsx_debug_trace(self.handle, None, 0, ctypes.byref(grid), ctypes.byref(per))
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())
        buf = np.zeros((grid.value, per.value, 4), dtype=np.uint32)
        rc = tsx_debug_trace(self.handle, buf.ctypes.data, buf.size, None, None)
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())
        return buf

    def info(self, op: str = "copy", row_sums: bool = False) -> dict:
        """The plan and its launch for `op` (of reduce_rows with row_sums)."""
        info = tsx_plan_info()
        code = _code(OPS, op) | (TSX_ROW_SUMS if row_sums else 0)
        rc = tsx_plan_get_info(self.handle, code, ctypes.byref(info))
        if rc != TSX_OK:
            raise TsxError(rc, tsx_last_error())
        return info.as_dict()

    def close(self) -> None:
        if getattr(self, "handle", None):
            tsx_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
