"""The C ABI on the host: the library loads, exports every declared symbol,
and its planner agrees with the oracle's structure models (no GPU needed)."""

import ctypes
import glob
import itertools
import os
import re

import pytest

from oracle import structure as st

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def tsx():
    import __graft_entry__

    __graft_entry__.build()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _declared_functions():
    """Every function any header under include/ declares."""
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(tsx_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("tsx_plan_create", "tsx_ewise", "tsx_plan_destroy", "tsx_plan_status", "tsx_last_error",
                     "tsx_reduce_rows", "tsx_ewise_noalloc", "tsx_plan_tune", "tsx_debug_trace"):
        assert required in names


def test_library_exports_every_declared_symbol(tsx):
    lib = ctypes.CDLL(tsx.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_uses_the_c_names(tsx):
    for n in _declared_functions():
        assert hasattr(tsx, n), n


def test_calls_on_a_null_plan_are_invalid(tsx):
    """Host-side argument checks that need no GPU."""
    info = tsx.tsx_plan_info()
    assert tsx.tsx_plan_tune(None, 0, None, None, None, None, None, 10, ctypes.byref(info)) == tsx.TSX_ERR_INVALID
    assert tsx.tsx_ewise(None, 0, None, None, None, None, None) == tsx.TSX_ERR_INVALID
    assert tsx.tsx_plan_get_info(None, 0, ctypes.byref(info)) == tsx.TSX_ERR_INVALID


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_query_matches_oracle_split_and_encode(tsx, dtype):
    es = st.ELEM_SIZE[dtype]
    for br, bc, variant in itertools.product((1, 7, 8, 32, 64, 128, 256, 300, 512), (8, 16, 32, 64, 128, 192, 256),
                                             ("tma", "tma_rank3")):
        rows, cols = 1000, 4096
        mode = "rank3" if variant == "tma_rank3" else "rank2"
        sp = st.split(dtype, br, bc, mode, cols=cols)
        why = ""
        try:
            q = tsx.query(dtype, rows, cols, (br, bc), 2, variant, "add")
        except tsx.TsxError as e:
            q, why = None, str(e)
        if sp is None:
            assert q is None, (br, bc, variant)
            continue
        if q is None:
            # a legal split the library declines for one of its own limits:
            # the stages do not fit in shared memory, or (rank 3) the atoms of
            # a swizzled box would not each start on the 1024-byte period
            assert "shared memory" in why or "1024" in why, (br, bc, variant, why)
            continue
        assert q["loads_per_operand"] == sp.loads_per_operand
        assert q["bytes_per_load"] == sp.bytes_per_load
        assert q["tx_bytes"] == sp.tx_bytes(2)
        assert q["inner_elems"] == sp.inner_elems and q["atoms"] == sp.atoms
        assert q["rows_per_load"] == sp.rows_per_load and q["row_chunks"] == sp.row_chunks
        enc = st.encode_args(dtype, rows, cols, sp)
        rank = enc[1]
        assert q["rank"] == rank
        assert q["global_dim"][:rank] == list(enc[2:2 + rank])
        assert q["global_stride_bytes"][:rank - 1] == list(enc[2 + rank:1 + 2 * rank])
        assert q["box_dim"][:rank] == list(enc[1 + 2 * rank:1 + 3 * rank])
        assert (q["interleave"], q["swizzle"], q["l2_promotion"], q["oob_fill"]) == enc[-4:]


def test_query_mixed_variant_stages_all_but_b(tsx):
    """The mixed variant stages a (and c) through TMA; b is read directly,
    so expect_tx counts one operand fewer for binary ops and fma."""
    for op, n_tma in (("copy", 1), ("sqrt", 1), ("add", 1), ("mul", 1), ("fma", 2)):
        q = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma_mixed", op)
        sp = st.split("f32", 8, 128)
        assert q["tx_bytes"] == sp.tx_bytes(n_tma)
        assert q["stage_bytes"] == n_tma * q["slot_bytes"]
        full = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", op)
        assert (q["loads_per_operand"], q["box_dim"], q["swizzle"]) == \
            (full["loads_per_operand"], full["box_dim"], full["swizzle"])


def test_query_rank3_demo_tuple(tsx):
    """The 8x256 float16 tile with the 128-B swizzle: the encode arguments
    printed by the TVM page ("copy_async -> tma", Generated TIRx IR)."""
    q = tsx.query("f16", 8, 256, (8, 256), 1, "tma_rank3", "copy")
    got = (3, *q["global_dim"][:3], *q["global_stride_bytes"][:2], *q["box_dim"][:3], *q["element_strides"][:3],
           q["interleave"], q["swizzle"], q["l2_promotion"], q["oob_fill"])
    assert got == (3, 64, 8, 4, 512, 128, 64, 8, 4, 1, 1, 1, 0, 3, 2, 0)


def test_query_workload_plans(tsx):
    q = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "fma")
    assert (q["loads_per_operand"], q["tx_bytes"], q["box_dim"][:2]) == (4, 12288, [32, 8])
    q = tsx.query("bf16", 16384, 16384, (128, 128), 4, "tma", "exp")
    assert (q["loads_per_operand"], q["tx_bytes"], q["box_dim"][:2]) == (2, 32768, [64, 128])
    q = tsx.query("f32", 500, 4096, (32, 32), 2, "tma", "sqrt")
    assert (q["vec"], q["tiles"]) == (4, 16 * 128)
    # + the producer warp and the store warps
    assert q["block_threads"] == q["threads"] + 32 * (1 + q["store_warps"])


def test_query_partition_of_the_smem_sqrt_demo(tsx):
    """With 256 elementwise threads, a 32x32 float32 tile is one round of
    float4 vectors (TVM "elementwise -> smem", Algorithm step 2)."""
    q = tsx.query("f32", 500, 4096, (32, 32), 2, "tma", "sqrt", tuning={"threads": 256})
    assert (q["vec"], q["outer"], q["threads"]) == (4, 1, 256)


def test_query_default_threads_share_the_sm(tsx):
    """About 256 elementwise threads per SM, split over the CTAs that fit in
    its shared memory, 2 to 8 compute warps per CTA."""
    q = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "fma")      # 4 CTAs / SM
    assert (q["threads"], q["block_threads"]) == (64, 128)
    assert tsx.query("bf16", 16384, 16384, (128, 128), 3, "tma", "exp")["threads"] == 128   # 2 CTAs / SM
    assert tsx.query("bf16", 16384, 16384, (128, 128), 4, "tma", "exp")["threads"] == 256   # 1 CTA / SM
    assert tsx.query("f32", 500, 4096, (32, 32), 2, "tma", "sqrt")["threads"] == 64          # many small CTAs
    assert tsx.query("f16", 500, 4096, (128, 32), 2, "ldgsts", "sqrt")["threads"] == 128


def test_query_partition_matches_oracle(tsx):
    # TMA elementwise stage: 16-byte vectors over 256 threads
    for dtype, br, bc in (("f32", 32, 32), ("f16", 64, 64), ("f32", 8, 128), ("bf16", 128, 128)):
        q = tsx.query(dtype, 1024, 4096, (br, bc), 2, "tma", "copy")
        want = st.partition(br * bc, q["threads"], st.ELEM_SIZE[dtype], run_bytes=bc * st.ELEM_SIZE[dtype],
                            align_bytes=16)
        assert (q["vec"], q["outer"]) == want
    # cp.async: 128x32 fp16 over 128 threads -> 16-byte copies, vec 8, outer 4
    q = tsx.query("f16", 500, 4096, (128, 32), 2, "ldgsts", "sqrt")
    assert q["threads"] == 128 and q["copy_vec_bytes"] == 16
    assert st.partition(128 * 32, 128, 2, 64, 16, st.LDGSTS_VEC_BITS) == (8, 4)
    assert (q["copy_vec_bytes"] // 2, (128 * 32 * 2) // (q["copy_vec_bytes"] * q["threads"])) == (8, 4)
    # copy width narrows with the row pitch (8-byte and 4-byte rows)
    assert tsx.query("f16", 64, 4100, (8, 4), 2, "ldgsts", "copy")["copy_vec_bytes"] == 8
    assert tsx.query("f16", 64, 4098, (8, 2), 2, "ldgsts", "copy")["copy_vec_bytes"] == 4


@pytest.mark.parametrize("args,code", [
    (("f32", 100, 102, (8, 32), 2, "tma", "copy"), -2),       # row pitch 408 B: not a 16-B multiple
    (("f32", 100, 128, (8, 40), 2, "tma", "copy"), -2),       # 160-B tile row
    (("f32", 100, 128, (257, 32), 2, "tma", "copy"), -2),     # 257 rows: no equal chunks <= 256
    (("f32", 100, 128, (8, 32), 0, "tma", "copy"), -2),       # stages < 1
    (("f32", 100, 128, (8, 32), 17, "tma", "copy"), -2),      # stages > 16
    (("f32", 100, 128, (0, 32), 2, "tma", "copy"), -2),       # empty box
    (("f16", 8, 100, (8, 256), 1, "tma_rank3", "copy"), -2),  # cols not a whole number of atoms
    (("f16", 64, 4097, (8, 1), 2, "ldgsts", "copy"), -2),     # 2-byte rows: below the 4-byte cp_size
    (("f32", 1 << 31, 128, (8, 32), 2, "tma", "copy"), -2),   # rows >= 2^31
    (("f32", 100, 128, (256, 256), 4, "tma", "fma"), -2),     # stages do not fit in shared memory
    (("f32", -1, 128, (8, 32), 2, "tma", "copy"), -1),
    (("f32", 100, 128, (8, 32), 2, "tma", 9), -1),            # unknown op
])
def test_query_declines(tsx, args, code):
    with pytest.raises(tsx.TsxError) as ei:
        tsx.query(*args)
    assert ei.value.code == code
    assert tsx.tsx_last_error()


def test_query_accumulate_flag(tsx):
    acc = tsx.TSX_ACCUMULATE
    q = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", tsx.OPS["fma"] | acc)
    assert q["tx_bytes"] == 12288 and q["op"] == tsx.OPS["fma"]
    tsx.query("f16", 64, 256, (8, 256), 2, "tma_rank3", tsx.OPS["copy"] | acc)
    for variant in ("ldgsts", "sync", "tma_mixed"):
        with pytest.raises(tsx.TsxError) as ei:
            tsx.query("f32", 64, 256, (8, 64), 2, variant, tsx.OPS["add"] | acc)
        assert ei.value.code == tsx.TSX_ERR_UNSUPPORTED
    with pytest.raises(tsx.TsxError) as ei:
        tsx.query("f32", 64, 256, (8, 64), 2, "tma", tsx.OPS["add"] | 0x200)
    assert ei.value.code == tsx.TSX_ERR_INVALID


def test_query_pitched_rows(tsx):
    """Rows `pitch` elements apart: the tensor map's row stride is the pitch,
    which TMA needs to be a multiple of 16 bytes; the copy variants narrow
    their width to what divides it."""
    q = tsx.query("f32", 100, 100, (8, 32), 2, "tma", "copy", pitch=104)
    assert q["pitch"] == 104 and q["global_stride_bytes"][0] == 416 and q["global_dim"][:2] == [100, 100]
    q = tsx.query("f16", 8, 256, (8, 256), 1, "tma_rank3", "copy", pitch=320)
    assert q["global_stride_bytes"][:2] == [640, 128]
    with pytest.raises(tsx.TsxError) as ei:
        tsx.query("f32", 100, 100, (8, 32), 2, "tma", "copy", pitch=102)        # 408-byte rows
    assert ei.value.code == tsx.TSX_ERR_UNSUPPORTED
    with pytest.raises(tsx.TsxError) as ei:
        tsx.query("f32", 100, 100, (8, 32), 2, "tma", "copy", pitch=96)         # shorter than a row
    assert ei.value.code == tsx.TSX_ERR_INVALID
    assert tsx.query("f16", 64, 64, (8, 64), 2, "ldgsts", "copy", pitch=68)["copy_vec_bytes"] == 8
    assert tsx.query("f16", 64, 64, (8, 64), 2, "sync", "copy", pitch=66)["copy_vec_bytes"] == 4
    assert tsx.query("f32", 100, 128, (8, 32), 2, "tma", "copy")["pitch"] == 128


def test_query_promoted_matches_oracle(tsx):
    """One box spans the tile row, its element widened along 1 -> 2 -> 4 ->
    8 bytes until the row holds at most 256 (oracle: structure.promote)."""
    n = 0
    for dtype, es in st.ELEM_SIZE.items():
        for bc in (8, 64, 128, 200, 256, 384, 512, 768, 1024, 2048):
            for cols in (4096, 4100, 1000):
                row_bytes, cols_bytes = bc * es, cols * es
                pes = st.promote(es, row_bytes, cols_bytes) if row_bytes % 16 == 0 else None
                try:
                    q = tsx.query(dtype, 64, cols, (8, bc), 2, "tma_promoted", "add")
                except tsx.TsxError as e:
                    assert pes is None or "shared memory" in str(e) or cols_bytes % 16, (dtype, bc, cols, str(e))
                    continue
                assert pes is not None, (dtype, bc, cols)
                assert q["tma_elem_bytes"] == pes and q["swizzle"] == 0 and q["atoms"] == 1
                assert q["box_dim"][:2] == [row_bytes // pes, 8]
                assert q["global_dim"][:2] == [cols_bytes // pes, 64]
                assert q["loads_per_operand"] == 1 and q["tx_bytes"] == 2 * 8 * row_bytes
                n += 1
    assert n > 20


def test_query_empty_tensor_is_legal(tsx):
    q = tsx.query("f32", 0, 128, (8, 32), 2, "tma", "copy")
    assert q["tiles"] == 0


def test_query_store_warps_never_exceed_the_stages(tsx):
    """A store warp's parity wait is exact only if the stage's previous phase
    has completed, which holds when there are no more store warps than
    stages: the planner clamps the knob."""
    for stages in (1, 2, 3):
        q = tsx.query("f32", 64, 1024, (8, 128), stages, "tma", "add", tuning={"store_warps": 2})
        assert q["store_warps"] == min(2, stages)
        assert q["block_threads"] == q["threads"] + 32 * (1 + q["store_warps"])
    with pytest.raises(tsx.TsxError) as ei:
        tsx.query("f32", 64, 1024, (8, 128), 2, "tma", "add", tuning={"store_warps": 3})
    assert ei.value.code == tsx.TSX_ERR_INVALID


@pytest.mark.parametrize("op,stages,box,want", [
    # (store warps, lag, wait style: 1 every lane, 2 lane 0)
    ("fma", 2, (32, 128), (2, 0, 1)), ("fma", 3, (32, 128), (1, 1, 1)), ("fma", 4, (32, 128), (1, 1, 1)),
    ("fma", 6, (32, 128), (1, 2, 1)),
    ("exp", 2, (128, 128), (1, 0, 2)),         # 32 KB tiles stored in two groups: one warp
    ("exp", 2, (64, 128), (2, 0, 2)), ("exp", 3, (128, 128), (1, 1, 2)), ("exp", 4, (128, 128), (2, 0, 2)),
    ("exp", 4, (32, 128), (1, 1, 2)),         # stages under 16 KB keep lag 1
    ("exp", 8, (32, 128), (1, 2, 2)), ("sqrt", 4, (128, 128), (2, 0, 2)),
    ("copy", 2, (32, 128), (2, 0, 1)), ("copy", 4, (128, 128), (1, 1, 1)), ("mul", 3, (32, 128), (1, 1, 1)),
    ("exp", 1, (32, 128), (1, 0, 2)),
])
def test_query_store_schedule(tsx, op, stages, box, want):
    """The planner's store side per op, stage count and stage size, and the
    knobs that override it (the table is the planner's, from GB300
    measurements)."""
    q = tsx.query("bf16", 256, 4096, box, stages, "tma", op)
    assert (q["store_warps"], q["store_lag"], q["role_wait"]) == want
    f = tsx.query("bf16", 256, 4096, box, stages, "tma", op,
                  tuning={"store_warps": 1, "store_lag": 1, "role_wait": 1})
    assert (f["store_warps"], f["store_lag"], f["role_wait"]) == (1, 1, 1)


def test_query_two_stage_rings(tsx):
    """Two-stage rings on streams of 8192 tiles or more share 512 compute
    threads per SM (256 for copy) among enough CTAs for about 96 KB of
    stages per SM (copy, add, mul), 128 KB (sqrt, exp) or 144 KB (fma),
    halves rounding up; the CTA cap shows in a plan's launch on a GPU.
    Short streams, other variants and forced knobs keep the usual share."""
    big = ("bf16", 16384, 16384)
    assert tsx.query(*big, (128, 128), 2, "tma", "exp")["threads"] == 256    # 2 CTAs of 64 KB
    assert tsx.query(*big, (128, 128), 2, "tma", "sqrt")["threads"] == 256
    assert tsx.query(*big, (64, 128), 2, "tma", "exp")["threads"] == 128     # 4 CTAs of 32 KB
    assert tsx.query(*big, (128, 128), 2, "tma", "copy")["threads"] == 128   # 1.5 rounds up to 2
    assert tsx.query(*big, (128, 128), 2, "tma", "mul")["threads"] == 512    # one CTA of 128 KB
    assert tsx.query(*big, (32, 128), 2, "tma", "add")["threads"] == 160     # 3 CTAs of 32 KB
    assert tsx.query(*big, (32, 128), 2, "tma", "fma")["threads"] == 160     # 3 CTAs of 48 KB
    assert tsx.query(*big, (64, 64), 2, "tma_rank3", "add")["threads"] == 160
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 2, "tma", "copy")["threads"] == 32   # 12 CTAs wanted
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 2, "tma", "fma")["threads"] == 64    # 6 CTAs of 24 KB
    assert tsx.query("f16", 1024, 8192, (64, 64), 2, "tma", "add")["threads"] == 64       # 2048 tiles
    assert tsx.query("f32", 500, 4096, (32, 32), 2, "tma", "sqrt")["threads"] == 64       # 2048 tiles
    assert tsx.query(*big, (128, 128), 2, "ldgsts", "exp")["threads"] == 512
    assert tsx.query(*big, (128, 128), 2, "tma", "exp", tuning={"ctas_per_sm": 3})["threads"] == 64
    assert tsx.query(*big, (128, 128), 3, "tma", "exp")["threads"] == 128    # three stages
    assert tsx.query(*big, (64, 512), 2, "tma_promoted", "exp")["threads"] == 512   # 8192 tiles, one CTA


@pytest.mark.parametrize("op,stages,want", [
    ("copy", 2, 2), ("copy", 3, 1), ("copy", 4, 2), ("copy", 5, 1), ("copy", 1, 1),
    ("add", 3, 2), ("add", 5, 2), ("exp", 3, 2), ("add", 1, 1),
])
def test_query_two_store_warps_and_the_stage_count(tsx, op, stages, want):
    """Two store warps need at most as many warps as stages; for copy, whose
    store waits on the loads' barriers (completed in any order across
    stages), they must also divide the stage count, so that a stage's
    previous tile was the same warp's."""
    q = tsx.query("bf16", 256, 4096, (32, 128), stages, "tma", op, tuning={"store_warps": 2, "store_lag": 0})
    assert q["store_warps"] == want


def test_query_mixed_prefetch_lead(tsx):
    """The mixed variant's L2 prefetch of b keeps about 40 KB of prefetched b
    per SM: T = max(1, round(40 KB / (b tile bytes x CTAs))) tiles of lead,
    of which the producer's own S - 2 come for free.  tsx_plan_query counts
    the CTAs that shared memory alone fits; the knob overrides."""
    for dtype, box, stages in (("f32", (8, 128), 2), ("f32", (8, 128), 4), ("bf16", (128, 128), 2),
                               ("bf16", (128, 128), 3), ("bf16", (64, 128), 2)):
        q = tsx.query(dtype, 1024, 1 << 16, box, stages, "tma_mixed", "mul")
        ctas = 233472 // (q["smem_bytes"] + 1024)
        per_sm = q["slot_bytes"] * ctas
        lead = max(1, (2 * 40960 + per_sm) // (2 * per_sm))
        assert q["b_prefetch"] == max(0, min(8, lead - (stages - 2))), (dtype, box, stages)
    assert tsx.query("f32", 1024, 1 << 16, (8, 128), 4, "tma_mixed", "mul", tuning={"b_prefetch": 5})["b_prefetch"] == 5
    assert tsx.query("f32", 1024, 1 << 16, (8, 128), 4, "tma", "mul")["b_prefetch"] == 0


def test_query_tile_order(tsx):
    """TMA copies take tiles in the dynamic order unless told otherwise (the
    last `dynamic_share` percent claimed from a counter: all past the static
    prefix for tiles of 16 KB or more, the last quarter for smaller ones);
    every other op, and the reduce-store, keep the static order; the
    ablations and row sums have no tile order."""
    q = tsx.query("bf16", 16384, 16384, (128, 128), 3, "tma", "copy")
    assert (q["tile_order"], q["dynamic_share"]) == (2, 100)
    assert tsx.query("bf16", 16384, 16384, (128, 128), 3, "tma_rank3", "copy")["tile_order"] == 2
    assert tsx.query("bf16", 16384, 16384, (128, 128), 3, "tma_mixed", "copy")["tile_order"] == 2
    q = tsx.query("bf16", 16384, 16384, (128, 128), 3, "tma", "copy", tuning={"dynamic_share": 25})
    assert (q["tile_order"], q["dynamic_share"]) == (2, 25)
    q = tsx.query("bf16", 16384, 16384, (128, 128), 3, "tma", "copy", tuning={"tile_order": 1})
    assert (q["tile_order"], q["dynamic_share"]) == (1, 0)
    for op in ("sqrt", "exp", "add", "mul", "fma"):
        q = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", op, tuning={"tile_order": 2})
        assert (q["tile_order"], q["dynamic_share"]) == (1, 0), op
    q = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "copy")      # 4 KB tiles: the last quarter claimed
    assert (q["tile_order"], q["dynamic_share"]) == (2, 25)
    q = tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "copy", tuning={"dynamic_share": 60})
    assert (q["tile_order"], q["dynamic_share"]) == (2, 60)
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 4, "ldgsts", "copy")["tile_order"] == 0
    with pytest.raises(tsx.TsxError, match="tile_order"):
        tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "copy", tuning={"tile_order": 3})
    with pytest.raises(tsx.TsxError, match="dynamic_share"):
        tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "copy", tuning={"dynamic_share": 101})


def test_query_store_split(tsx):
    """Two groups of boxes for ops with a compute step, an even number of
    boxes per tile and every operand staged; by default for sqrt and exp
    with tiles of 16 KB or more."""
    q = lambda *a, **k: tsx.query(*a, **k)["compute_groups"]
    assert q("bf16", 16384, 16384, (128, 128), 2, "tma", "exp") == 2
    assert q("bf16", 16384, 16384, (128, 128), 3, "tma", "sqrt") == 2
    assert q("bf16", 16384, 16384, (64, 64), 3, "tma", "exp") == 1      # 8 KB tiles
    assert q("bf16", 16384, 16384, (128, 128), 3, "tma", "mul") == 1
    assert q("f32", 128, 1 << 20, (8, 128), 4, "tma", "exp") == 1       # 4 KB tiles
    assert q("bf16", 16384, 16384, (128, 128), 2, "tma", "exp", tuning={"store_split": 1}) == 1
    assert q("bf16", 16384, 16384, (128, 128), 2, "tma", "exp", tuning={"store_split": 2}) == 2
    assert q("bf16", 16384, 16384, (128, 128), 2, "tma_rank3", "exp", tuning={"store_split": 2}) == 1  # 1 box
    assert q("bf16", 16384, 16384, (128, 128), 2, "tma", "copy", tuning={"store_split": 2}) == 1
    assert q("f32", 128, 1 << 20, (8, 128), 4, "tma", "fma", tuning={"store_split": 2}) == 2
    assert q("f32", 128, 1 << 20, (8, 128), 4, "tma_mixed", "fma", tuning={"store_split": 2}) == 1
    assert q("f32", 128, 1 << 20, (8, 96), 4, "tma", "fma", tuning={"store_split": 2}) == 1   # 3 boxes
    assert q("f32", 128, 1 << 20, (8, 128), 4, "ldgsts", "fma", tuning={"store_split": 2}) == 0
    with pytest.raises(tsx.TsxError, match="store_split"):
        q("f32", 128, 1 << 20, (8, 128), 4, "tma", "fma", tuning={"store_split": 3})


def test_query_small_exp_rings(tsx):
    """Rings of four or more small sqrt / exp stages take about 256 compute
    threads per SM (576 for fp32 sqrt) over enough CTAs for about 144 KB of
    stages; shorter rings keep the usual share."""
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "exp")["threads"] == 32    # 9 CTAs of 16 KB
    assert tsx.query("f32", 128, 1 << 20, (8, 256), 4, "tma", "exp")["threads"] == 64    # 4 CTAs of 32 KB
    assert tsx.query("bf16", 16384, 16384, (64, 64), 6, "tma", "sqrt")["threads"] == 64  # 3 CTAs of 48 KB
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "sqrt")["threads"] == 64   # 9 CTAs, 576 threads
    assert tsx.query("f32", 128, 1 << 20, (16, 128), 8, "tma", "sqrt")["threads"] == 288  # 2 CTAs of 64 KB
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 3, "tma", "exp")["threads"] == 64    # three stages
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "exp", tuning={"threads": 128})["threads"] == 128


def test_query_mixed_threads(tsx):
    """The mixed variant's add, mul and fma take as few compute threads as
    hold b a tile ahead (four 16-byte units each); given knobs win."""
    for S in (2, 4, 6, 8):
        assert tsx.query("f32", 128, 1 << 20, (8, 128), S, "tma_mixed", "fma")["threads"] == 64   # 256 units
    assert tsx.query("f32", 128, 1 << 20, (8, 64), 4, "tma_mixed", "fma")["threads"] == 32
    assert tsx.query("f32", 128, 1 << 20, (16, 128), 4, "tma_mixed", "add")["threads"] == 128
    assert tsx.query("bf16", 16384, 16384, (64, 128), 4, "tma_mixed", "mul")["threads"] == 256
    assert tsx.query("bf16", 16384, 16384, (128, 128), 3, "tma_mixed", "mul")["threads"] == 512
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 6, "tma_mixed", "fma", tuning={"threads": 128})["threads"] == 128


def test_query_add_mul_rings(tsx):
    """add and mul on long streams from three stages on take enough CTAs for
    about 144 KB of stages per SM when that leaves two or more; short
    streams (the stated fp16 add workload) and single-CTA rings keep the
    usual share, and two-stage rings have a rule of their own."""
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 4, "tma", "add")["threads"] == 64     # 4 CTAs of 32 KB
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 3, "tma", "mul")["threads"] == 32     # 6 CTAs of 24 KB
    assert tsx.query("bf16", 16384, 16384, (64, 64), 4, "tma", "add")["threads"] == 128   # 2 CTAs of 64 KB
    assert tsx.query("bf16", 16384, 16384, (64, 64), 6, "tma", "add")["threads"] == 128   # the usual share: 1 CTA would be the target
    assert tsx.query("f16", 1024, 8192, (64, 64), 3, "tma", "add")["threads"] == 64        # 2048 tiles
    assert tsx.query("f32", 128, 1 << 20, (8, 128), 2, "tma", "add")["threads"] == 64     # two stages: their own rule
