"""Pins for the oracle's structure models against the values the pages print
and against brute force."""

import itertools

import pytest

from oracle import structure as st


# ------------------------------------------------------------ partition

def test_partition_smem_sqrt_demo():
    """TVM "elementwise -> smem", Algorithm step 2: 32x32 float32 over 256
    threads gives vec = 4, outer = 1."""
    assert st.partition(32 * 32, 256, 4, run_bytes=32 * 4, align_bytes=16) == (4, 1)


def test_partition_generated_ir_index():
    """Same page, Generated TIRx IR: element ``tid * 4 + vec`` of round 0."""
    for tid in (0, 1, 17, 255):
        for v in range(4):
            assert st.linear_element(0, tid, v, threads=256, vec=4) == tid * 4 + v


def test_partition_ldgsts_demo():
    """TVM "copy_async -> ldgsts", Algorithm step 1: 128x32 float16 over 128
    threads, cp_size capped at 16 B, gives vec = 8, outer = 4."""
    assert st.partition(128 * 32, 128, 2, run_bytes=32 * 2, align_bytes=16,
                        vec_bits=st.LDGSTS_VEC_BITS) == (8, 4)


@pytest.mark.parametrize("case,es,align,want", [
    ("float16 aligned", 2, 16, (8, 4)),
    ("float32 aligned", 4, 16, (4, 8)),
    ("8-B aligned only", 2, 8, (4, 8)),     # 8 B copies, outer doubles
    ("4-B aligned only", 2, 4, (2, 16)),    # 4 B copies, outer x4
    ("below 4 B", 2, 2, None),              # no legal cp_size: declines
])
def test_partition_ldgsts_table(case, es, align, want):
    """The table under "How inputs change the algorithm" on the ldgsts page:
    4096 elements over 128 threads."""
    got = st.partition(4096, 128, es, run_bytes=64, align_bytes=align, vec_bits=st.LDGSTS_VEC_BITS)
    assert got == want, case


def test_partition_brute_force_covers_region():
    """Every (round, thread, lane) hits a distinct element and all are hit."""
    for elems, threads, es in [(1024, 256, 4), (4096, 128, 2), (2048, 64, 2), (512, 32, 4)]:
        vec, outer = st.partition(elems, threads, es, run_bytes=128, align_bytes=16)
        seen = {st.linear_element(f, t, v, threads, vec)
                for f in range(outer) for t in range(threads) for v in range(vec)}
        assert seen == set(range(elems))


# ------------------------------------------------------------------ split

def test_split_box_rows_over_256_take_several_loads():
    """nvFuser PR #2833, Lowering Details: box dims are at most 256, so a
    taller tile takes several loads."""
    sp = st.split("f32", 512, 32)
    assert (sp.row_chunks, sp.rows_per_load, sp.loads_per_operand) == (2, 256, 2)
    assert st.split("f32", 256, 32).loads_per_operand == 1


def test_split_fma_workload_four_loads_per_stage():
    """The fp32 fma workload: an 8x128 stage tile of four 8x32 boxes."""
    sp = st.split("f32", 8, 128)
    assert (sp.inner_elems, sp.atoms, sp.rows_per_load, sp.loads_per_operand) == (32, 4, 8, 4)
    assert sp.bytes_per_load == 8 * 32 * 4
    assert sp.tx_bytes(3) == 3 * 4 * 1024 == 12288


def test_split_exp_workload_two_loads_per_stage():
    """The bf16 exp workload: a 128x128 tile as two 128x64 boxes."""
    sp = st.split("bf16", 128, 128)
    assert (sp.inner_elems, sp.rows_per_load, sp.loads_per_operand) == (64, 128, 2)
    assert sp.tx_bytes(1) == 2 * 128 * 64 * 2 == 32768


def test_split_brute_force_invariants():
    """expect_tx = bytes per load x loads = the whole stage tile (nvFuser PR
    #2833, Lowering Details); every box dim <= 256; the inner box fits the
    128-B swizzle atom (TVM "copy_async -> tma", What it accepts)."""
    for dtype, es in st.ELEM_SIZE.items():
        for br in (1, 7, 8, 31, 64, 100, 256, 300, 512, 768):
            for bc in (8, 16, 24, 32, 48, 64, 96, 128, 192, 256, 512):
                for mode in ("rank2", "rank3"):
                    sp = st.split(dtype, br, bc, mode, cols=4096)
                    if sp is None:
                        continue
                    for n_in in (1, 2, 3):
                        assert sp.tx_bytes(n_in) == n_in * br * bc * es
                    assert sp.inner_bytes <= 128 and sp.inner_bytes % 16 == 0
                    assert sp.rows_per_load <= 256 and sp.inner_elems <= 256 and sp.atoms <= 256
                    assert sp.rows_per_load * sp.row_chunks == br
                    assert sp.inner_elems * sp.atoms == bc


def test_split_declines():
    assert st.split("f16", 8, 4) is None        # 8-byte tile rows: not a 16-B multiple
    assert st.split("f32", 8, 40) is None       # 160 B: not a whole number of 128-B atoms
    assert st.split("f32", 257, 32) is None     # 257 rows cannot be cut into equal chunks <= 256
    assert st.split("f32", 0, 32) is None
    assert st.split("f16", 8, 256, "rank3", cols=100) is None   # row not a whole number of atoms


def test_promotion_chain():
    """TVM docs "copy_async -> tma": a box over 256 elements is widened along
    1 -> 2 -> 4 -> 8 bytes."""
    assert st.promote(2, 256 * 2, 4096) == 2          # 256 fp16: no promotion needed
    assert st.promote(2, 512 * 2, 4096) == 4          # 512 fp16 -> 256 four-byte elements
    assert st.promote(2, 1024 * 2, 4096) == 8         # 1024 fp16 -> 256 eight-byte elements
    assert st.promote(2, 2048 * 2, 8192) is None      # 512 eight-byte elements: declines
    assert st.promote(4, 512 * 4, 4096) == 8
    assert st.promote(1, 300, 600) == 2               # 1 -> 2 bytes: 150 elements
    assert st.promote(2, 520 * 2, 1040 * 2) == 8      # 1040 B rows: 4 B gives 260, 8 B gives 130
    assert st.promote(2, 514 * 2, 4112) is None       # 1028 B rows: 4 B gives 257, 8 B does not divide
    assert st.promote(2, 512 * 2, 2 * 1025) is None   # the tensor row (2050 B) is no whole number of 4 B
    for es in (1, 2, 4):
        for n in range(1, 3000):
            pes = st.promote(es, n * es, 4 * n * es)
            if pes is not None:
                assert pes in st.PROMOTION_CHAIN and pes >= es and (n * es) // pes <= 256
                smaller = [q for q in st.PROMOTION_CHAIN if es <= q < pes and (n * es) % q == 0]
                assert all((n * es) // q > 256 for q in smaller)


def test_encode_args_rank3_demo_tuple():
    """TVM "copy_async -> tma", Generated TIRx IR: the 8x256 float16 tile
    with the 128-B swizzle is one rank-3 load with exactly this encode."""
    sp = st.split("f16", 8, 256, "rank3", cols=256)
    assert sp.loads_per_operand == 1
    assert st.encode_args("f16", 8, 256, sp) == (
        "float16", 3, 64, 8, 4, 512, 128, 64, 8, 4, 1, 1, 1, 0, 3, 2, 0)


def test_encode_args_rank2():
    sp = st.split("f16", 8, 256)
    assert sp.loads_per_operand == 4
    assert st.encode_args("f16", 8, 256, sp) == (
        "float16", 2, 256, 8, 512, 64, 8, 1, 1, 0, 3, 2, 0)


# --------------------------------------------------------------- schedule

def test_schedule_trip_counts():
    """nvFuser PR #2833, Detailed Pseudo-Code: the prologue issues S - 1
    loads, the main loop runs N - (S - 1) times, the epilogue S - 1 times."""
    for S in (2, 3, 4):
        for N in (S - 1, S, 10, 37):
            assert st.trip_counts(N, S) == (S - 1, N - (S - 1), S - 1)
    assert st.trip_counts(5, 1) == (0, 5, 0)


def test_schedule_brute_force_invariants():
    for N, S in itertools.product(range(0, 41), range(1, 7)):
        ev = st.schedule(N, S)
        assert ev[:S] == [("init", s) for s in range(S)]
        assert ev[-S:] == [("inval", s) for s in range(S)]
        loads = [e for e in ev if e[0] == "load"]
        waits = [e for e in ev if e[0] == "wait"]
        assert [e[1] for e in loads] == list(range(N))
        assert [e[1] for e in waits] == list(range(N))
        pos = {e: i for i, e in enumerate(ev)}
        for k in range(N):
            ld, wt = ("load", k, k % S), ("wait", k, k % S, (k // S) & 1)
            assert pos[ld] < pos[wt] < pos[("body", k)]
            # WAR: tile k reuses stage k mod S only after tile k - S's body
            if k >= S:
                assert pos[("body", k - S)] < pos[ld]
        # at most S - 1 loads are outstanding beyond the tile being consumed
        issued = consumed = 0
        for e in ev:
            if e[0] == "load":
                issued += 1
            elif e[0] == "wait":
                assert issued - consumed <= S
                consumed += 1
            elif e[0] == "body":
                assert issued - consumed <= S - 1


def test_persistent_tiles_partition_the_grid():
    for T, G in itertools.product(range(0, 30), range(1, 9)):
        got = sorted(t for c in range(G) for t in st.cta_tiles(T, G, c))
        assert got == list(range(T))


def test_ldgsts_pending_allowed_brute_force():
    """Simulate one commit group per tile: after waiting until at most the
    allowed number are pending, tile i's group is complete."""
    for N, S in itertools.product(range(0, 25), range(2, 7)):
        for i in range(N):
            allowed = st.ldgsts_pending_allowed(i, N, S)
            committed_before = min(N, i + S - 1)
            assert committed_before >= i + 1
            assert committed_before - allowed == i + 1        # groups 0..i done, no more
            assert allowed == (S - 2 if i + S - 1 < N else N - 1 - i)


def test_tile_origin_row_major():
    assert st.tile_count(500, 4096, 32, 32) == 16 * 128
    assert st.tile_origin(0, 500, 4096, 32, 32) == (0, 0)
    assert st.tile_origin(129, 500, 4096, 32, 32) == (32, 32)
    assert st.tile_origin(16 * 128 - 1, 500, 4096, 32, 32) == (480, 4064)


@pytest.mark.parametrize("mode,period", [(32, 256), (64, 512), (128, 1024)])
def test_swizzle_invariants(mode, period):
    """The swizzle model moves whole 16-byte chunks, permutes the chunks of
    each period (its own inverse, so a bijection), keeps the first 128-byte
    line in place, and only ever moves a chunk within its own 128-byte line.
    (The pages print no swizzled address; these are the properties any
    reading of "128-byte swizzle" as a chunk XOR must have.)"""
    for base in (0, period, 5 * period):
        images = [st.swizzle(base + o, mode) for o in range(period)]
        assert sorted(images) == list(range(base, base + period))
        for o in range(period):
            x = base + o
            y = st.swizzle(x, mode)
            assert st.swizzle(y, mode) == x
            assert y % 16 == x % 16 and y // 128 == x // 128
            if o < 128:
                assert y == x
    # the 128-byte mode uses three line bits: lines 0..7 permute the chunks
    # of their line in eight different ways, and line 8 starts over
    perms = {tuple(st.swizzle(line * 128 + c * 16, 128) // 16 % 8 for c in range(8)) for line in range(8)}
    assert len(perms) == 8
    assert [st.swizzle(8 * 128 + c * 16, 128) for c in range(8)] == [8 * 128 + c * 16 for c in range(8)]


def test_swizzle_mode_none_is_row_major():
    assert all(st.swizzle(o, 0) == o for o in range(4096))
