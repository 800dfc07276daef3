"""The oracle's structure models, and the host planner, against the values
the pages print, kept as small fixtures under tests/golden/ (each with the
passage it comes from)."""

import json
import os

import pytest

from oracle import structure as st

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load("partition_examples.json")["cases"], ids=lambda c: c["cite"][:60])
def test_partition_examples(case):
    got = st.partition(case["elems"], case["threads"], case["elem_bytes"], run_bytes=case["run_bytes"],
                       align_bytes=case["align_bytes"], vec_bits=tuple(case["vec_bits"]))
    want = None if case["vec"] is None else (case["vec"], case["outer"])
    assert got == want, case["cite"]


def test_rank3_encode_tuple():
    g = _load("rank3_encode_tuple.json")
    rows, cols = g["tile"]
    sp = st.split("f16", rows, cols, mode="rank3", cols=cols)
    assert list(st.encode_args("f16", rows, cols, sp)) == g["encode_args"], g["cite"]


def test_rank3_encode_tuple_from_the_library():
    """The host planner's encode arguments for the same tile (tsx_plan_query,
    no GPU needed), in the page's order: reversed shape, strides, box."""
    tsx = pytest.importorskip("pipelined_elementwise_streaming_gb300")
    g = _load("rank3_encode_tuple.json")
    rows, cols = g["tile"]
    q = tsx.query("f16", rows, cols, (rows, cols), 1, "tma_rank3", "copy")
    r = q["rank"]
    args = ["float16", r, *q["global_dim"][:r], *q["global_stride_bytes"][:r - 1], *q["box_dim"][:r],
            *q["element_strides"][:r], q["interleave"], q["swizzle"], q["l2_promotion"], q["oob_fill"]]
    assert args == g["encode_args"]


@pytest.mark.parametrize("case", _load("loop_structure.json")["cases"], ids=lambda c: f"N{c['N']}S{c['S']}")
def test_loop_structure_trip_counts(case):
    assert st.trip_counts(case["N"], case["S"]) == (case["prologue"], case["main"], case["epilogue"])
    ev = st.schedule(case["N"], case["S"])
    assert sum(1 for e in ev if e[0] == "init") == case["S"] == sum(1 for e in ev if e[0] == "inval")


@pytest.mark.parametrize("case", _load("split_rules.json")["cases"], ids=lambda c: c["what"][:40])
def test_split_rules(case):
    sp = st.split(case["dtype"], *case["box"])
    assert sp.loads_per_operand == case["loads_per_operand"]
    assert sp.bytes_per_load == case["bytes_per_load"]
    assert max(sp.rows_per_load, sp.inner_elems) <= st.BOX_MAX
    for key, n_in in (("tx_bytes_n_in_1", 1), ("tx_bytes_n_in_3", 3)):
        if key in case:
            assert sp.tx_bytes(n_in) == case[key]
