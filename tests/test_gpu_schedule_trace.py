"""The device schedule of the TMA circular buffer against the oracle's model
of the loop structure of nvFuser PR #2833 ("Loop Structure", "Detailed
Pseudo-Code"): oracle.structure.schedule / trip_counts.

A plan with tracing enabled (tsx_debug_plan_enable_trace) runs a traced kernel that records, per
CTA, the load of each tile (prologue or main loop), the producer's reuse of
a released stage, the compute warps' wait and body, and the store warp's
store and release, numbered in the order they happened.  Per CTA the test
checks that
  * loads, waits and bodies come in the model's order, with the model's
    stage k mod S and phase parity (k / S) mod 2, and the prologue issues
    exactly the model's min(S - 1, N) tiles;
  * every tile is loaded, waited on, computed and stored once;
  * a tile is waited on and stored only after its load was issued, and
    stored only after it was computed;
  * tile k reuses stage k mod S only after the store of tile k - S released
    it (write-after-read), which also bounds the loads in flight at S.
Warp specialisation runs the roles concurrently, so only these orders are
fixed; the model's single interleaving is not required."""

import numpy as np
import pytest

import oracle
from oracle import structure as st
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu

LOAD, REUSE, WAIT, BODY, STORE, RELEASE = 1, 2, 3, 4, 5, 6


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _run(tsx, op, tiles, stages, variant="tma", tuning=None):
    """fp32 [8 * tiles, 32] with 8x32 boxes: one tile per row band, at most
    one CTA per SM.  Returns (trace [G, cap, 4], effective store lag, store
    warps)."""
    rows, cols = 8 * tiles, 32
    a = random_bits("f32", (rows, cols), tiles + stages)
    b = random_bits("f32", (rows, cols), tiles + stages + 1)
    with tsx.Plan("f32", rows, cols, box=(8, 32), stages=stages, variant=variant,
                  tuning=dict(tuning or {}, ctas_per_sm=1)) as plan:
        plan.enable_trace(256)
        da, db = to_dev(a, "f32"), to_dev(b, "f32")
        out = plan.ewise(op, da, db if op == "add" else None)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
        trace = plan.trace()
        info = plan.info(op)
        W = info["store_warps"]
        lag = min(info["store_lag"], (stages - 1) // W)
    want = oracle.ewise(op, "f32", a, b) if op == "add" else a
    compare(op, "f32", bits_of(out, "f32"), want, f"traced {op}")
    return trace, lag, W


def _check_cta(ev, N, S, lag, op, W=1):
    """One CTA's events against the model; W store warps take the CTA's
    tiles in turn (warp w: tiles w, w + W, ...), each releasing its tile j
    after storing its tile j + lag."""
    ev = ev[ev[:, 1] != 0]
    assert np.array_equal(ev[:, 0], np.arange(len(ev))), "sequence numbers are not dense"
    kind, k, a, b = ev[:, 1], ev[:, 2].astype(np.int64), ev[:, 3] & 0xFFFF, ev[:, 3] >> 16
    seq = {}
    for i, (kd, kk) in enumerate(zip(kind, k)):
        assert (kd, kk) not in seq, f"event {kd} of tile {kk} recorded twice"
        seq[(int(kd), int(kk))] = i

    sim = st.schedule(N, S)
    sim_loads = [(e[1], e[2]) for e in sim if e[0] == "load"]
    sim_waits = [(e[1], e[2], e[3]) for e in sim if e[0] == "wait"]
    sim_bodies = [e[1] for e in sim if e[0] == "body"]
    pro = st.trip_counts(N, S)[0]

    loads = [(int(x), int(y)) for x, y in zip(k[kind == LOAD], a[kind == LOAD])]
    assert loads == sim_loads
    assert list(b[kind == LOAD]) == [0] * pro + [1] * (N - pro), "prologue / main-loop split"
    stores = [(int(x), int(y)) for x, y in zip(k[kind == STORE], a[kind == STORE])]
    releases = [(int(x), int(y)) for x, y in zip(k[kind == RELEASE], a[kind == RELEASE])]
    assert sorted(stores) == [(i, i % S) for i in range(N)]
    want_released = []
    for w in range(W):
        mine = list(range(w, N, W))
        # each store warp stores its tiles in order and releases all but its last `lag`
        assert [x for x in stores if x[0] % W == w] == [(i, i % S) for i in mine]
        kept = mine[:max(0, len(mine) - lag)]
        assert [x for x in releases if x[0] % W == w] == [(i, i % S) for i in kept]
        want_released += kept
    assert sorted(x[0] for x in releases) == sorted(want_released)
    for i in want_released:
        assert seq[(STORE, i)] < seq[(RELEASE, i)], f"tile {i} released before its store"
    reuses = [(int(x), int(y), int(z)) for x, y, z in zip(k[kind == REUSE], a[kind == REUSE], b[kind == REUSE])]
    assert reuses == [(i, i % S, ((i // S) - 1) & 1) for i in range(S, N)]
    if op != "copy":
        waits = [(int(x), int(y), int(z)) for x, y, z in zip(k[kind == WAIT], a[kind == WAIT], b[kind == WAIT])]
        assert waits == sim_waits
        assert [int(x) for x in k[kind == BODY]] == sim_bodies

    for i in range(N):
        assert seq[(LOAD, i)] < seq[(STORE, i)]
        if op != "copy":
            assert seq[(LOAD, i)] < seq[(WAIT, i)] < seq[(BODY, i)] < seq[(STORE, i)]
        if i >= S:
            assert seq[(RELEASE, i - S)] < seq[(REUSE, i)] < seq[(LOAD, i)], f"stage of tile {i} reused early"


@pytest.mark.parametrize("op", ["add", "copy"])
@pytest.mark.parametrize("tiles,stages", [(1000, 1), (1000, 2), (1000, 3), (1000, 4),
                                          (456, 4), (100, 4), (160, 3)])
def test_device_schedule_matches_the_model(tsx, op, tiles, stages):
    trace, lag, W = _run(tsx, op, tiles, stages)
    G = trace.shape[0]
    assert G == min(tiles, G) and G <= tiles
    for c in range(G):
        N = len(st.cta_tiles(tiles, G, c))
        _check_cta(trace[c], N, stages, lag, op, W)


@pytest.mark.parametrize("op", ["add", "copy"])
@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("store_warps,store_lag", [(1, 0), (2, 0), (2, 1)])
def test_store_warps_follow_the_model(tsx, op, stages, store_warps, store_lag):
    """One or two store warps, each releasing its stage `lag` of its own
    tiles later (lag capped so that lag * W <= S - 1).  Copy, whose store
    waits on the loads' barriers (completed in any order), takes two store
    warps only when they divide the stage count."""
    tiles = 900
    trace, lag, W = _run(tsx, op, tiles, stages, tuning={"store_warps": store_warps, "store_lag": store_lag})
    want_w = min(store_warps, stages)
    if op == "copy" and stages % want_w:
        want_w = 1
    assert W == want_w and lag == min(store_lag, (stages - 1) // W)
    G = trace.shape[0]
    for c in range(G):
        _check_cta(trace[c], len(st.cta_tiles(tiles, G, c)), stages, lag, op, W)


def test_rank3_plan_traces_too(tsx):
    trace, lag, W = _run(tsx, "add", 700, 3, variant="tma_rank3")
    for c in range(trace.shape[0]):
        _check_cta(trace[c], len(st.cta_tiles(700, trace.shape[0], c)), 3, lag, "add", W)


def test_trace_is_refused_where_no_traced_kernel_exists(tsx):
    a = torch.zeros(64, 64, device="cuda")
    with tsx.Plan("f32", 64, 64, box=(8, 32), stages=2) as plan:
        plan.enable_trace(64)
        with pytest.raises(tsx.TsxError) as ei:
            plan.ewise("exp", a)
        assert ei.value.code == tsx.TSX_ERR_UNSUPPORTED
        # turning tracing off again gives the plain kernel back
        plan.enable_trace(0)
        plan.ewise("exp", a)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
    with tsx.Plan("f32", 64, 64, box=(8, 32), stages=2) as plan:
        plan.ewise("add", a, a)
        with pytest.raises(tsx.TsxError) as ei:
            plan.trace()
        assert ei.value.code == tsx.TSX_ERR_INVALID
