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
fixed; the model's single interleaving is not required.

Tiles are counted per CTA (its k-th tile).  In the static tile order CTA c
of G takes tiles c, c + G, ...; in the dynamic order (copy) its first P are
the same and the rest are claimed from a counter: there the test also
checks that the claimed tiles of all CTAs together are every tile once, in
increasing order within a CTA, and that a store warp hands back every stage
it holds once the tiles have run out."""

import numpy as np
import pytest

import oracle
from oracle import structure as st
from tests import _gpu
from tests._gpu import bits_of, compare, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu

LOAD, REUSE, WAIT, BODY, STORE, RELEASE, TILE = 1, 2, 3, 4, 5, 6, 7


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def _run(tsx, op, tiles, stages, variant="tma", tuning=None, cols=32):
    """fp32 [8 * tiles, cols] with 8 x cols boxes (one box per 32 columns):
    one tile per row band, at most one CTA per SM.  Returns (trace [G, cap,
    4], effective store lag, store warps, the dynamic order's static tiles
    per CTA, the tile order)."""
    rows = 8 * tiles
    a = random_bits("f32", (rows, cols), tiles + stages)
    b = random_bits("f32", (rows, cols), tiles + stages + 1)
    with tsx.Plan("f32", rows, cols, box=(8, cols), stages=stages, variant=variant,
                  tuning=dict({"ctas_per_sm": 1}, **(tuning or {}))) as plan:
        plan.enable_trace(256)
        da, db = to_dev(a, "f32"), to_dev(b, "f32")
        out = plan.ewise(op, da, db if op == "add" else None)
        torch.cuda.synchronize()
        assert plan.status() == tsx.TSX_OK
        trace = plan.trace()
        info = plan.info(op)
        W = info["store_warps"]
        if op == "copy" and stages % W:
            W = 1
        lag = min(info["store_lag"], (stages - 1) // W)
        # the dynamic order is the copy's (by default); other ops are static
        assert info["tile_order"] == ((tuning or {}).get("tile_order", 2) if op == "copy" else 1)
        share = info["dynamic_share"]
        order = info["tile_order"]
    want = oracle.ewise(op, "f32", a, b) if op == "add" else a
    compare(op, "f32", bits_of(out, "f32"), want, f"traced {op}")
    G = trace.shape[0]
    # the CTAs' static tiles in the dynamic order (the host's rule)
    P = max(max(1, stages - 1), (tiles // G) * (100 - share) // 100)
    return trace, lag, W, P, order


def _tiles_of(trace, c):
    """The tensor tiles CTA c took, by its k (dynamic order: TILE events)."""
    ev = trace[c][trace[c][:, 1] != 0]
    m = ev[:, 1] == TILE
    return ev[m][np.argsort(ev[m][:, 2]), 3].astype(np.int64)


def _check_dynamic(trace, tiles, P):
    """Dynamic order over all CTAs: each CTA's first P tiles are c, c + G,
    ...; later ones were claimed in increasing order; together every tile
    once.  Returns each CTA's tile count."""
    G = trace.shape[0]
    seen, counts = [], []
    for c in range(G):
        t = _tiles_of(trace, c)
        static = [x for x in (c + k * G for k in range(P)) if x < tiles]
        assert list(t[:len(static)]) == static, f"CTA {c}: static tiles {list(t[:P])}"
        claimed = t[len(static):]
        assert np.all(np.diff(claimed) > 0) and np.all(claimed >= P * G), f"CTA {c}: claims {claimed[:8]}"
        if len(static) < P:
            assert len(claimed) == 0
        seen.append(t)
        counts.append(len(t))
    seen = np.sort(np.concatenate(seen))
    assert np.array_equal(seen, np.arange(tiles)), "claimed tiles are not every tile once"
    return counts


def _check_cta(ev, N, S, lag, op, W=1, dynamic=False, split=False):
    """One CTA's events against the model; W store warps take the CTA's
    tiles in turn (warp w: tiles w, w + W, ...), each releasing its tile j
    after storing its tile j + lag (in the dynamic order also its last
    `lag` tiles once the tiles have run out).  With split stores the store of
    a tile's first half starts before its compute ends: the tile must then be
    computed before its stage is released."""
    ev = ev[ev[:, 1] != 0]
    assert np.array_equal(ev[:, 0], np.arange(len(ev))), "sequence numbers are not dense"
    kind, k, a, b = ev[:, 1], ev[:, 2].astype(np.int64), ev[:, 3] & 0xFFFF, ev[:, 3] >> 16
    seq = {}
    for i, (kd, kk) in enumerate(zip(kind, k)):
        assert (kd, kk) not in seq, f"event {kd} of tile {kk} recorded twice"
        seq[(int(kd), int(kk))] = i
    assert N == int(np.sum(kind == LOAD))
    if dynamic:
        assert [int(x) for x in k[kind == TILE]] == list(range(N))
    else:
        assert not np.any(kind == TILE)

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
        kept = mine if dynamic else mine[:max(0, len(mine) - lag)]
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
        if op != "copy" and not split:
            assert seq[(LOAD, i)] < seq[(WAIT, i)] < seq[(BODY, i)] < seq[(STORE, i)]
        if split:
            assert seq[(LOAD, i)] < seq[(WAIT, i)] < seq[(STORE, i)]
            if (RELEASE, i) in seq:
                assert seq[(BODY, i)] < seq[(RELEASE, i)]
        if i >= S:
            assert seq[(RELEASE, i - S)] < seq[(REUSE, i)] < seq[(LOAD, i)], f"stage of tile {i} reused early"


def _check_all(trace, tiles, stages, lag, op, W, order, P, split=False):
    G = trace.shape[0]
    assert G <= tiles
    if order == 2:
        counts = _check_dynamic(trace, tiles, P)
    else:
        counts = [len(st.cta_tiles(tiles, G, c)) for c in range(G)]
    for c in range(G):
        _check_cta(trace[c], counts[c], stages, lag, op, W, dynamic=order == 2, split=split)


ORDERS = [{"tile_order": 1}, {"tile_order": 2}, {"tile_order": 2, "dynamic_share": 100},
          {"tile_order": 2, "dynamic_share": 50}]


@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("op", ["add", "copy"])
@pytest.mark.parametrize("tiles,stages", [(1000, 1), (1000, 2), (1000, 3), (1000, 4),
                                          (456, 4), (100, 4), (160, 3), (152, 3), (153, 2)])
def test_device_schedule_matches_the_model(tsx, op, tiles, stages, order):
    trace, lag, W, P, got = _run(tsx, op, tiles, stages, tuning=order)
    _check_all(trace, tiles, stages, lag, op, W, got, P)


@pytest.mark.parametrize("order", ORDERS[:3])
@pytest.mark.parametrize("op", ["add", "copy"])
@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("store_warps,store_lag", [(1, 0), (2, 0), (2, 1), (1, 2)])
def test_store_warps_follow_the_model(tsx, op, stages, store_warps, store_lag, order):
    """One or two store warps, each releasing its stage `lag` of its own
    tiles later (lag capped so that lag * W <= S - 1).  Copy, whose store
    waits on the loads' barriers (completed in any order), takes two store
    warps only when they divide the stage count."""
    tiles = 900
    trace, lag, W, P, got = _run(tsx, op, tiles, stages,
                                 tuning=dict(order, store_warps=store_warps, store_lag=store_lag))
    want_w = min(store_warps, stages)
    if op == "copy" and stages % want_w:
        want_w = 1
    assert W == want_w and lag == min(store_lag, (stages - 1) // W)
    _check_all(trace, tiles, stages, lag, op, W, got, P)


@pytest.mark.parametrize("op", ["add", "copy"])
@pytest.mark.parametrize("order", ORDERS)
def test_rank3_plan_traces_too(tsx, order, op):
    trace, lag, W, P, got = _run(tsx, op, 700, 3, variant="tma_rank3", tuning=order)
    _check_all(trace, 700, 3, lag, op, W, got, P)


@pytest.mark.parametrize("share", [100, 10])
@pytest.mark.parametrize("ctas", [2, 0])
def test_dynamic_order_with_several_ctas_per_sm(tsx, ctas, share):
    """More CTAs than SMs claim from one counter: still every tile once."""
    trace, lag, W, P, got = _run(tsx, "copy", 3000, 2, tuning={"ctas_per_sm": ctas, "tile_order": 2,
                                                               "dynamic_share": share})
    assert got == 2
    _check_all(trace, 3000, 2, lag, "copy", W, 2, P)


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


@pytest.mark.parametrize("store_warps,store_lag", [(1, 0), (1, 1), (2, 0), (1, 2)])
@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_split_stores_follow_the_model(tsx, stages, store_warps, store_lag):
    """Two groups of boxes per tile (the first half stored while the second
    is computed): the schedule is the model's, the results the oracle's."""
    tiles = 900
    trace, lag, W, P, got = _run(tsx, "add", tiles, stages, cols=64,
                                 tuning={"store_split": 2, "store_warps": store_warps, "store_lag": store_lag})
    _check_all(trace, tiles, stages, lag, "add", W, got, P, split=True)
