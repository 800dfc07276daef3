// The TMA circular-buffer elementwise kernel.
//
// A persistent CTA c of G takes tiles c, c + G, c + 2G, ... (row-major tile
// order) and streams them through S stage buffers in shared memory; a long
// copy takes its first tiles that way and claims the rest from a counter
// (the dynamic tile order, below).  The warps of a CTA have three roles:
//
//   warp 0      the producer: lane 0 arrives once on the stage's `full`
//               mbarrier with expect_tx = the bytes of the stage's loads,
//               then every lane issues its share of the cp.async.bulk.tensor
//               loads (one box per lane; the pages issue them from one
//               thread); the TMA unit completes the phase when the bytes
//               have landed (TVM docs "copy_async -> tma", "Demonstration
//               program"; nvFuser PR #2833 "Add TMA support for circular
//               buffering pass", "Lowering Details").
//   warps 1..W  the store warps (W = 1 or 2; warp 1 + w takes the CTA's
//               tiles w, w + W, ...): each waits until its tile is computed,
//               each lane issues its share of the TMA stores from the stage,
//               and lane 0 hands the stage back to the producer (`empty`)
//               once every lane's stores have finished reading shared memory.
//   the rest    the compute warps: wait on `full` (parity (i / S) mod 2 for
//               their i-th tile), apply the op to 16-byte vectors (f *
//               threads + tid) of each operand's slot, write the result over
//               operand a's slot and arrive on `computed` (TVM docs
//               "elementwise -> smem", "Algorithm").  In the mixed variant
//               operand b is not staged: the compute warps read it from
//               global memory with plain vector loads at the positions of
//               the staged vectors, one tile ahead into registers (nvFuser
//               PR #2833, "Testing Setup", Pointwise: one tensor by TMA
//               circular buffering, the other by Set circular buffering).
//
// The producer follows the loop structure of the nvFuser page ("Loop
// Structure", "Detailed Pseudo-Code"): a pre-prologue that initialises the
// barriers, a prologue that issues the first S - 1 tiles, a main loop that
// issues tile i + S - 1 into stage (i + S - 1) mod S while the compute warps
// wait on tile i in stage i mod S, and a post-epilogue that invalidates the
// barriers; the consumers' loop over their tiles is the main loop plus the
// epilogue.  Stage reuse is ordered by the `empty` barrier: a store warp
// releases tile i's stage once the bulk stores up to tile i have read shared
// memory, which it checks `lag` of its own tiles later
// (cp.async.bulk.wait_group.read) so that a draining store does not hold up
// the next tile's stores; with two store warps the other warp stores the
// next tile meanwhile, so each can release its stage as soon as its own
// stores have read it.
//
// In the split instantiations (sqrt and exp with large tiles) the compute
// warps hand a tile over in two halves of its boxes, each with its own
// `computed` barrier, and the store warp stores the first half while the
// second is computed.
//
// Every mbarrier wait is bounded in time and also gives up when another
// thread has raised the CTA's abort flag.  A wait that runs out records
// TSX_ERR_TIMEOUT in the status word and raises the flag; every role then
// leaves its loop, the producer waits (again bounded) for the loads it still
// has in flight, the store warp for its stores, and the CTA exits.

#include "tsx_tma_common.cuh"

namespace tsx {
namespace {

using namespace dev;

// The store warp's TMA stores of one tile from the slot at shared address
// `slot`: each of the first `lanes` lanes stores the boxes numbered lane,
// lane + lanes, ... of the n_boxes of a full tile (`mine` is its first) and
// commits them as one bulk group of its own; with ACC a reduce-store that
// adds the tile into global memory.
template <bool ACC>
__device__ __forceinline__ void store_tile(const TmaMaps& maps, const TmaArgs& p, const TileCursor& tc,
                                           const BoxRef& mine, int n_boxes, int lanes, uint32_t slot)
{
    const int lane = static_cast<int>(threadIdx.x & 31);
    const TileBoxes b = boxes_at(p, tc.band, tc.ct);
    for (int L = lane; L < n_boxes; L += lanes) {
        const BoxRef x = L == lane ? mine : box_ref(maps, p, L, 3);
        if (!box_in(x, b))
            continue;
        const uint32_t src = slot + x.off;
        const int y = b.row0 + x.dy;
        if (p.rank3) {
            const int z = static_cast<int>(tc.ct * p.atoms);
            if constexpr (ACC)
                tma_reduce_add_3d(x.map, src, 0, y, z);
            else
                tma_store_3d(x.map, src, 0, y, z);
        } else {
            const int xc = (b.col0 >> p.promote_shift) + x.dx;
            if constexpr (ACC)
                tma_reduce_add_2d(x.map, src, xc, y);
            else
                tma_store_2d(x.map, src, xc, y);
        }
    }
    bulk_commit();
}

// The store warp's TMA stores of boxes [lo, hi) of one tile (box numbering
// as in store_tile), lanes lo + lane, lo + lane + lanes, ..., committed as
// one bulk group per lane.
template <bool ACC>
__device__ __forceinline__ void store_boxes(const TmaMaps& maps, const TmaArgs& p, const TileCursor& tc, int lo,
                                            int hi, int lanes, uint32_t slot)
{
    const int lane = static_cast<int>(threadIdx.x & 31);
    const TileBoxes b = boxes_at(p, tc.band, tc.ct);
    for (int L = lo + lane; L < hi; L += lanes) {
        const BoxRef x = box_ref(maps, p, L, 3);
        if (!box_in(x, b))
            continue;
        const uint32_t src = slot + x.off;
        const int y = b.row0 + x.dy;
        if (p.rank3) {
            const int z = static_cast<int>(tc.ct * p.atoms);
            if constexpr (ACC)
                tma_reduce_add_3d(x.map, src, 0, y, z);
            else
                tma_store_3d(x.map, src, 0, y, z);
        } else {
            const int xc = (b.col0 >> p.promote_shift) + x.dx;
            if constexpr (ACC)
                tma_reduce_add_2d(x.map, src, xc, y);
            else
                tma_store_2d(x.map, src, xc, y);
        }
    }
    bulk_commit();
}

// Operand b of the mixed variant is not staged by TMA.  The compute threads
// load it from global memory with plain 16-byte loads at the elements their
// staged vectors hold: the "Set" circular buffering of the nvFuser page's
// Pointwise test, kept in registers.  A thread's first kSetUnits units of a
// tile (tid, tid + threads, ...) are loaded one tile ahead, before the wait
// on the tile's stage, so the loads are in flight while the thread waits and
// computes; any further units load on use.  The planner gives the mixed
// variant enough threads that every unit is among the first kSetUnits.

// The producer of the mixed variant asks the TMA unit to bring b's boxes
// into L2 (tensor map slot 2 holds b's map) for the CTA's tile
// b_prefetch_ahead tiles beyond the one it loads, a few tiles before the
// compute threads read them into registers, so those plain loads mostly hit
// L2.  Measured on GB300, fp32 fma [128, 2^20] at 4 stages: 6547 GB/s
// without it, 6765 prefetching the loaded tile, 6932 two tiles beyond.
__device__ __forceinline__ void prefetch_b_tile(const TmaMaps& maps, const TmaArgs& p, const TileCursor& tc)
{
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int per_op = p.row_chunks * p.atoms;
    for (int L = lane; L < per_op; L += 32) {
        const TileBoxes b = boxes_at(p, tc.band, tc.ct);
        const int r = L / p.atoms, a = L - r * p.atoms;
        if (r < b.chunks && a < b.atoms)
            tma_prefetch_l2_2d(&maps.m[2], b.col0 + a * p.inner_elems, b.row0 + r * p.rows_per_load);
    }
}

// Where unit u of a staged slot sits in its tile: every tile of a plan is
// staged with the same layout, so the unit holds the same (row, column) of
// every tile.  The box, the swizzle inverse and the divisions are worked out
// once per thread, not per tile.  Padding after a box has row -1.
struct UnitPos {
    int row, col;
};

template <int DT>
__device__ __forceinline__ UnitPos unit_pos(const TmaArgs& p, uint32_t u)
{
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
    const uint32_t inner_bytes = static_cast<uint32_t>(p.inner_elems) * ES;
    const uint32_t off = u * 16;
    const uint32_t load = off / p.load_smem_bytes;
    const uint32_t within = off - load * p.load_smem_bytes;
    UnitPos q{-1, 0};
    if (u < p.vec16_per_slot && within < p.box_bytes) {
        const uint32_t lo = unswizzle(within, p.swizzle_mask);
        q.row = static_cast<int>((load / p.atoms) * p.rows_per_load + lo / inner_bytes);
        q.col = static_cast<int>((load % p.atoms) * p.inner_elems + (lo % inner_bytes) / ES);
    }
    return q;
}

// b at the unit at position q of the tile with boxes tb (zero outside the
// tensor and in the padding after a box).  Loaded through L2 only: b may be
// the output, whose other tiles TMA stores overwrite meanwhile.
template <int DT>
__device__ __forceinline__ uint4 load_b_at(const TmaArgs& p, const TileBoxes& tb, const UnitPos& q)
{
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
    uint4 vb = make_uint4(0, 0, 0, 0);
    const int64_t row = static_cast<int64_t>(tb.row0) + q.row;
    const int64_t col = static_cast<int64_t>(tb.col0) + q.col;
    if (q.row >= 0 && row < p.rows && col < p.cols)
        vb = __ldcg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.set_operand) + (row * p.pitch + col) * ES));
    return vb;
}

template <int DT>
__device__ __forceinline__ uint4 load_b_unit(const TmaArgs& p, const TileBoxes& tb, uint32_t u)
{
    return load_b_at<DT>(p, tb, unit_pos<DT>(p, u));
}

template <int DT>
__device__ __forceinline__ void load_b_ahead(const TmaArgs& p, const TileBoxes& tb, const UnitPos (&pos)[kSetUnits],
                                             uint4 (&v)[kSetUnits])
{
#pragma unroll
    for (int k = 0; k < kSetUnits; ++k)
        v[k] = load_b_at<DT>(p, tb, pos[k]);
}

// The op on one staged tile of the mixed variant: a (and c) from the slots,
// b from the registers loaded ahead (bv) or, past those, from global memory.
template <int DT, int OP>
__device__ __forceinline__ void compute_tile_mixed(const TmaArgs& p, uint4* A, const uint4* C, const TileBoxes& tb,
                                                   uint32_t tid, uint32_t threads, const uint4 (&bv)[kSetUnits])
{
#pragma unroll
    for (int k = 0; k < kSetUnits; ++k) {
        const uint32_t u = tid + k * threads;
        if (u < p.vec16_per_slot) {
            const uint4 va = A[u];
            const uint4 vc = op_arity(OP) > 2 ? C[u] : va;
            A[u] = op_vec16<DT, OP>(va, bv[k], vc);
        }
    }
    for (uint32_t u = tid + kSetUnits * threads; u < p.vec16_per_slot; u += threads) {
        const uint4 vb = load_b_unit<DT>(p, tb, u);
        const uint4 va = A[u];
        const uint4 vc = op_arity(OP) > 2 ? C[u] : va;
        A[u] = op_vec16<DT, OP>(va, vb, vc);
    }
}

// Test hook of the traced instantiations: record one event in the CTA's
// ring, numbered by a shared-memory counter.  A thread records an event
// before the barrier arrival that lets other roles act on it, so the
// numbering respects the order the barriers impose.
template <bool TRACE>
__device__ __forceinline__ void trace_event(const TmaArgs& p, uint32_t* counter, int kind, int64_t k, uint32_t a,
                                            uint32_t b)
{
    if constexpr (TRACE) {
        const uint32_t i = atomicAdd(counter, 1u);
        if (i < static_cast<uint32_t>(p.trace_cap))
            reinterpret_cast<uint4*>(p.trace)[static_cast<size_t>(blockIdx.x) * p.trace_cap + i] =
                make_uint4(i, static_cast<uint32_t>(kind), static_cast<uint32_t>(k), a | (b << 16));
    }
}

// Registers: at most 56 a thread (96 in the mixed variant, whose compute
// threads hold b a tile ahead).  A warp's registers are allocated in blocks
// of 256, so at 58 a warp takes 2048 instead of 1792 and one CTA of 128
// threads per SM fewer fits: on GB300 such a build ran fp32 sqrt 7 % slower.
template <int DT, int OP, bool MIXED, bool ACC, bool TRACE = false, bool SPLIT = false>
__global__ void __maxnreg__(MIXED ? kMixedMaxRegs : kMaxRegs)
    tma_ewise(const __grid_constant__ TmaMaps maps, const TmaArgs p)
{
    constexpr int NIN = op_arity(OP);
    // operands in the stage: all of them, or all but b in the mixed variant
    constexpr int NT = MIXED ? tma_operands(TSX_TMA_MIXED, OP) : NIN;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1);
    uint8_t* const smem = smem_raw + (base - raw);
    const int S = p.stages;
    const uint32_t full = base + static_cast<uint32_t>(S) * p.stage_bytes;   // S barriers
    // two per stage (computed + 16 s + 8 g): group g of the stage's boxes computed
    const uint32_t computed = full + 8u * S;
    const uint32_t empty = computed + 16u * S;
    // groups of boxes the compute warps hand to the store warps one by one:
    // two in the split instantiations (ops with a compute step)
    constexpr int CG = SPLIT && !MIXED && OP != TSX_COPY ? 2 : 1;
    // dynamic tile order: the tile each stage holds (-1: no more tiles)
    volatile int64_t* tile_of = reinterpret_cast<volatile int64_t*>(smem + (empty + 8u * S - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + (empty + 16u * S - base));
    uint32_t* trace_counter = reinterpret_cast<uint32_t*>(smem + (empty + 16u * S - base) + 4);

    const int warp = threadIdx.x / 32;
    const int role_warps = tma_role_warps(p.store_warps);
    const int compute_warps = blockDim.x / 32 - role_warps;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int64_t N = cta < p.tiles ? (p.tiles - 1 - cta) / G + 1 : 0;
    const bool elected = warp < 2 && elect_one();   // one lane of warp 0 and of warp 1
    // Dynamic tile order (copy only): the CTA's first P tiles are c, c + G,
    // ..., c + (P - 1) G as in the static order (P >= 1, set by the host);
    // every later tile is claimed from the launch's counter (tiles P G,
    // P G + 1, ... in claim order), so CTAs that stream faster take more of
    // the last tiles and all finish together.  The producer hands each
    // claimed tile's index to the store warps through shared memory and
    // ends the CTA's stream with one "no more tiles" stage per store warp.
    // In a static-order launch the CTAs of a copy finished up to 40 % apart
    // (GB300); ops with a compute step measured slower with the dynamic
    // order, and slower still with its code merely compiled in, so their
    // instantiations are built without it.
    constexpr bool kDynamic = OP == TSX_COPY && !MIXED && !ACC;
    const bool dyn = kDynamic && p.tile_counter != nullptr;
    const int64_t P = p.static_tiles > 0 ? p.static_tiles : 1;

    // Pre-prologue: the barriers of every stage; descriptor prefetch.
    if (warp == 0 && elected) {
        for (int j = 0; j < NT; ++j)
            prefetch_tensormap(&maps.m[j]);
        for (int s = 0; s < S; ++s) {
            mbar_init(full + 8u * s, 1);
            for (int g = 0; g < CG; ++g)
                mbar_init(computed + 16u * s + 8u * g, static_cast<uint32_t>(compute_warps));
            mbar_init(empty + 8u * s, 1);
        }
        *abort_flag = 0;
        *trace_counter = 0;
        fence_proxy_async_smem();
    }
    if (warp == 1 && elected)
        prefetch_tensormap(&maps.m[3]);
    __syncthreads();

    const int lane = static_cast<int>(threadIdx.x & 31);
    if (warp == 0) {
        // ---------------------------------------------------- producer
        const int n_loads = NT * (p.rank3 ? p.row_chunks : p.row_chunks * p.atoms);
        const BoxRef mine = box_ref(maps, p, lane < n_loads ? lane : 0, 0);
        TileCursor tc(p, cta, G);
        // mixed variant: the tile whose b the producer prefetches into L2
        TileCursor pf(p, cta + static_cast<int64_t>(MIXED ? p.b_prefetch_ahead : 0) * G, G);
        StageCursor st;
        int64_t issued = 0;
        if (!dyn) {
            const int64_t pro = N < S - 1 ? N : S - 1;
            // Prologue: the first S - 1 tiles, into stages that start empty.
            for (; issued < pro; ++issued) {
                if (lane == 0)
                    trace_event<TRACE>(p, trace_counter, kTraceLoad, issued, st.s, 0);
                issue_tile_lanes<NT>(maps, p, tc, mine, n_loads, base + st.s * p.stage_bytes, full + 8u * st.s);
                if constexpr (MIXED && NIN >= 2) {
                    if (pf.tile(p) < p.tiles)
                        prefetch_b_tile(maps, p, pf);
                    pf.next(p);
                }
                tc.next(p);
                st.next(S);
            }
            // Main loop: tile k = i + S - 1 into stage k mod S, once the
            // store warp has released that stage's previous tile (k - S).
            for (; issued < N; ++issued) {
                if (issued >= S && !role_wait(empty + 8u * st.s, st.phase ^ 1u, p, abort_flag, p.lane0_wait != 0))
                    break;
                if (lane == 0) {
                    if (issued >= S)
                        trace_event<TRACE>(p, trace_counter, kTraceReuse, issued, st.s, st.phase ^ 1u);
                    trace_event<TRACE>(p, trace_counter, kTraceLoad, issued, st.s, 1);
                }
                issue_tile_lanes<NT>(maps, p, tc, mine, n_loads, base + st.s * p.stage_bytes, full + 8u * st.s);
                if constexpr (MIXED && NIN >= 2) {
                    if (pf.tile(p) < p.tiles)
                        prefetch_b_tile(maps, p, pf);
                    pf.next(p);
                }
                tc.next(p);
                st.next(S);
            }
        } else {
            // The same prologue and main loop over the CTA's k-th tile, k =
            // 0, 1, ... until the tiles run out.  The first P tiles follow
            // the static cursor; every role knows them without being told.
            // Lane 0 claims the tile of k + 1 as soon as it knows the tile
            // of k, so the atomic's round trip overlaps the wait for a free
            // stage, and publishes each claimed tile in the stage's slot.
            // one "no more tiles" stage per store warp that takes tiles
            const int W = OP == TSX_COPY && S % p.store_warps != 0 ? 1 : p.store_warps;
            const int64_t static_end = P * G;
            int64_t claim = p.tiles;   // lane 0: the claimed tile of the next k (>= tiles: none)
            int ended = 0;             // "no more tiles" stages issued
            for (;; ++issued) {
                const bool claimed = issued >= P;
                const int64_t t = claimed ? __shfl_sync(0xffffffffu, static_cast<long long>(claim), 0)
                                          : cta + issued * G;
                if (lane == 0 && issued + 1 >= P && t < p.tiles)
                    claim = static_end + static_cast<int64_t>(atomicAdd(p.tile_counter, 1ull));
                if (issued >= S && !role_wait(empty + 8u * st.s, st.phase ^ 1u, p, abort_flag, p.lane0_wait != 0))
                    break;
                if (t < p.tiles) {
                    if (lane == 0) {
                        if (issued >= S)
                            trace_event<TRACE>(p, trace_counter, kTraceReuse, issued, st.s, st.phase ^ 1u);
                        trace_event<TRACE>(p, trace_counter, kTraceTile, issued, static_cast<uint32_t>(t) & 0xffffu,
                                           static_cast<uint32_t>(t) >> 16);
                        trace_event<TRACE>(p, trace_counter, kTraceLoad, issued, st.s, issued < S - 1 ? 0 : 1);
                        if (claimed)
                            tile_of[st.s] = t;   // published by the arrival on `full`
                    }
                    if (claimed)
                        tc.seek(p, t);
                    issue_tile_lanes<NT>(maps, p, tc, mine, n_loads, base + st.s * p.stage_bytes,
                                         full + 8u * st.s);
                    if (!claimed)
                        tc.next(p);
                } else {
                    if (lane == 0) {
                        tile_of[st.s] = -1;
                        mbar_arrive(full + 8u * st.s);
                    }
                    __syncwarp();
                    if (++ended == W) {
                        ++issued;
                        break;
                    }
                }
                st.next(S);
            }
        }
        if (*abort_flag && lane == 0) {
            // let the loads still in flight land before shared memory goes away
            const int64_t first = issued > S ? issued - S : 0;
            for (int64_t k = first; k < issued; ++k)
                (void)mbar_wait(full + 8u * (k % S), static_cast<uint32_t>((k / S) & 1), p.timeout_ns);
        }
    } else if (warp < role_warps) {
        // ------------------------------------------------ store warps
        // A store warp's parity wait on a stage is exact only once the
        // stage's previous phase has completed.  The computed barriers
        // complete in tile order; copy waits on the full barriers, which the
        // loads complete in any order, so there the stage's previous tile
        // must be this warp's own: W must divide S (the planner ensures it;
        // a second store warp that would break it stays idle).
        const int W = OP == TSX_COPY && S % p.store_warps != 0 ? 1 : p.store_warps;
        const int sw = warp - 1;   // this warp takes the CTA's tiles sw, sw + W, ...
        const int n_boxes = p.rank3 ? p.row_chunks : p.row_chunks * p.atoms;
        // lanes issuing stores: one per box, except that reduce-stores go out
        // from lane 0 alone (measured faster on GB300)
        const int lanes = ACC ? 1 : n_boxes < 32 ? n_boxes : 32;
        const BoxRef mine = box_ref(maps, p, lane < n_boxes ? lane : 0, 3);
        // the lag is counted in this warp's tiles: tile i releases tile
        // i - lag W, which must come before the producer needs its stage
        // again for tile i - lag W + S, so lag W <= S - 1
        const int most = (S - 1) / W;
        const int lag = p.store_lag < most ? p.store_lag : most;
        TileCursor tc(p, cta + sw * G, W * G);
        StageCursor st = StageCursor::at(sw, S), released = st;   // tile i and tile i - lag W
        int64_t stored = 0;   // tiles this warp has stored
        int64_t i = sw;
        for (; sw < W && (dyn || i < N); i += W, ++stored) {
            // copy has no compute step: the loaded tile goes straight back
            const uint32_t ready = OP == TSX_COPY ? full + 8u * st.s : computed + 16u * st.s;
            if (!role_wait(ready, st.phase, p, abort_flag, p.lane0_wait != 0))
                break;
            if (dyn) {
                if (i < P) {
                    // a static tile: past the last band means no more tiles
                    if (tc.band >= p.tiles_r)
                        break;
                } else {
                    // a claimed tile: lane 0 has seen the barrier complete
                    int64_t t = 0;
                    if (lane == 0)
                        t = tile_of[st.s];
                    t = __shfl_sync(0xffffffffu, static_cast<long long>(t), 0);
                    if (t < 0)
                        break;
                    tc.seek(p, t);
                }
            }
            if (lane == 0)
                trace_event<TRACE>(p, trace_counter, kTraceStore, i, st.s, st.phase);
            // release tile i - lag W once every lane's stores of it have read
            // shared memory (lanes without boxes keep out of the bulk groups)
            if constexpr (CG == 1) {
                if (lane < lanes) {
                    store_tile<ACC>(maps, p, tc, mine, n_boxes, lanes, base + st.s * p.stage_bytes);
                    bulk_wait_read(lag);
                }
            } else {
                // the first half of the boxes goes out while the compute warps
                // finish the second
                const int half = n_boxes / 2;
                const int lanes_g = ACC ? 1 : half < 32 ? half : 32;
                if (lane < lanes_g)
                    store_boxes<ACC>(maps, p, tc, 0, half, lanes_g, base + st.s * p.stage_bytes);
                if (!role_wait(computed + 16u * st.s + 8u, st.phase, p, abort_flag, p.lane0_wait != 0))
                    break;
                if (lane < lanes_g) {
                    store_boxes<ACC>(maps, p, tc, half, n_boxes, lanes_g, base + st.s * p.stage_bytes);
                    bulk_wait_read(2 * lag);
                }
            }
            __syncwarp();
            if (stored >= lag) {
                if (lane == 0) {
                    trace_event<TRACE>(p, trace_counter, kTraceRelease, i - int64_t(lag) * W, released.s, 0);
                    mbar_arrive(empty + 8u * released.s);
                }
                released.advance(W, S);
            }
            tc.next(p);   // the static order (a claimed tile seeks its own)
            st.advance(W, S);
        }
        if (dyn && !*abort_flag && sw < W) {
            // No more tiles: hand back the stages still held for the lag, so
            // that the producer can end the other store warp's stream too.
            if (lane < lanes)
                bulk_wait_read(0);
            __syncwarp();
            for (int64_t r = stored > lag ? stored - lag : 0; r < stored; ++r) {
                if (lane == 0) {
                    trace_event<TRACE>(p, trace_counter, kTraceRelease, sw + r * W, released.s, 0);
                    mbar_arrive(empty + 8u * released.s);
                }
                released.advance(W, S);
            }
        }
        if (lane < lanes)
            bulk_wait_all();
    } else if (OP != TSX_COPY) {
        // ---------------------------------------------- compute warps
        const uint32_t tid = threadIdx.x - 32u * role_warps;
        const uint32_t threads = blockDim.x - 32u * role_warps;
        StageCursor st;
        // mixed variant: b of the next tile, loaded ahead into registers
        constexpr bool kSet = MIXED && NIN >= 2;
        uint4 b_next[kSetUnits];
        UnitPos b_pos[kSetUnits];
        TileCursor tc(p, cta, G);
        if constexpr (kSet) {
#pragma unroll
            for (int k = 0; k < kSetUnits; ++k)
                b_pos[k] = unit_pos<DT>(p, tid + k * threads);
            if (N > 0)
                load_b_ahead<DT>(p, boxes_at(p, tc.band, tc.ct), b_pos, b_next);
        }
        for (int64_t i = 0; i < N; ++i) {
            uint4 b_cur[kSetUnits];
            TileBoxes tb;
            if constexpr (kSet) {
#pragma unroll
                for (int k = 0; k < kSetUnits; ++k)
                    b_cur[k] = b_next[k];
                tb = boxes_at(p, tc.band, tc.ct);
                tc.next(p);
                if (i + 1 < N)
                    load_b_ahead<DT>(p, boxes_at(p, tc.band, tc.ct), b_pos, b_next);
            }
            if (!wait_or_abort(full + 8u * st.s, st.phase, p, abort_flag))
                break;
            if (tid == 0)
                trace_event<TRACE>(p, trace_counter, kTraceWait, i, st.s, st.phase);
            uint4* A = reinterpret_cast<uint4*>(smem + static_cast<size_t>(st.s) * p.stage_bytes);
            if constexpr (kSet) {
                compute_tile_mixed<DT, OP>(p, A, A + p.slot_bytes / 16, tb, tid, threads, b_cur);
            } else {
                const uint4* B = A + p.slot_bytes / 16;
                const uint4* C = A + 2 * (p.slot_bytes / 16);
                const uint32_t n = p.vec16_per_slot;
                uint32_t u = tid;
                if constexpr (CG == 2) {
                    // the units of the first half of the boxes, handed to the
                    // store warp before those of the second
                    for (; u < n / 2; u += threads) {
                        const uint4 va = A[u];
                        const uint4 vb = NIN > 1 ? B[u] : va;
                        const uint4 vc = NIN > 2 ? C[u] : va;
                        A[u] = op_vec16<DT, OP>(va, vb, vc);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if ((threadIdx.x & 31) == 0)
                        mbar_arrive(computed + 16u * st.s);
                }
                for (; u < n; u += threads) {
                    const uint4 va = A[u];
                    const uint4 vb = NIN > 1 ? B[u] : va;
                    const uint4 vc = NIN > 2 ? C[u] : va;
                    A[u] = op_vec16<DT, OP>(va, vb, vc);
                }
            }
            // this thread's generic-proxy writes become visible to the TMA store
            fence_proxy_async_smem();
            if (tid == 0)
                trace_event<TRACE>(p, trace_counter, kTraceBody, i, st.s, 0);
            __syncwarp();
            if ((threadIdx.x & 31) == 0)
                mbar_arrive(computed + 16u * st.s + 8u * (CG - 1));
            st.next(S);
        }
    }

    // Post-epilogue.
    __syncthreads();
    if (warp == 0 && elected) {
        for (int s = 0; s < S; ++s) {
            mbar_inval(full + 8u * s);
            for (int g = 0; g < CG; ++g)
                mbar_inval(computed + 16u * s + 8u * g);
            mbar_inval(empty + 8u * s);
        }
    }
    if (dyn && threadIdx.x == 0) {
        // the launch's last CTA to finish zeroes the counter for the next
        // launch on the stream (every CTA has made its last claim by now)
        __threadfence();
        if (atomicAdd(p.tile_counter + 1, 1ull) == static_cast<unsigned long long>(G) - 1) {
            atomicExch(p.tile_counter, 0ull);
            atomicExch(p.tile_counter + 1, 0ull);
        }
    }
}

#define TSX_ROW(DT, M, A) \
    {(const void*)tma_ewise<DT, 0, M, A>, (const void*)tma_ewise<DT, 1, M, A>, (const void*)tma_ewise<DT, 2, M, A>, \
     (const void*)tma_ewise<DT, 3, M, A>, (const void*)tma_ewise<DT, 4, M, A>, (const void*)tma_ewise<DT, 5, M, A>}
#define TSX_KIND(M, A) {TSX_ROW(TSX_F16, M, A), TSX_ROW(TSX_BF16, M, A), TSX_ROW(TSX_F32, M, A)}
// the split instantiations (copy has no compute step to split: its plain one)
#define TSX_SPLIT_ROW(DT) \
    {(const void*)tma_ewise<DT, 0, false, false>, (const void*)tma_ewise<DT, 1, false, false, false, true>, \
     (const void*)tma_ewise<DT, 2, false, false, false, true>, (const void*)tma_ewise<DT, 3, false, false, false, true>, \
     (const void*)tma_ewise<DT, 4, false, false, false, true>, (const void*)tma_ewise<DT, 5, false, false, false, true>}
// indexed by TmaKind: plain, mixed, accumulate, split
const void* const kKernels[4][3][6] = {TSX_KIND(false, false), TSX_KIND(true, false), TSX_KIND(false, true),
                                       {TSX_SPLIT_ROW(TSX_F16), TSX_SPLIT_ROW(TSX_BF16), TSX_SPLIT_ROW(TSX_F32)}};
#undef TSX_SPLIT_ROW
#undef TSX_KIND
#undef TSX_ROW

}  // namespace

// the traced instantiations (test hook)
const void* traced_kernel(int dtype, int op, bool split)
{
    if (dtype != TSX_F32)
        return nullptr;
    if (op == TSX_COPY && !split)
        return (const void*)tma_ewise<TSX_F32, TSX_COPY, false, false, true>;
    if (op == TSX_ADD)
        return split ? (const void*)tma_ewise<TSX_F32, TSX_ADD, false, false, true, true>
                     : (const void*)tma_ewise<TSX_F32, TSX_ADD, false, false, true>;
    return nullptr;
}

const void* tma_kernel(int dtype, int op, int kind)
{
    if (kind == kTmaTraced || kind == kTmaTracedSplit)
        return traced_kernel(dtype, op, kind == kTmaTracedSplit);
    return kKernels[kind][dtype][op];
}

cudaError_t launch_tma(int dtype, int op, int kind, int grid, int threads, size_t smem, cudaStream_t stream,
                       const CUtensorMap* maps, const TmaArgs& args)
{
    TmaMaps m;
    for (int j = 0; j < 4; ++j)
        m.m[j] = maps[j];
    TmaArgs a = args;
    void* params[] = {&m, &a};
    return cudaLaunchKernel(tma_kernel(dtype, op, kind), dim3(grid), dim3(threads), params, smem, stream);
}

}  // namespace tsx
