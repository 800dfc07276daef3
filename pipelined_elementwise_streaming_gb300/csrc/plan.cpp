// Host planner of libtsx: argument validation, the TMA box split, the
// tensor-map encode arguments, the [outer, threads, vec] partition and the
// shared-memory budget.  Pure integer arithmetic: no CUDA call happens here,
// so tsx_plan_query works on a machine without a GPU.

#include <cstdio>
#include <cstring>
#include <string>

#include "plan.h"

namespace tsx {

namespace {

bool fail(std::string* why, const char* fmt, long long a = 0, long long b = 0)
{
    if (why) {
        char buf[256];
        std::snprintf(buf, sizeof buf, fmt, a, b);
        *why = buf;
    }
    return false;
}

uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

}  // namespace

// Stage bytes per SM that rings of small sqrt / exp stages, and of add / mul
// stages on long streams, aim at (make_op_geometry).
constexpr int64_t kSmallRingPerSm = 144 * 1024;
constexpr int64_t kLongStreamTiles = 32768;
// Staged bytes per SM that the mixed variant's add and mul aim at.
constexpr int64_t kMixedRingPerSm = 96 * 1024;
// Two-stage rings on streams of at least this many tiles take the targets
// of two_stage_ring_per_sm.
constexpr int64_t kTwoStageStreamTiles = 8192;

int default_threads(const Geometry& g, int op, size_t smem_bytes, uint32_t units, int store_warps)
{
    (void)op;
    // Threads of the elementwise stage.  TMA paths: about 256 compute
    // threads per SM in all, shared by the CTAs that fit in its shared
    // memory, between 2 and 8 compute warps per CTA (beside the producer
    // and store warps); the mixed variant, whose compute threads also load
    // b one tile ahead for at most kSetUnits of the slot's `units` 16-byte
    // vectors each, aims at about 512 per SM, rounded to the nearest warp,
    // and at least enough threads to cover the slot that way.  Rules of
    // make_op_geometry replace these shares where no knob is given.
    // The cp.async / synchronous ablations give each thread about four
    // 16-byte units of the slot, between 128 threads (the TVM ldgsts
    // demonstration program's count, which its 128x32 fp16 tile gets) and
    // 512.  A forced count (tsx_tuning.threads) wins.
    const int variant = g.variant;
    const bool tma = is_tma_variant(variant);
    if (g.knobs.threads > 0)
        return g.knobs.threads;
    int fallback = int((units / 4 + 31) / 32 * 32);
    fallback = fallback < 128 ? 128 : fallback > 512 ? 512 : fallback;
    if (tma) {
        const bool mixed = variant == TSX_TMA_MIXED;
        const size_t per_cta = smem_bytes + kSmemPerCtaReserved;
        const int ctas = per_cta ? int(kSmemPerSm / per_cta) : 1;
        const int share = (mixed ? 512 : 256) / (ctas < 1 ? 1 : ctas);
        const int cap = mixed ? 512 : 256;
        const int warps = mixed ? (share + 16) / 32 : share / 32;
        fallback = share < 64 ? 64 : share > cap ? cap : warps * 32;
        if (mixed) {
            const int cover = int((units + kSetUnits - 1) / kSetUnits + 31) / 32 * 32;
            const int most = kMixedMaxThreads - 32 * tma_role_warps(store_warps);
            fallback = fallback > cover ? fallback : cover < most ? cover : most;
        }
    }
    return fallback;
}

// One-operand compute ops (their compute warps do more per byte than copy
// and reach a stage from one operand only).
static bool one_operand_compute(int op) { return op == TSX_SQRT || op == TSX_EXP; }

// Groups of a tile's boxes that the compute warps hand to the store warps
// one by one (TMA variants).  Two need a compute step, an even box count and
// every operand staged; measured on GB300, the one-operand sqrt and exp gain
// 1-4 % with tiles of 16 KB or more, while ops with two or three operands,
// and small tiles, lose.
static int compute_groups_of(const Geometry& g, int op)
{
    const int boxes = g.variant == TSX_TMA_RANK3 ? g.row_chunks : g.row_chunks * g.atoms;
    const bool can_split = op != TSX_COPY && boxes % 2 == 0 && !(g.variant == TSX_TMA_MIXED && op_arity(op) >= 2);
    const bool split_pays = one_operand_compute(op) && g.slot_bytes >= 16384;
    const bool split = g.knobs.store_split == 2 || (g.knobs.store_split == 0 && split_pays);
    return can_split && split ? 2 : 1;
}

// Stage bytes per SM that a two-stage ring aims at: copy, add and mul 96 KB,
// the one-operand sqrt and exp 128 KB, fma 144 KB (make_op_geometry).
static int64_t two_stage_ring_per_sm(int op)
{
    if (op == TSX_FMA)
        return 144 * 1024;
    return one_operand_compute(op) ? 128 * 1024 : 96 * 1024;
}

int mixed_prefetch_ahead(const Geometry& g, int ctas_per_sm)
{
    // The producer runs S - 1 tiles ahead of the compute threads, which read
    // b one tile ahead: prefetching the tile it loads gives b S - 2 tiles of
    // lead in L2.  The best lead keeps about 40 KB of prefetched b per SM:
    // T = max(1, round(40 KB / (b's tile bytes x CTAs per SM))) tiles, so
    // the producer prefetches T - (S - 2) tiles beyond its load (never
    // behind).  Measured on GB300, this picks the best or a near-best lead
    // in every case swept: fp32 fma [128, 2^20] 2..6 stages (4 stages:
    // 6749 GB/s with no extra lead, 6940 with the rule's one), bf16 mul
    // [16384, 16384] 2 and 3 stages, bf16 add with 64x128 tiles 2..4 stages.
    if (g.knobs.b_prefetch >= 0)
        return g.knobs.b_prefetch;
    const int64_t per_sm = int64_t(g.slot_bytes) * (ctas_per_sm < 1 ? 1 : ctas_per_sm);
    int64_t lead = (2 * 40960 + per_sm) / (2 * per_sm);   // rounded
    lead = lead < 1 ? 1 : lead;
    const int64_t ahead = lead - (g.stages - 2);
    return ahead < 0 ? 0 : ahead > 8 ? 8 : int(ahead);
}

StoreSchedule store_schedule(const Geometry& g, int op, uint32_t stage_bytes)
{
    // How a stage comes back to the producer.  A store warp stores tile i
    // and releases the stage of its tile i - lag once that tile's stores
    // have read shared memory; with two store warps taking tiles in turn, a
    // warp can wait for its own store (lag 0) while the other stores the
    // next tile.  Measured on GB300 (all settings give identical results):
    //  - 2 stages: two store warps, lag 0: with one warp the ring holds a
    //    stage back for a whole tile (bf16 exp [16384, 16384] 4298 -> 5893
    //    GB/s, fp32 fma [128, 2^20] 6690 -> 7135).  Except where sqrt or
    //    exp stores tiles of 32 KB or more in two groups: there one warp at
    //    lag 0 streams faster (bf16 exp [16384, 16384] in 128x128 tiles 6261
    //    -> 6459, bf16 sqrt 6396 -> 6462; with 16 KB tiles it was mixed,
    //    bf16 exp in 64x128 tiles -5.6 %, fp32 exp and sqrt in 16x256 tiles
    //    +3.4 and +4.6 %);
    //  - 3 to 5 stages: one store warp, lag 1 (bf16 exp 6457 against 5763
    //    at lag 0; fp32 fma 7160 at 4 stages against 6827), except that the
    //    one-operand ops sqrt and exp with stages of 16 KB or more take two
    //    warps at lag 0 from 4 stages (bf16 exp 6545 against 5755; with
    //    4 KB stages fp32 exp keeps lag 1, 6415 against 6282);
    //  - 6 stages and more: one store warp, lag 2 (fp32 fma 7129 against
    //    6757 at lag 1).
    // The producer and store warps of the one-operand ops sqrt and exp
    // wait on lane 0 alone, the others with every lane (bf16 sqrt at 3
    // stages 6502 against 6020; bf16 mul at 3 stages 6830 against 6295 the
    // other way round).
    const int S = g.stages;
    const bool one_operand = one_operand_compute(op);
    StoreSchedule r;
    if (S <= 2) {
        const bool large_split = one_operand && S == 2 && g.slot_bytes >= 32768 && compute_groups_of(g, op) == 2;
        r.store_warps = large_split ? 1 : 2;
        r.store_lag = 0;
    } else if (S < 6) {
        r.store_warps = one_operand && S >= 4 && stage_bytes >= 16384 ? 2 : 1;
        r.store_lag = r.store_warps == 2 ? 0 : 1;
    } else {
        r.store_warps = 1;
        r.store_lag = 2;
    }
    r.lane0_wait = one_operand;
    if (g.knobs.store_warps > 0)
        r.store_warps = g.knobs.store_warps;
    if (g.knobs.store_lag >= 0)
        r.store_lag = g.knobs.store_lag;
    if (g.knobs.role_wait > 0)
        r.lane0_wait = g.knobs.role_wait == 2;
    // A store warp waits on a stage's barrier for the phase of its tile i
    // having seen only its own earlier tiles (i - W, i - 2 W, ...) complete.
    // A parity wait is exact only once the stage's previous phase (tile
    // i - S) has completed.  The compute warps complete tiles in order, so
    // for every op with a compute step (the store waits on `computed`)
    // W <= S is enough.  Copy's store waits on `full`, whose phases the TMA
    // loads complete in any order across stages: there the stage's previous
    // phase must be the same warp's own tile, i.e. W must divide S.
    if (r.store_warps > S)
        r.store_warps = S;
    if (op == TSX_COPY && S % r.store_warps != 0)
        r.store_warps = 1;
    return r;
}

int resolve_knobs(const tsx_tuning* t, Knobs* k, std::string* why)
{
    *k = Knobs{};
    if (!t)
        return TSX_OK;
    if (t->threads > 0) {
        if (t->threads % 32 || t->threads > kMaxThreads)
            return fail(why, "tuning.threads must be a multiple of 32 of at most %lld (got %lld)", kMaxThreads,
                        t->threads),
                   TSX_ERR_INVALID;
        k->threads = t->threads;
    }
    k->ctas_per_sm = t->ctas_per_sm > 0 ? t->ctas_per_sm : 0;
    if (t->store_lag > 3)
        return fail(why, "tuning.store_lag must be at most 3 (got %lld)", t->store_lag), TSX_ERR_INVALID;
    k->store_lag = t->store_lag;
    if (t->store_warps > kMaxStoreWarps)
        return fail(why, "tuning.store_warps must be at most %lld (got %lld)", kMaxStoreWarps, t->store_warps),
               TSX_ERR_INVALID;
    k->store_warps = t->store_warps > 0 ? t->store_warps : 0;
    if (t->role_wait > 2)
        return fail(why, "tuning.role_wait must be 0, 1 or 2 (got %lld)", t->role_wait), TSX_ERR_INVALID;
    k->role_wait = t->role_wait > 0 ? t->role_wait : 0;
    if (t->b_prefetch > 8)
        return fail(why, "tuning.b_prefetch must be at most 8 (got %lld)", t->b_prefetch), TSX_ERR_INVALID;
    k->b_prefetch = t->b_prefetch;
    if (t->tile_order > 2)
        return fail(why, "tuning.tile_order must be 1 (static) or 2 (dynamic) (got %lld)", t->tile_order),
               TSX_ERR_INVALID;
    k->tile_order = t->tile_order > 0 ? t->tile_order : 0;
    if (t->dynamic_share > 100)
        return fail(why, "tuning.dynamic_share must be 1..100 percent (got %lld)", t->dynamic_share),
               TSX_ERR_INVALID;
    k->dynamic_share = t->dynamic_share > 0 ? t->dynamic_share : 0;
    if (t->store_split > 2)
        return fail(why, "tuning.store_split must be 1 or 2 (got %lld)", t->store_split), TSX_ERR_INVALID;
    k->store_split = t->store_split > 0 ? t->store_split : 0;
    if (t->l2_promotion > 3)
        return fail(why, "tuning.l2_promotion must be 0..3 (got %lld)", t->l2_promotion), TSX_ERR_INVALID;
    k->l2_promotion = t->l2_promotion < 0 ? 2 : t->l2_promotion;
    k->timeout_ms = t->timeout_ms > 0 ? t->timeout_ms : 1000;
    k->checked = t->checked != 0;
    return TSX_OK;
}

int make_geometry(int dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows, int box_cols, int stages,
                  int variant, const Knobs& knobs, Geometry* g, std::string* why)
{
    *g = Geometry{};
    g->knobs = knobs;
    if (dtype < TSX_F16 || dtype > TSX_F32)
        return fail(why, "unknown dtype %lld", dtype), TSX_ERR_INVALID;
    if (variant < TSX_TMA || variant > TSX_TMA_PROMOTED)
        return fail(why, "unknown variant %lld", variant), TSX_ERR_INVALID;
    if (rows < 0 || cols < 0)
        return fail(why, "negative shape %lld x %lld", rows, cols), TSX_ERR_INVALID;
    if (pitch < cols)
        return fail(why, "the row pitch (%lld) is shorter than a row (%lld)", pitch, cols), TSX_ERR_INVALID;
    if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31) || pitch >= (int64_t(1) << 40))
        return fail(why, "rows and cols must be < 2^31 (got %lld x %lld)", rows, cols), TSX_ERR_UNSUPPORTED;
    if (box_rows < 1 || box_cols < 1)
        return fail(why, "box dims must be >= 1 (got %lld x %lld)", box_rows, box_cols), TSX_ERR_UNSUPPORTED;
    if (stages < 1 || stages > kMaxStages)
        return fail(why, "stages must be in [1, %lld] (got %lld)", kMaxStages, stages), TSX_ERR_UNSUPPORTED;

    const int es = elem_size(dtype);
    g->dtype = dtype;
    g->es = es;
    g->variant = variant;
    g->rows = rows;
    g->cols = cols;
    g->pitch = pitch;
    g->box_rows = box_rows;
    g->box_cols = box_cols;
    g->stages = stages;
    g->tiles_r = rows == 0 ? 0 : (rows + box_rows - 1) / box_rows;
    g->tiles_c = cols == 0 ? 0 : (cols + box_cols - 1) / box_cols;
    g->tiles = g->tiles_r * g->tiles_c;

    const int64_t row_bytes = int64_t(box_cols) * es;
    const int64_t tile_bytes = row_bytes * box_rows;
    if (tile_bytes > kMaxDynSmem)
        return fail(why, "a %lld-byte stage tile cannot fit in shared memory", tile_bytes), TSX_ERR_UNSUPPORTED;

    if (is_tma_variant(variant)) {
        // Global strides of a tensor map are multiples of 16 bytes.
        if ((pitch * es) % 16)
            return fail(why, "TMA needs a row pitch that is a multiple of 16 bytes (pitch * elem = %lld)",
                        pitch * es),
                   TSX_ERR_UNSUPPORTED;
        // The innermost box spans at most one 128-byte swizzle atom and a
        // whole number of 16-byte units; a wider tile row is several atoms.
        if (row_bytes % 16)
            return fail(why, "a tile row of %lld bytes is not a multiple of 16", row_bytes), TSX_ERR_UNSUPPORTED;
        // Element-type promotion: one box spans the whole tile row, with no
        // swizzle, viewed in elements widened along 1 -> 2 -> 4 -> 8 bytes
        // until the row holds at most 256 of them.
        int tma_es = es;
        if (variant == TSX_TMA_PROMOTED) {
            tma_es = 0;
            for (int pes : {1, 2, 4, 8}) {
                if (pes < es || row_bytes % pes || (cols * es) % pes)
                    continue;
                if (row_bytes / pes <= kBoxMax) {
                    tma_es = pes;
                    break;
                }
            }
            if (!tma_es)
                return fail(why, "no element of 8 bytes or less holds a %lld-byte tile row in 256", row_bytes),
                       TSX_ERR_UNSUPPORTED;
        }
        g->tma_es = tma_es;
        const int inner_bytes = variant == TSX_TMA_PROMOTED ? int(row_bytes)
                              : row_bytes < kSwizzleAtom ? int(row_bytes) : kSwizzleAtom;
        if (row_bytes % inner_bytes)
            return fail(why, "a tile row of %lld bytes is not a whole number of 128-byte atoms", row_bytes),
                   TSX_ERR_UNSUPPORTED;
        // Every box dimension is at most 256: taller tiles take several
        // equal row chunks.
        const int chunks = (box_rows + kBoxMax - 1) / kBoxMax;
        if (box_rows % chunks)
            return fail(why, "%lld tile rows cannot be cut into equal chunks of at most 256", box_rows),
                   TSX_ERR_UNSUPPORTED;
        g->inner_bytes = inner_bytes;
        g->inner_elems = inner_bytes / es;
        g->atoms = int(row_bytes / inner_bytes);
        g->row_chunks = chunks;
        g->rows_per_load = box_rows / chunks;
        g->swizzle_bytes = variant != TSX_TMA_PROMOTED && (inner_bytes == 32 || inner_bytes == 64 || inner_bytes == 128)
                               ? inner_bytes : 0;
        const uint32_t atom_bytes = uint32_t(g->rows_per_load) * inner_bytes;
        if (variant != TSX_TMA_RANK3) {
            g->loads_per_operand = g->atoms * g->row_chunks;
            g->bytes_per_load = int(atom_bytes);
            // each box lands on its own 1024-byte boundary: the swizzle
            // pattern repeats every 1024 bytes
            g->load_smem_bytes = round_up(atom_bytes, g->swizzle_bytes ? kSmemAlign : 128);
        } else {
            if (cols % g->inner_elems)
                return fail(why, "the rank-3 form needs cols to be a whole number of %lld-element atoms",
                            g->inner_elems),
                       TSX_ERR_UNSUPPORTED;
            if (g->atoms > kBoxMax)
                return fail(why, "%lld atoms per tile row exceed a box dimension", g->atoms), TSX_ERR_UNSUPPORTED;
            if (g->swizzle_bytes && atom_bytes % kSmemAlign)
                return fail(why, "the rank-3 form needs rows_per_load * 128 B to be a multiple of 1024 (%lld)",
                            atom_bytes),
                       TSX_ERR_UNSUPPORTED;
            g->loads_per_operand = g->row_chunks;
            g->bytes_per_load = int(atom_bytes) * g->atoms;
            g->load_smem_bytes = round_up(uint32_t(g->bytes_per_load), g->swizzle_bytes ? kSmemAlign : 128);
        }
        g->slot_bytes = g->load_smem_bytes * uint32_t(g->loads_per_operand);
        g->copy_vec_bytes = 0;
    } else {
        // cp.async copies 16, 8 or 4 bytes; the synchronous variant uses the
        // same widths.  The widest one dividing the row pitch and the tile
        // row is taken (base pointers are checked per call).
        int vb = 0;
        for (int cand : {16, 8, 4}) {
            if ((pitch * es) % cand == 0 && row_bytes % cand == 0) {
                vb = cand;
                break;
            }
        }
        if (!vb)
            return fail(why, "no copy width of 16, 8 or 4 bytes divides the rows (%lld-byte tile row)", row_bytes),
                   TSX_ERR_UNSUPPORTED;
        g->copy_vec_bytes = vb;
        g->slot_bytes = round_up(uint32_t(tile_bytes), 16);
    }
    // the tensor maps' L2 promotion (the TVM page passes 128 B)
    g->l2_promotion = knobs.l2_promotion;
    if (is_tma_variant(variant) && knobs.threads > kMaxThreads - 32 * tma_role_warps(kMaxStoreWarps))
        return fail(why, "tuning.threads: at most %lld compute threads beside the TMA role warps",
                    kMaxThreads - 32 * tma_role_warps(kMaxStoreWarps)),
               TSX_ERR_INVALID;
    return TSX_OK;
}

int make_op_geometry(const Geometry& g, int op, int max_smem, OpGeometry* og, std::string* why)
{
    *og = OpGeometry{};
    if (op < TSX_COPY || op > TSX_FMA)
        return fail(why, "unknown op %lld", op), TSX_ERR_INVALID;
    og->op = op;
    og->n_in = op_arity(op);
    const bool tma = is_tma_variant(g.variant);
    og->n_tma = tma ? tma_operands(g.variant, op) : 0;
    og->stage_bytes = g.slot_bytes * uint32_t(tma ? og->n_tma : og->n_in);
    const int stages = g.variant == TSX_SYNC ? 1 : g.stages;
    if (tma) {
        // expect_tx of a stage: every load of every operand
        og->tx_bytes = uint32_t(og->n_tma) * uint32_t(g.loads_per_operand) * uint32_t(g.bytes_per_load);
        // stages, three barriers per stage, the abort flag, alignment slack
        og->smem_bytes = size_t(stages) * og->stage_bytes + size_t(stages) * kTmaBarrierBytes + 16 + kSmemAlign;
    } else {
        og->tx_bytes = 0;
        og->smem_bytes = size_t(stages) * og->stage_bytes;
    }
    if (og->smem_bytes > size_t(max_smem))
        return fail(why, "%lld bytes of shared memory needed, %lld available", (long long)og->smem_bytes, max_smem),
               TSX_ERR_UNSUPPORTED;
    if (tma) {
        const StoreSchedule ss = store_schedule(g, op, og->stage_bytes);
        og->store_warps = ss.store_warps;
        og->store_lag = ss.store_lag;
        og->lane0_wait = ss.lane0_wait;
        // the dynamic order is built into the copy kernels only (ops with a
        // compute step measured slower with it on GB300).  Tiles of 16 KB or
        // more have every tile past the static prefix claimed; smaller ones
        // the last quarter only (claiming all of them, an fp32 copy in 4 KB
        // tiles ran at half the speed; the last quarter gained up to 33 %)
        og->tile_order = op == TSX_COPY ? (g.knobs.tile_order > 0 ? g.knobs.tile_order : 2) : 1;
        const int share = g.slot_bytes >= kDynamicAllTileBytes ? 100 : 25;
        og->dynamic_share = og->tile_order == 2 ? (g.knobs.dynamic_share > 0 ? g.knobs.dynamic_share : share) : 0;
        og->compute_groups = compute_groups_of(g, op);
    }
    // every CTA that fits, unless forced or capped by a rule below
    og->ctas_cap = g.knobs.ctas_per_sm > 0 ? g.knobs.ctas_per_sm : 0;
    // the mixed variant's L2 prefetch of b, for the CTAs that shared memory
    // alone would fit (the launch recomputes it for the resident CTAs)
    if (g.variant == TSX_TMA_MIXED && og->n_in >= 2) {
        const size_t per_cta = og->smem_bytes + kSmemPerCtaReserved;
        og->b_prefetch_ahead = mixed_prefetch_ahead(g, int(kSmemPerSm / per_cta));
    }
    og->threads = default_threads(g, op, og->smem_bytes, g.slot_bytes / 16, og->store_warps);
    if (g.variant == TSX_TMA_MIXED && og->n_in >= 2 &&
        og->threads + 32 * tma_role_warps(og->store_warps) > kMixedMaxThreads)
        return fail(why, "the mixed variant runs at most %lld threads per CTA (%lld asked)", kMixedMaxThreads,
                    og->threads + 32 * tma_role_warps(og->store_warps)),
               TSX_ERR_UNSUPPORTED;
    const bool tma_rules = tma && g.variant != TSX_TMA_MIXED && g.knobs.threads <= 0 && g.knobs.ctas_per_sm <= 0;
    // Two-stage rings on long streams: enough CTAs for the op's target of
    // stage bytes per SM (halves round up), sharing 512 compute threads per
    // SM (256 for copy).  One stage loads while the other is computed and
    // stored, so the CTAs that fit hold too much or too little in flight.
    // Measured on GB300 over fp32 8x128, 8x256 and 16x128 tiles and bf16
    // 128x128, 64x128, 32x128 and 64x64 tiles of every op, against every
    // CTA that fits with the usual thread share: +0 to +41 % (bf16 exp in
    // 64x128 tiles 4483 -> 6343 GB/s, fp32 add in 16x128 tiles 5248 -> 6730,
    // fp32 add in 8x128 tiles 6303 -> 6870), nowhere lower by more than the
    // noise.  bf16 exp [16384, 16384] in 128x128 tiles keeps its two CTAs of
    // 256 threads (6467 GB/s against 5760 with the three that fit).  Short
    // streams (a few tiles per CTA, bound by latency) keep the usual share.
    if (tma_rules && g.stages == 2 && g.tiles >= kTwoStageStreamTiles) {
        const int64_t ring = 2 * int64_t(og->stage_bytes);
        int64_t want = (two_stage_ring_per_sm(op) + ring / 2) / ring;   // halves round up
        want = want < 1 ? 1 : want;
        og->ctas_cap = int(want);
        const int threads = int((op == TSX_COPY ? 256 : 512) / want) / 32 * 32;
        og->threads = threads < 32 ? 32 : threads;
    }
    // Rings of four or more small stages (under 16 KB) of sqrt and exp:
    // enough CTAs for about 144 KB of stages per SM, sharing about 256
    // compute threads (one warp at least), or 576 (two warps at least) for
    // fp32 sqrt, which needs more threads per byte.  Measured on GB300 over
    // fp32 8x128, 8x256 and 16x128 tiles and bf16 32x128, 64x64 and 16x256
    // tiles at 4, 6 and 8 stages, against every CTA that fits with the usual
    // thread share: exp and 16-bit sqrt +1 to +22 %, fp32 sqrt -2 to +31 %;
    // three stages were mixed (two have the rule above).
    const bool sqrt32 = op == TSX_SQRT && g.es == 4;
    if (tma_rules && (op == TSX_EXP || op == TSX_SQRT) && og->stage_bytes < 16384 && g.stages >= 4) {
        const int64_t ring = int64_t(g.stages) * og->stage_bytes;
        int64_t want = (kSmallRingPerSm + ring / 2 - 1) / ring;   // halves round down
        want = want < 1 ? 1 : want;
        og->ctas_cap = int(want);
        const int least = sqrt32 ? 64 : 32;
        int threads = int((sqrt32 ? 576 : 256) / want) / 32 * 32;
        og->threads = threads < least ? least : threads > 512 ? 512 : threads;
    }
    // The same target for add and mul on long streams (at least 32768 tiles)
    // from three stages on, where it leaves two CTAs per SM or more:
    // measured on GB300 over fp32 8x128 and 8x64 tiles and bf16 64x64 and
    // 32x128 tiles, +0 to +12 % (a single CTA lost 1-9 %; two stages have
    // the rule above).
    if (tma_rules && (op == TSX_ADD || op == TSX_MUL) && g.stages >= 3 && g.tiles >= kLongStreamTiles) {
        const int64_t ring = int64_t(g.stages) * og->stage_bytes;
        const int64_t want = (kSmallRingPerSm + ring / 2 - 1) / ring;
        if (want >= 2) {
            og->ctas_cap = int(want);
            const int threads = int(256 / want) / 32 * 32;
            og->threads = threads < 32 ? 32 : threads;
        }
    }
    // The mixed variant: as few compute threads as hold b a tile ahead
    // (kSetUnits 16-byte units each), so that registers leave room for more
    // CTAs; fma (two operands staged) keeps every CTA that fits, add and mul
    // (a alone staged) aim at about 96 KB of stages per SM.  Measured on
    // GB300 against the thread share above over fp32 8x64, 8x128, 8x256 and
    // 16x128 tiles and bf16 32x64, 32x128, 64x64, 64x128 and 128x128 tiles at
    // 2 to 8 stages: +0 to +49 % (fp32 fma 8x128 at 6 stages 5959 -> 6943
    // GB/s, at 8 stages 4433 -> 6624; bf16 add 64x64 at 6 stages 6005 ->
    // 6679), never below the share by more than the noise.
    if (g.knobs.threads <= 0 && g.knobs.ctas_per_sm <= 0 && g.variant == TSX_TMA_MIXED && og->n_in >= 2) {
        const int cover = int((g.slot_bytes / 16 + kSetUnits - 1) / kSetUnits + 31) / 32 * 32;
        const int most = kMixedMaxThreads - 32 * tma_role_warps(og->store_warps);
        og->threads = cover < most ? cover : most;
        if (og->n_in == 2) {
            const int64_t ring = int64_t(g.stages) * og->stage_bytes;
            const int64_t want = (kMixedRingPerSm + ring / 2 - 1) / ring;   // halves round down
            og->ctas_cap = int(want < 1 ? 1 : want);
        } else {
            og->ctas_cap = 0;
        }
    }
    og->block_threads = og->threads + (tma ? 32 * tma_role_warps(og->store_warps) : 0);
    // [outer, threads, vec] of the elementwise stage: 16-byte vectors
    og->vec = 16 / g.es;
    const uint32_t units = g.slot_bytes / 16;
    og->outer = int((units + og->threads - 1) / og->threads);
    og->vec16_per_slot = units;
    return TSX_OK;
}

void fill_info(const Geometry& g, const OpGeometry& og, tsx_plan_info* info)
{
    std::memset(info, 0, sizeof *info);
    info->dtype = g.dtype;
    info->variant = g.variant;
    info->op = og.op;
    info->n_in = og.n_in;
    info->elem_size = g.es;
    info->box_rows = g.box_rows;
    info->box_cols = g.box_cols;
    info->stages = g.stages;
    info->rows = g.rows;
    info->cols = g.cols;
    info->pitch = g.pitch;
    info->tiles = g.tiles;
    info->tiles_r = g.tiles_r;
    info->tiles_c = g.tiles_c;
    info->inner_elems = g.inner_elems;
    info->inner_bytes = g.inner_bytes;
    info->atoms = g.atoms;
    info->rows_per_load = g.rows_per_load;
    info->row_chunks = g.row_chunks;
    info->loads_per_operand = g.loads_per_operand;
    info->bytes_per_load = g.bytes_per_load;
    info->tx_bytes = int32_t(og.tx_bytes);
    info->threads = og.threads;
    info->block_threads = og.block_threads;
    info->tma_elem_bytes = g.tma_es;
    info->store_lag = is_tma_variant(g.variant) ? og.store_lag : 0;
    info->store_warps = is_tma_variant(g.variant) ? og.store_warps : 0;
    info->role_wait = is_tma_variant(g.variant) ? (og.lane0_wait ? 2 : 1) : 0;
    info->b_prefetch = og.b_prefetch_ahead;
    info->tile_order = og.tile_order;
    info->dynamic_share = og.dynamic_share;
    info->compute_groups = is_tma_variant(g.variant) ? og.compute_groups : 0;
    info->timeout_ms = g.knobs.timeout_ms;
    info->vec = og.vec;
    info->outer = og.outer;
    info->copy_vec_bytes = g.copy_vec_bytes;
    info->slot_bytes = int32_t(g.slot_bytes);
    info->stage_bytes = int32_t(og.stage_bytes);
    info->smem_bytes = int32_t(og.smem_bytes);
    if (is_tma_variant(g.variant)) {
        TensorMapArgs m;
        tensor_map_args(g, &m);
        info->rank = m.rank;
        for (int d = 0; d < m.rank; ++d) {
            info->global_dim[d] = m.dims[d];
            info->box_dim[d] = m.box[d];
            info->element_strides[d] = 1;
        }
        for (int d = 0; d + 1 < m.rank; ++d)
            info->global_stride_bytes[d] = m.strides[d];
        info->interleave = 0;                       // CU_TENSOR_MAP_INTERLEAVE_NONE
        info->swizzle = m.swizzle;
        info->l2_promotion = m.l2_promotion;        // CUtensorMapL2promotion value
        info->oob_fill = 0;                         // CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE: zeros
    }
}

void fill_tma_args(const Geometry& g, const OpGeometry& og, int* status, int64_t fault_tile, TmaArgs* args)
{
    *args = TmaArgs{};
    args->tiles = g.tiles;
    args->tiles_c = g.tiles_c;
    args->tiles_r = g.tiles_r;
    args->pitch = g.pitch;
    args->fault_tile = fault_tile;
    args->status = status;
    args->timeout_ns = uint64_t(g.knobs.timeout_ms) * 1000000ull;
    args->rows = int(g.rows);
    args->cols = int(g.cols);
    args->box_rows = g.box_rows;
    args->box_cols = g.box_cols;
    args->stages = g.stages;
    args->inner_elems = g.inner_elems;
    args->atoms = g.atoms;
    args->rows_per_load = g.rows_per_load;
    args->row_chunks = g.row_chunks;
    args->rank3 = g.variant == TSX_TMA_RANK3;
    args->load_smem_bytes = g.load_smem_bytes;
    args->slot_bytes = g.slot_bytes;
    args->stage_bytes = og.stage_bytes;
    args->bytes_per_load = uint32_t(g.bytes_per_load);
    args->vec16_per_slot = og.vec16_per_slot;
    args->store_lag = og.store_lag;
    args->store_warps = og.store_warps;
    args->lane0_wait = og.lane0_wait ? 1 : 0;
    args->b_prefetch_ahead = og.b_prefetch_ahead;
    args->promote_shift = g.tma_es == 8 * g.es ? 3 : g.tma_es == 4 * g.es ? 2 : g.tma_es == 2 * g.es ? 1 : 0;
    args->box_bytes = uint32_t(g.rows_per_load) * uint32_t(g.inner_bytes);
    args->swizzle_mask = g.swizzle_bytes == 128 ? 7 : g.swizzle_bytes == 64 ? 3 : g.swizzle_bytes == 32 ? 1 : 0;
}

int64_t static_tiles_per_cta(const Geometry& g, const OpGeometry& og, int64_t grid)
{
    const int64_t least = g.stages > 1 ? g.stages - 1 : 1;
    if (grid < 1)
        return least;
    const int64_t share = og.dynamic_share > 0 ? og.dynamic_share : 100;
    const int64_t most = (g.tiles / grid) * (100 - share) / 100;
    return most > least ? most : least;
}

void tensor_map_args(const Geometry& g, TensorMapArgs* m)
{
    *m = TensorMapArgs{};
    m->l2_promotion = g.l2_promotion;
    m->swizzle = g.swizzle_bytes == 128 ? 3 : g.swizzle_bytes == 64 ? 2 : g.swizzle_bytes == 32 ? 1 : 0;
    // dims[0] is the innermost (contiguous) dimension
    const uint64_t rows = uint64_t(g.rows), cols = uint64_t(g.cols);
    if (g.variant == TSX_TMA_RANK3) {
        // [cols / atom, rows, atom]: the atom axis strides by one atom
        m->rank = 3;
        m->dims[0] = uint64_t(g.inner_elems);
        m->dims[1] = rows;
        m->dims[2] = cols / uint64_t(g.inner_elems);
        m->strides[0] = uint64_t(g.pitch) * uint64_t(g.es);
        m->strides[1] = uint64_t(g.inner_bytes);
        m->box[0] = uint32_t(g.inner_elems);
        m->box[1] = uint32_t(g.rows_per_load);
        m->box[2] = uint32_t(g.atoms);
    } else {
        // rank 2; a promoted map counts the row in its wider elements
        const uint64_t widen = uint64_t(g.tma_es) / uint64_t(g.es);
        m->rank = 2;
        m->dims[0] = cols / widen;
        m->dims[1] = rows;
        m->strides[0] = uint64_t(g.pitch) * uint64_t(g.es);
        m->box[0] = uint32_t(uint64_t(g.inner_elems) / widen);
        m->box[1] = uint32_t(g.rows_per_load);
    }
}

}  // namespace tsx

extern "C" void tsx_tuning_defaults(tsx_tuning* t)
{
    if (!t)
        return;
    t->threads = 0;
    t->ctas_per_sm = 0;
    t->store_lag = -1;
    t->store_warps = 0;
    t->role_wait = 0;
    t->b_prefetch = -1;
    t->tile_order = 0;
    t->dynamic_share = 0;
    t->store_split = 0;
    t->l2_promotion = -1;
    t->timeout_ms = 0;
    t->checked = 0;
}

extern "C" int tsx_plan_query_tuned(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                                    int box_cols, int stages, tsx_variant variant, const tsx_tuning* tuning,
                                    tsx_op op_arg, tsx_plan_info* info)
{
    std::string why;
    tsx::Geometry g;
    tsx::Knobs knobs;
    int op;
    bool accumulate;
    if (!tsx::split_op(op_arg, &op, &accumulate)) {
        tsx::set_last_error("unknown op");
        return TSX_ERR_INVALID;
    }
    if (accumulate && variant != TSX_TMA && variant != TSX_TMA_RANK3) {
        tsx::set_last_error("TSX_ACCUMULATE needs TSX_TMA or TSX_TMA_RANK3");
        return TSX_ERR_UNSUPPORTED;
    }
    int rc = tsx::resolve_knobs(tuning, &knobs, &why);
    if (rc == TSX_OK)
        rc = tsx::make_geometry(dtype, rows, cols, pitch, box_rows, box_cols, stages, variant, knobs, &g, &why);
    if (rc == TSX_OK) {
        tsx::OpGeometry og;
        rc = tsx::make_op_geometry(g, op, tsx::kMaxDynSmem, &og, &why);
        if (rc == TSX_OK && info)
            tsx::fill_info(g, og, info);
    }
    tsx::set_last_error(rc == TSX_OK ? "" : why.c_str());
    return rc;
}

extern "C" int tsx_plan_query_pitched(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                                      int box_cols, int stages, tsx_variant variant, tsx_op op, tsx_plan_info* info)
{
    return tsx_plan_query_tuned(dtype, rows, cols, pitch, box_rows, box_cols, stages, variant, nullptr, op, info);
}

extern "C" int tsx_plan_query(tsx_dtype dtype, int64_t rows, int64_t cols, int box_rows, int box_cols, int stages,
                              tsx_variant variant, tsx_op op, tsx_plan_info* info)
{
    return tsx_plan_query_tuned(dtype, rows, cols, cols, box_rows, box_cols, stages, variant, nullptr, op, info);
}
