/*
 * tsx.h -- tile-elementwise streaming on NVIDIA GB300 (sm_103a).
 *
 * One operation: stream a dense row-major 2-D tensor [rows, cols] tile by
 * tile from global into shared memory through an S-stage circular buffer
 * whose stages are guarded by mbarriers, apply an elementwise op to each
 * staged tile in shared memory, and write the result tile back to global.
 *
 * Sources for the operation (cited by page title and section):
 *  - TVM docs "copy_async -> tma": one elected thread issues a
 *    descriptor-driven bulk tensor copy; the descriptor is encoded once on
 *    the host; completion is signalled on the caller's mbarrier
 *    (introduction, "Demonstration program", "Algorithm" steps 2-4).
 *  - TVM docs "elementwise -> smem": the op is applied to operands that all
 *    live in shared memory under an [outer, threads, vec] partition
 *    ("Algorithm", "Generated CUDA").
 *  - nvFuser PR #2833 "Add TMA support for circular buffering pass": the
 *    pre-prologue / prologue / main / epilogue / post-epilogue loops, box
 *    dimensions of at most 256, and expect_tx = bytes per load x loads per
 *    stage ("Lowering Details", "Loop Structure", "Detailed Pseudo-Code").
 *  - TVM docs "copy_async -> ldgsts": the cp.async variant kept as an
 *    ablation ("Algorithm", table under "How inputs change the algorithm").
 *
 * Conventions for every entry point:
 *  - Device pointers are CUDA device (or managed) addresses on the device
 *    that was current when the plan was created (TSX_LDGSTS and TSX_SYNC
 *    also take pinned host memory; see tsx_ewise).  The caller owns every
 *    buffer and keeps it alive until the work queued on the stream is done.
 *  - Tensors are row-major: element (r, c) sits at byte offset
 *    (r * pitch + c) * element_size from the base pointer, pitch = cols
 *    unless the plan was created with tsx_plan_create_pitched.
 *  - Functions returning int return a tsx_status (0 = TSX_OK, negative =
 *    error).  On an error nothing was queued on the stream, and
 *    tsx_last_error() describes it.
 *  - A plan may be used by one host thread at a time; different plans are
 *    independent.
 */
#ifndef TSX_H
#define TSX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  Arithmetic on 16-bit types is carried out in fp32 and
 * rounded once to nearest-even into the element type; fma and sqrt use the
 * native 16-bit instructions, one rounding of the exact result. */
typedef enum { TSX_F16 = 0, TSX_BF16 = 1, TSX_F32 = 2 } tsx_dtype;

/* How stages are filled.
 *  TSX_TMA       the producer warp issues the cp.async.bulk.tensor loads of
 *                a tile, one box per lane (one rank-2 box per 128-byte atom
 *                of a tile row and per <= 256-row chunk), completing on the
 *                stage's mbarrier, whose expect_tx lane 0 announces (the
 *                pages issue from one elected thread); the result goes back
 *                with cp.async.bulk.tensor stores.  The primary path.
 *  TSX_LDGSTS    every thread issues cp.async (LDGSTS) copies of 16, 8 or 4
 *                bytes; commit_group / wait_group per stage; the result is
 *                written with vector stores.  Ablation.
 *  TSX_SYNC      plain synchronous vector loads into shared memory, one
 *                stage; ablation (stages is ignored beyond validation).
 *  TSX_TMA_RANK3 as TSX_TMA, but one rank-3 box covers all 128-byte atoms of
 *                a row chunk ("copy_async -> tma", "Generated TIRx IR");
 *                needs cols to be a whole number of atoms.
 *  TSX_TMA_MIXED as TSX_TMA for a (and c), while b is read by the compute
 *                threads with plain vector loads from global memory, one
 *                tile ahead into registers: one operand through the TMA
 *                circular buffer, the other through Set circular buffering
 *                (nvFuser PR #2833, "Testing Setup", Pointwise).  Unary ops
 *                run as TSX_TMA.
 *  TSX_TMA_PROMOTED  one box per <= 256-row chunk spans the whole tile row,
 *                with no swizzle: the tensor map counts in elements widened
 *                along 1 -> 2 -> 4 -> 8 bytes until the row holds at most
 *                256 of them ("copy_async -> tma", table under "How inputs
 *                change the algorithm": box > 256 triggers element-type
 *                promotion).  Declines when even 8 bytes cannot. */
typedef enum {
    TSX_TMA = 0, TSX_LDGSTS = 1, TSX_SYNC = 2, TSX_TMA_RANK3 = 3, TSX_TMA_MIXED = 4, TSX_TMA_PROMOTED = 5
} tsx_variant;

/* Elementwise ops ("elementwise -> smem", table under "How inputs change
 * the algorithm").  copy moves bits unchanged; sqrt and add/mul/fma are
 * correctly rounded; exp is within 2 ulp (fp32) or 1 ulp (fp16, bf16) of the
 * exact value.
 *
 * TSX_ACCUMULATE, OR-ed into an op, turns the store into a TMA reduce-store
 * ("copy_async -> tma", table under "How inputs change the algorithm":
 * s2g with a reduce op): out = out + op(a, b, c), the sum rounded to nearest
 * even into the element type and added by the TMA unit in global memory.
 * Offered by TSX_TMA and TSX_TMA_RANK3 (else TSX_ERR_UNSUPPORTED).
 *
 * TSX_ROW_SUMS, OR-ed into an op, is understood by tsx_plan_get_info only:
 * it asks for the launch tsx_reduce_rows makes for that op. */
typedef enum {
    TSX_COPY = 0, TSX_SQRT = 1, TSX_EXP = 2, TSX_ADD = 3, TSX_MUL = 4, TSX_FMA = 5,
    TSX_ACCUMULATE = 0x100,
    TSX_ROW_SUMS = 0x200
} tsx_op;

typedef enum {
    TSX_OK = 0,
    TSX_ERR_INVALID = -1,     /* bad handle, op, shape, NULL / extra operand */
    TSX_ERR_UNSUPPORTED = -2, /* no legal plan for this shape / variant ("declines") */
    TSX_ERR_ALIGN = -3,       /* a base pointer is not aligned as the variant needs */
    TSX_ERR_CUDA = -4,        /* a CUDA runtime or driver call failed */
    TSX_ERR_TIMEOUT = -5,     /* a device-side wait gave up (see tsx_plan_status) */
    TSX_ERR_NOMEM = -6        /* host or device allocation failed */
} tsx_status;

/* A CUDA stream: the same type as cudaStream_t (pass 0 for the legacy
 * default stream). */
struct CUstream_st;
typedef struct CUstream_st *tsx_stream_t;

typedef struct tsx_plan *tsx_plan_t;

/* Everything the planner decided, as plain numbers (see tsx_plan_query). */
typedef struct tsx_plan_info {
    int32_t dtype, variant, op, n_in, elem_size;
    int32_t box_rows, box_cols, stages;
    int64_t rows, cols, tiles, tiles_r, tiles_c;
    /* TMA box split ("Lowering Details"): loads per operand and stage, and
     * the expect_tx byte count of one stage = n_in * loads * bytes_per_load */
    int32_t inner_elems, inner_bytes, atoms, rows_per_load, row_chunks;
    int32_t loads_per_operand, bytes_per_load, tx_bytes;
    /* tensor-map encode arguments, innermost dimension first */
    int32_t rank;
    uint64_t global_dim[5];
    uint64_t global_stride_bytes[4];
    uint32_t box_dim[5];
    uint32_t element_strides[5];
    int32_t interleave, swizzle, l2_promotion, oob_fill; /* CUtensorMap* enum values */
    /* [outer, threads, vec] of the shared-memory elementwise stage, in
     * elements of the element type (vec = 16 bytes); copy_vec_bytes is the
     * width of one cp.async / vector copy for TSX_LDGSTS and TSX_SYNC */
    int32_t threads, vec, outer, copy_vec_bytes;
    /* shared memory: one operand's slot, one stage, the whole CTA */
    int32_t slot_bytes, stage_bytes;
    int32_t smem_bytes;
    /* launch (0 from tsx_plan_query, which does not look at a GPU) */
    int32_t ctas_per_sm, grid, sm_count;
    /* threads of one CTA: for the TMA variants the elementwise threads plus
     * a producer warp and a store warp */
    int32_t block_threads;
    /* elements between the starts of consecutive rows (cols for dense rows) */
    int64_t pitch;
    /* element size the tensor map counts in: elem_size, or the wider one
     * of TSX_TMA_PROMOTED */
    int32_t tma_elem_bytes;
    /* TMA variants: tiles between a store's issue and the release of its
     * stage (the store warp checks cp.async.bulk.wait_group.read that many
     * tiles later) */
    int32_t store_lag;
    /* limit of every device-side wait, in milliseconds */
    int32_t timeout_ms;
    /* TMA variants: store warps, which take a CTA's tiles in turn (each
     * counts store_lag in its own tiles), and how the producer and store
     * warps wait on their mbarriers (1 every lane, 2 lane 0 alone) */
    int32_t store_warps, role_wait;
    /* TSX_TMA_MIXED: how many of a CTA's tiles beyond the tile it loads the
     * producer prefetches b into L2 (from the CTAs per SM: tsx_plan_query
     * assumes the CTAs that shared memory alone fits) */
    int32_t b_prefetch;
    /* TMA variants: the order CTAs take tiles in, 1 static (CTA c of G takes
     * c, c + G, ...), 2 dynamic (TSX_COPY: each CTA's first tiles as in the
     * static order, every later one claimed from a per-launch counter) */
    int32_t tile_order;
    /* dynamic order: the share of the tiles, in percent, claimed from the
     * counter (the launch takes the CTAs' static tiles from it) */
    int32_t dynamic_share;
    /* TMA variants: groups of a tile's boxes that the compute warps hand to
     * the store warps one by one (2: the first half is stored while the
     * second is computed) */
    int32_t compute_groups;
} tsx_plan_info;

/* Launch knobs of a plan.  Every field has a "planner's choice" value; start
 * from tsx_tuning_defaults() and set only what you want to force.  None of
 * them changes a result: the tests hold every setting to the oracle.
 *  threads       compute threads of a CTA ([outer, threads, vec]: the
 *                partition the TVM docs "elementwise -> smem" page
 *                synthesizes from the thread count, "Algorithm" step 2); a
 *                multiple of 32; <= 0: the planner's choice
 *  ctas_per_sm   at most this many resident CTAs per SM in the persistent
 *                grid; <= 0: the planner's (as many as occupancy allows,
 *                unless a rule measured on GB300 aims at a number of
 *                stage bytes per SM: two-stage rings on long streams,
 *                rings of four or more small sqrt / exp stages, add and
 *                mul on long streams, the mixed variant's add and mul,
 *                fp32 row sums; tsx_plan_get_info reports the launch's
 *                count).  For tsx_ewise, setting threads or ctas_per_sm
 *                turns those rules off; for row sums each knob replaces its
 *                own half of the rule
 *  store_lag     TMA variants: 0..3 of a store warp's tiles between a
 *                store's issue and the release of its stage; < 0: the
 *                planner's
 *  store_warps   TMA variants: 1 or 2 store warps, taking a CTA's tiles in
 *                turn, so that one can wait for its store to leave shared
 *                memory while the other stores the next tile; clamped to
 *                the stage count (a store warp's wait on a stage's phase is
 *                exact only if the stage's previous phase is behind it);
 *                <= 0: the planner's
 *  role_wait     TMA variants: how the producer and store warps wait on an
 *                mbarrier, 1 with every lane, 2 with lane 0 alone while the
 *                others take its answer; <= 0: the planner's
 *  b_prefetch    TSX_TMA_MIXED: the producer asks for b's boxes in L2 this
 *                many of the CTA's tiles beyond the tile it loads (0..8);
 *                < 0: the planner's
 *  tile_order    TMA variants, TSX_COPY: 1 static (CTA c of G takes tiles
 *                c, c + G, ...), 2 dynamic (a CTA's first tiles as in the
 *                static order, then tiles claimed in order from a counter,
 *                so that CTAs streaming faster take more tiles); <= 0: the
 *                planner's: dynamic for launches of at least 16 tiles per
 *                CTA (the host-only query, which knows no grid, reports
 *                that case).  The other ops, and TSX_ACCUMULATE, always
 *                take the static order
 *  dynamic_share dynamic order: about this percentage of the tiles (the
 *                last ones) is claimed from the counter, 1..100 (a CTA
 *                takes at least max(1, S - 1) tiles in the static order
 *                first); <= 0: the planner's (100 for tiles of 16 KB or
 *                more, 25 for smaller ones)
 *  store_split   TMA variants, ops with a compute step and an even number
 *                of boxes per tile (not the mixed variant's binary ops): 2
 *                stores the first half of a tile's boxes while the compute
 *                warps work on the second, 1 stores the tile at once; <= 0:
 *                the planner's (2 for sqrt and exp with tiles of 16 KB or
 *                more)
 *  l2_promotion  CUtensorMapL2promotion of the tensor maps, 0..3 (none, 64,
 *                128, 256 B); < 0: 128 B, the value of TVM docs
 *                "copy_async -> tma" ("Generated TIRx IR")
 *  timeout_ms    limit of every device-side wait; <= 0: 1000
 *  checked       non-zero: tsx_ewise / tsx_reduce_rows synchronize the
 *                stream and return the device status (debugging) */
typedef struct tsx_tuning {
    int32_t threads, ctas_per_sm, store_lag, l2_promotion, timeout_ms, checked, store_warps, role_wait;
    int32_t b_prefetch, tile_order, dynamic_share, store_split;
} tsx_tuning;

/* Fill *t with the planner's-choice value of every field.  No source on the
 * pages: the knobs are this library's (the measurement side of its spec
 * chooses stage count and box shape from counters; these are the rest). */
void tsx_tuning_defaults(tsx_tuning *t);

/* Create a plan for [rows, cols] tensors of `dtype`, streamed in stage
 * tiles of box_rows x box_cols through `stages` stages by `variant`.
 * Source: the library's specified call list (the pages describe a DSL, not a
 * library); what the plan fixes is the host side of TVM docs
 * "copy_async -> tma", "Algorithm" steps 2-3 (encode the descriptor once on
 * the host) and nvFuser PR #2833 "Lowering Details" (box <= 256, loads per
 * stage, expect_tx bytes).
 * Binds the plan to the current CUDA device and allocates one 4-byte device
 * status word.  rows or cols may be 0 (every call is then a no-op).
 * Limits: rows, cols < 2^31; 1 <= stages <= 16; box dims >= 1; TMA variants
 * need cols * element_size to be a multiple of 16 bytes and a tile row of a
 * whole number of 16-byte units (and of 128-byte atoms when wider than one).
 * Returns NULL on failure (tsx_last_error() says why). */
tsx_plan_t tsx_plan_create(tsx_dtype dtype, int64_t rows, int64_t cols, int box_rows, int box_cols,
                           int stages, tsx_variant variant);

/* tsx_plan_create for tensors whose rows start `pitch` elements apart
 * (pitch >= cols; the elements between a row's end and the next row's start
 * are neither read nor written): element (r, c) is at byte offset
 * (r * pitch + c) * element_size.  Every operand and the output use this
 * pitch.  TMA variants need pitch * element_size to be a multiple of 16
 * bytes; TSX_LDGSTS / TSX_SYNC narrow their copy width to what divides it.
 * This is the strided form of the tensors of TVM docs "copy_async -> tma"
 * ("Algorithm" step 3: the global strides passed to the tensor map). */
tsx_plan_t tsx_plan_create_pitched(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                                   int box_cols, int stages, tsx_variant variant);

/* tsx_plan_create_pitched with launch knobs (see tsx_tuning; NULL: every
 * field the planner's choice).  Out-of-range knobs give NULL with
 * TSX_ERR_INVALID in tsx_last_error(). */
tsx_plan_t tsx_plan_create_tuned(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                                 int box_cols, int stages, tsx_variant variant, const tsx_tuning *tuning);

/* out = op(a, b, c) element by element over the plan's [rows, cols]
 * (out += op(a, b, c) with TSX_ACCUMULATE).  Source: the library's specified
 * call list; the operation is TVM docs "copy_async -> tma" ("Algorithm"
 * steps 2-4: load a tile to shared memory, signal an mbarrier) with the op
 * applied in shared memory as in TVM docs "elementwise -> smem"
 * ("Algorithm", "Generated CUDA"), pipelined over tiles as in nvFuser PR
 * #2833 ("Loop Structure", "Detailed Pseudo-Code").
 * a is required; b is required by add / mul / fma and must be NULL
 * otherwise; c is required by fma and must be NULL otherwise (else
 * TSX_ERR_INVALID).  out may be exactly a, b or c; any other overlap is
 * undefined.  For an empty tensor (rows or cols 0) the call does nothing
 * and the pointers are not examined.  Buffers are device memory; TSX_LDGSTS
 * and TSX_SYNC plans also take page-locked host memory that the device
 * addresses directly (cudaHostAlloc, or a pinned torch tensor), in any mix
 * with device buffers: the kernel then reads and writes it over the host
 * link, with no staging copy.  Base pointers must be 16-byte aligned
 * for the TMA variants;
 * TSX_LDGSTS / TSX_SYNC narrow their copy width to the pointers' alignment
 * (16, 8 or 4 bytes) and return TSX_ERR_ALIGN below 4.
 * Asynchronous on `stream`: returns once the kernel is queued.  A device-side
 * wait that exceeds its time limit (1 s unless tsx_tuning.timeout_ms says
 * otherwise) makes the kernel record TSX_ERR_TIMEOUT in the plan's status
 * word and return; read it with tsx_plan_status.  On a plan created with
 * tsx_tuning.checked the call synchronizes the stream and returns the
 * device status instead.  After a
 * plan's first call of an op (which sets up its launch) later calls of that
 * op only launch on `stream`, so they can be captured into a CUDA graph. */
int tsx_ewise(tsx_plan_t plan, tsx_op op, const void *a, const void *b, const void *c, void *out,
              tsx_stream_t stream);

/* Row sums: row_sums[r] = sum over c of op(a, b, c)[r, c] for the plan's
 * [rows, cols]; each op result is rounded into the element type, then summed
 * in fp32 (the reduction schedules of nvFuser PR #2833, "Testing Setup":
 * Reduction, InnerPersistent).  row_sums: device fp32 [rows], 4-byte
 * aligned, overwritten.  The persistent grid splits the tiles, in row-major
 * order, into one contiguous range per CTA, so a band of box_rows rows may
 * be cut between CTAs; the shares of a cut band go through scratch that the
 * plan allocates on its first row reduction of an op, or the first
 * tsx_plan_get_info with TSX_ROW_SUMS (TSX_ERR_NOMEM if that fails), and
 * owns until it is destroyed.  Row reductions of one plan must
 * therefore not run concurrently on different streams.  The order of
 * additions depends on the plan alone, so results repeat bit for bit;
 * against the exact sum their error is at most gamma(cols - 1) * sum |x|,
 * gamma(k) = k u / (1 - k u), u = 2^-24.  TSX_TMA / TSX_TMA_RANK3 plans only
 * (else TSX_ERR_UNSUPPORTED); TSX_ACCUMULATE is rejected.  rows = 0 does
 * nothing; cols = 0 writes zeros.  Asynchronous on `stream`; device-side
 * timeouts are reported as for tsx_ewise, and results of the plan's row
 * reductions are undefined from a timeout until tsx_plan_status has been
 * read. */
int tsx_reduce_rows(tsx_plan_t plan, tsx_op op, const void *a, const void *b, const void *c, float *row_sums,
                    tsx_stream_t stream);

/* Measure the op's launch on the caller's own operands under a set of
 * candidate shapes, and keep the fastest for the plan's later tsx_ewise
 * calls of that op.  The candidates are the planner's own launch and
 * 1..8 CTAs per SM, each set sharing 256 or 512 compute threads per SM;
 * then, on the TMA variants, the fastest of those with one or two store
 * warps at lag 0 or 1 (unless the plan's knobs fix the store side).
 * Source: the measurement side of the library's specification, which
 * chooses a launch from measured throughput; the pages fix none.  Each
 * candidate is launched once, then timed over `launches` launches (<= 0:
 * 10; at most 1000) with CUDA events on `stream`, in two rounds; the
 * shortest round wins.  Results never depend on the shape, so `out` ends
 * holding op(a, b, c).  Because the op runs repeatedly, `out` must not alias
 * an input (TSX_ERR_INVALID), and TSX_ACCUMULATE is rejected
 * (TSX_ERR_INVALID).  Row sums are not tuned.  A plan created with
 * tsx_tuning.threads or ctas_per_sm keeps that shape and launches once.  A
 * traced plan is not tuned (TSX_ERR_UNSUPPORTED).  Synchronizes `stream`, so
 * it cannot be captured into a graph; the calls after it can.  Returns what
 * tsx_ewise would for the arguments, TSX_ERR_TIMEOUT if a launch's
 * device-side wait gave up (the status word is then cleared), or
 * TSX_ERR_CUDA for a CUDA error.  `chosen` may be NULL; otherwise it
 * receives the launch kept, as tsx_plan_get_info gives it. */
int tsx_plan_tune(tsx_plan_t plan, tsx_op op, const void *a, const void *b, const void *c, void *out,
                  tsx_stream_t stream, int32_t launches, tsx_plan_info *chosen);

/* Release the plan, its tensor-map cache and its device status word.
 * Source: the library's specified call list (no counterpart on the pages;
 * the post-epilogue's mbarrier.inval of nvFuser PR #2833 "Loop Structure"
 * is the device-side release, done by every launch).  NULL is ignored.  Work already queued must not need the plan's status
 * word afterwards (synchronize first). */
void tsx_plan_destroy(tsx_plan_t plan);

/* The first device-side error recorded by this plan's kernels since the
 * last call (TSX_OK if none), then clears it.  Source: the library's
 * specified call list; the pages have no error path (TVM docs
 * "copy_async -> tma" only says a variant declines, closing paragraph), so
 * the bounded mbarrier waits and this status word are this library's.  Call after synchronizing the
 * streams the plan was used on; this call itself blocks on a small
 * device-to-host copy. */
int tsx_plan_status(tsx_plan_t plan);

/* Message for the last error on the calling host thread ("" if none).  The
 * pointer stays valid until the next tsx_* call on this thread.  Source: the
 * library's specified call list (no counterpart on the pages). */
const char *tsx_last_error(void);

/* The plan tsx_plan_create would build and the launch tsx_ewise would make
 * for `op`, computed on the host alone: no CUDA call, no GPU needed
 * (ctas_per_sm, grid and sm_count are left 0).  Base pointers are assumed
 * 16-byte aligned.  Returns TSX_OK and fills *info, or the error
 * tsx_plan_create / tsx_ewise would return. */
int tsx_plan_query(tsx_dtype dtype, int64_t rows, int64_t cols, int box_rows, int box_cols, int stages,
                   tsx_variant variant, tsx_op op, tsx_plan_info *info);

/* tsx_plan_query for rows `pitch` elements apart (see tsx_plan_create_pitched). */
int tsx_plan_query_pitched(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows, int box_cols,
                           int stages, tsx_variant variant, tsx_op op, tsx_plan_info *info);

/* tsx_plan_query_pitched for a plan created with these launch knobs (NULL:
 * the planner's choices; ctas_per_sm does not show, as no GPU is looked at). */
int tsx_plan_query_tuned(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows, int box_cols,
                         int stages, tsx_variant variant, const tsx_tuning *tuning, tsx_op op, tsx_plan_info *info);

/* tsx_plan_query for an existing plan, including the launch it makes on its
 * device (occupancy-derived CTAs per SM and grid).  Both accept an op with
 * TSX_ACCUMULATE; this one also an op with TSX_ROW_SUMS, for the launch of
 * tsx_reduce_rows (threads, shared memory, grid), with the errors that call
 * would return.  Elsewhere TSX_ROW_SUMS is TSX_ERR_INVALID. */
int tsx_plan_get_info(tsx_plan_t plan, tsx_op op, tsx_plan_info *info);

/* tsx_ewise for callers that may not allocate device memory.  The paper has
 * no counterpart of this entry point: it is an addition for such callers.
 * Some callers cannot call cudaMalloc: a plugin that may only use the memory
 * its host engine hands it, a framework whose pooling allocator has reserved
 * the device memory, a latency-critical loop that cannot afford the device
 * synchronisation cudaMalloc / cudaFree may cause.  tsx_plan_create
 * allocates a device status word, so this one call does the whole job
 * without a plan and allocates nothing, host or device.
 *
 * It runs the same TMA kernel as tsx_ewise (variant TSX_TMA or
 * TSX_TMA_RANK3 only, else TSX_ERR_INVALID) with the same argument rules and
 * results: `a`..`out` as in tsx_ewise; dtype, shape, box, stages and variant
 * as in tsx_plan_create (TSX_ERR_UNSUPPORTED when no plan would be legal).
 * Tensor maps are encoded on every call.
 *
 * Scratch: the kernel's device status word lives in a file-scope device
 * array of 256 bytes, which every GPU that loads the library holds until the
 * process exits; a call needs 4 bytes of it (the library checks that at
 * compile time, so no call is ever turned away for size).  Device-side waits
 * are bounded by 1 s.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  Every
 * call on a device shares the array: each call clears the status word on
 * `stream` before its kernel, so calls whose work overlaps on the GPU (other
 * streams, or other host threads) race on it and may report each other's
 * status.
 *
 * Returns once the work is queued on `stream`, or an error code for a
 * host-side / launch failure (tsx_last_error() says why).  If `status_out`
 * is not NULL the call also waits for `stream` and stores the device status
 * there (TSX_OK, or TSX_ERR_TIMEOUT if a device-side wait gave up), reading
 * it in stream order (cudaMemcpyAsync on `stream`, then a synchronisation
 * of that stream alone).  *status_out is written only by a call that got as
 * far as its launch (or found the tensor empty). */
int tsx_ewise_noalloc(tsx_dtype dtype, int64_t rows, int64_t cols, int box_rows, int box_cols, int stages,
                      tsx_variant variant, tsx_op op, const void *a, const void *b, const void *c, void *out,
                      tsx_stream_t stream, int *status_out);

#ifdef __cplusplus
}
#endif

#endif /* TSX_H */
