/* tsx_debug.h -- test hook of libtsx: a trace of the circular buffer's
 * schedule on the device.  Nothing here is needed to use the library.
 *
 * The traced kernels record, per CTA, the order in which its producer,
 * compute and store threads pass the steps of the loop structure of nvFuser
 * PR #2833 "Add TMA support for circular buffering pass" ("Loop Structure",
 * "Detailed Pseudo-Code"): the prologue and main-loop loads of each tile,
 * the wait on its stage, its computation, and the stage's release, so that
 * a test can hold the device schedule against a model of that structure.
 *
 * Enabling: tsx_debug_plan_enable_trace(plan, n), 1 <= n <= 2^20.
 * tsx_ewise on such a plan then launches a traced kernel, offered for fp32
 * copy and fp32 add on TSX_TMA and TSX_TMA_RANK3 plans (other ops, dtypes,
 * variants and TSX_ACCUMULATE return TSX_ERR_UNSUPPORTED).  The plan owns a
 * device ring of n events per CTA, cleared before every launch.
 *
 * The header also holds the host-side fault hooks the failure-detection
 * tests use: a tile whose loads the producer announces but never issues, so
 * that a bounded device-side wait runs out and the kernel reports
 * TSX_ERR_TIMEOUT.  No GPU fault is involved: nothing traps, no address is
 * bad, and every wait ends.
 *
 * An event is four uint32 words {seq, kind, k, a | (b << 16)}: seq numbers
 * the CTA's events in the order they happened (a shared-memory counter;
 * every event is counted before the barrier arrival that lets another role
 * act on it), k is the CTA's tile counter (its k-th tile is tile
 * cta + k * grid), and kind is
 *   1 load     the producer is about to issue tile k into stage a;
 *              b = 0 in the prologue, 1 in the main loop
 *   2 reuse    the producer saw stage a's release for tile k (phase parity b)
 *   3 wait     a compute thread saw tile k's stage a full (phase parity b)
 *   4 body     compute thread 0 finished its share of tile k (stage a)
 *   5 store    the store warp is about to store tile k from stage a
 *   6 release  the store warp hands tile k's stage a back to the producer
 * Copy has no compute step (its store waits on the load), so no 3 and 4.
 * Slots after a CTA's last event are zero; events past n are dropped. */
#ifndef TSX_DEBUG_H
#define TSX_DEBUG_H

#include "tsx.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Make the plan's later launches record their schedule (traced kernels),
 * events_per_cta events per CTA; 0 turns tracing off.  Call between launches,
 * with the plan's earlier work finished (the old ring is freed).
 * TSX_ERR_INVALID for a NULL plan or n outside [0, 2^20]. */
int tsx_debug_plan_enable_trace(tsx_plan_t plan, int32_t events_per_cta);

/* Fault hook: in the plan's later launches (tsx_ewise and tsx_reduce_rows),
 * the producer announces tile `tile`'s bytes on its stage's mbarrier but
 * issues none of its loads, so the waits on that stage run out (after the
 * plan's timeout) and the kernel records TSX_ERR_TIMEOUT.  tile < 0 clears
 * the hook.  TSX_ERR_INVALID for a NULL plan. */
int tsx_debug_plan_set_fault_tile(tsx_plan_t plan, int64_t tile);

/* The same fault hook for tsx_ewise_noalloc, which has no plan: its later
 * calls made from the calling host thread skip tile `tile`'s loads (tile < 0
 * clears it) and bound every device-side wait by timeout_ms (<= 0: the
 * default 1000 ms). */
void tsx_debug_noalloc_set_fault(int64_t tile, int32_t timeout_ms);

/* The raw shared-memory image of one staged tile: tile `tile` (row-major
 * tile order) of operand `a` is loaded by the plan's TMA loads into a
 * cleared slot exactly as the elementwise kernel stages it (its box split,
 * each box on its own 1024-byte boundary, the plan's swizzle), and the
 * slot's slot_bytes bytes (tsx_plan_get_info) are copied unchanged to
 * `image`, a 16-byte aligned device buffer.  Bytes no load writes read as
 * zero.  One CTA of one warp, asynchronous on `stream`; a wait that runs out
 * is recorded in the plan's status word (image then all zero).  TMA
 * variants only (else TSX_ERR_UNSUPPORTED); TSX_ERR_INVALID for a NULL
 * argument or a tile outside [0, tiles); TSX_ERR_ALIGN for `a` or `image`
 * below 16-byte alignment. */
int tsx_debug_stage_image(tsx_plan_t plan, const void *a, int64_t tile, void *image, tsx_stream_t stream);

/* Copy the trace of the plan's last traced launch to host memory.
 * events: host buffer of `capacity` uint32 words, filled with [grid][per_cta][4]
 * words (as many as fit).  *grid and *per_cta (if not NULL) receive the
 * launch's CTA count and the ring size n.  Synchronous: waits for the
 * device.  TSX_ERR_INVALID if tracing is not enabled on the plan or it has
 * not launched a traced kernel yet. */
int tsx_debug_trace(tsx_plan_t plan, uint32_t *events, int64_t capacity, int32_t *grid, int32_t *per_cta);

#ifdef __cplusplus
}
#endif

#endif /* TSX_DEBUG_H */
