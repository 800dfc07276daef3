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
 * Enabling: env TSX_TRACE = n (1 <= n <= 2^20) when tsx_plan_create runs.
 * tsx_ewise on such a plan then launches a traced kernel, offered for fp32
 * copy and fp32 add on TSX_TMA and TSX_TMA_RANK3 plans (other ops, dtypes,
 * variants and TSX_ACCUMULATE return TSX_ERR_UNSUPPORTED).  The plan owns a
 * device ring of n events per CTA, cleared before every launch.
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

/* Copy the trace of the plan's last traced launch to host memory.
 * events: host buffer of `capacity` uint32 words, filled with [grid][per_cta][4]
 * words (as many as fit).  *grid and *per_cta (if not NULL) receive the
 * launch's CTA count and the ring size n.  Synchronous: waits for the
 * device.  TSX_ERR_INVALID if the plan was not created with TSX_TRACE or has
 * not launched a traced kernel yet. */
int tsx_debug_trace(tsx_plan_t plan, uint32_t *events, int64_t capacity, int32_t *grid, int32_t *per_cta);

#ifdef __cplusplus
}
#endif

#endif /* TSX_DEBUG_H */
