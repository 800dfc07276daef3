// Host-side plan geometry of libtsx (pure integer logic, see plan.cpp).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "tsx_internal.h"

namespace tsx {

// Launch knobs of a plan, resolved from a tsx_tuning (planner's choices
// filled in).  threads = 0 and ctas_per_sm = 0 leave those to the planner
// and to occupancy.
struct Knobs {
    int threads = 0;
    int ctas_per_sm = 0;
    int store_lag = -1;      // < 0: the planner's
    int store_warps = 0;     // 0: the planner's
    int role_wait = 0;       // 0: the planner's; 1: every lane waits; 2: lane 0 waits
    int b_prefetch = -1;     // < 0: the planner's
    int tile_order = 0;      // 0: the planner's; 1 static; 2 dynamic
    int dynamic_share = 0;   // 0: the planner's; else percent of the tiles claimed dynamically
    int store_split = 0;     // 0: the planner's; 1 one group of boxes; 2 two
    int l2_promotion = 2;    // CUtensorMapL2promotion
    int timeout_ms = 1000;
    bool checked = false;
};

// Everything fixed by (dtype, shape, box, stages, variant, knobs).
struct Geometry {
    int dtype = 0, es = 0, variant = 0, stages = 0;
    int64_t rows = 0, cols = 0;
    int64_t pitch = 0;       // elements between row starts (>= cols)
    int box_rows = 0, box_cols = 0;
    int64_t tiles_r = 0, tiles_c = 0, tiles = 0;
    // TMA split
    int inner_bytes = 0, inner_elems = 0, atoms = 0, row_chunks = 0, rows_per_load = 0;
    int loads_per_operand = 0, bytes_per_load = 0, swizzle_bytes = 0;
    int tma_es = 0;          // element size the tensor map uses (> es when promoted)
    int l2_promotion = 2;    // CUtensorMapL2promotion: 0 none, 1 64 B, 2 128 B, 3 256 B
    uint32_t load_smem_bytes = 0;
    // one operand's tile in shared memory
    uint32_t slot_bytes = 0;
    // copy width of the cp.async / synchronous variants (16-byte aligned bases)
    int copy_vec_bytes = 0;
    Knobs knobs;
};

// What additionally depends on the op (operand count).
struct OpGeometry {
    int op = 0, n_in = 0;
    int n_tma = 0;           // operands loaded through the TMA ring
    uint32_t stage_bytes = 0, tx_bytes = 0, vec16_per_slot = 0;
    size_t smem_bytes = 0;
    int threads = 0;         // threads of the elementwise stage ([outer, threads, vec])
    int block_threads = 0;   // threads of a CTA (TMA: + producer and store warps)
    int vec = 0, outer = 0;
    // TMA: how the store side runs (StoreSchedule)
    int store_warps = 1;     // store warps, taking the CTA's tiles in turn
    int store_lag = 1;       // a store warp's tiles between a store's issue and its stage's release
    bool lane0_wait = false; // the producer and store warps wait on lane 0 alone
    int ctas_cap = 0;        // at most this many CTAs per SM (0: occupancy)
    int b_prefetch_ahead = 0;  // mixed variant: b's L2 prefetch, tiles beyond the producer's loads
    int tile_order = 0;      // TMA: 1 static, 2 dynamic (tiles claimed from a counter)
    int dynamic_share = 0;   // dynamic order: percent of the tiles claimed
    int compute_groups = 1;  // TMA: groups of boxes handed from the compute to the store warps (1, 2)
};

// Dynamic order: the tiles each of `grid` CTAs takes in the static order
// before it claims, so that about dynamic_share percent of the tiles are
// claimed (at least max(1, S - 1)).
int64_t static_tiles_per_cta(const Geometry& g, const OpGeometry& og, int64_t grid);
// Dynamic order: tiles of at least this many bytes have every tile past the
// static prefix claimed; smaller ones only the last quarter.
constexpr uint32_t kDynamicAllTileBytes = 16384;

struct TensorMapArgs {
    int rank = 0;
    int l2_promotion = 2;
    uint64_t dims[5] = {};
    uint64_t strides[4] = {};
    uint32_t box[5] = {};
    int swizzle = 0;   // CUtensorMapSwizzle value
};

int default_threads(const Geometry& g, int op, size_t smem_bytes, uint32_t units, int store_warps);
// The store side of a TMA launch for `op` on geometry g: store warps, lag
// and wait style (the planner's table, unless the knobs force them).
struct StoreSchedule {
    int store_warps, store_lag;
    bool lane0_wait;
};
StoreSchedule store_schedule(const Geometry& g, int op, uint32_t stage_bytes);
// Mixed variant: how many of a CTA's tiles beyond the tile it loads the
// producer prefetches b into L2, for ctas_per_sm resident CTAs.
int mixed_prefetch_ahead(const Geometry& g, int ctas_per_sm);
// Validate a tsx_tuning (NULL: all defaults) into knobs.
int resolve_knobs(const tsx_tuning* t, Knobs* k, std::string* why);
int make_geometry(int dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows, int box_cols, int stages,
                  int variant, const Knobs& knobs, Geometry* g, std::string* why);
// Default knobs.
inline int make_geometry(int dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows, int box_cols,
                         int stages, int variant, Geometry* g, std::string* why)
{
    return make_geometry(dtype, rows, cols, pitch, box_rows, box_cols, stages, variant, Knobs{}, g, why);
}
int make_op_geometry(const Geometry& g, int op, int max_smem, OpGeometry* og, std::string* why);
void tensor_map_args(const Geometry& g, TensorMapArgs* m);
void fill_info(const Geometry& g, const OpGeometry& og, tsx_plan_info* info);
// Kernel arguments of the TMA kernels (elementwise and row sums) for one op:
// the device status word, and the tile whose loads the producer skips (test
// hook; -1 for none).
void fill_tma_args(const Geometry& g, const OpGeometry& og, int* status, int64_t fault_tile, TmaArgs* args);

// Thread-local message behind tsx_last_error (capi.cpp).
void set_last_error(const char* msg);

// Encode the tensor map of base pointer `ptr` for geometry g (capi.cpp).
int encode_tensor_map(const Geometry& g, const void* ptr, CUtensorMap* map);

}  // namespace tsx
