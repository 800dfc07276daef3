// Internal declarations shared by the host planner, the C ABI and the
// kernels of libtsx.  Not part of the public interface (include/tsx.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tsx.h"

#ifdef __CUDACC__
#define TSX_HD __host__ __device__
#else
#define TSX_HD
#endif

namespace tsx {

constexpr int kMaxStages = 16;
constexpr int kMaxThreads = 1024;
// CTA threads of the mixed variant's kernel (its compute threads hold b in
// registers one tile ahead)
constexpr int kMixedMaxThreads = 640;
// Register caps of the TMA elementwise kernels: every thread count up to
// kMaxThreads (kMixedMaxThreads) still fits the SM's 64 K registers.
constexpr int kMaxRegs = 56;
constexpr int kMixedMaxRegs = 96;
static_assert(kMaxRegs * kMaxThreads <= 65536 && kMixedMaxRegs * kMixedMaxThreads <= 65536, "register caps");
constexpr int kSmemAlign = 1024;       // 128-B swizzle pattern period
constexpr int kBoxMax = 256;           // per TMA box dimension
constexpr int kSwizzleAtom = 128;      // bytes
constexpr int kMaxDynSmem = 232448;    // 227 KiB opt-in per CTA on sm_100 / sm_103
constexpr int kSmemPerSm = 233472;     // 228 KiB of shared memory per SM
constexpr int kSmemPerCtaReserved = 1024;  // the system's share of each resident CTA
constexpr int kMaxStoreWarps = 2;      // TMA: store warps beside the producer warp
// TMA CTAs: the producer warp and the store warps come ahead of the compute warps
TSX_HD constexpr int tma_role_warps(int store_warps) { return 1 + store_warps; }
// per stage: the full mbarrier, two computed ones (one per group of boxes),
// the empty one and the index of the tile the stage holds (the dynamic tile
// order hands it to the consumers)
constexpr int kTmaBarrierBytes = 40;
// Tile counters of the dynamic tile order: a plan keeps this many, one per
// stream it launches on (two 64-bit words each: tiles claimed, CTAs done).
constexpr int kTileCounterSlots = 64;
// The planner takes the dynamic order only for launches with at least this
// many tiles per CTA (GB300: copies of 2 to 4 tiles per CTA were 12-14 %
// slower in it, of 36 or more 10-11 % faster).
constexpr int kDynamicMinTilesPerCta = 16;

TSX_HD constexpr int elem_size(int dtype) { return dtype == TSX_F32 ? 4 : 2; }
TSX_HD constexpr int op_arity(int op) { return op == TSX_FMA ? 3 : (op == TSX_ADD || op == TSX_MUL) ? 2 : 1; }
TSX_HD constexpr bool is_tma_variant(int v)
{
    return v == TSX_TMA || v == TSX_TMA_RANK3 || v == TSX_TMA_MIXED || v == TSX_TMA_PROMOTED;
}
// Operands that go through the TMA ring: all of them, except b for the mixed variant.
TSX_HD constexpr int tma_operands(int variant, int op)
{
    return variant == TSX_TMA_MIXED && op_arity(op) >= 2 ? op_arity(op) - 1 : op_arity(op);
}

// Units (16-byte vectors of a staged slot) per compute thread whose operand
// b the mixed variant loads one tile ahead into registers.
constexpr int kSetUnits = 4;

// Kernel arguments of the TMA circular-buffer kernel.
struct TmaArgs {
    int64_t tiles;          // T: tiles in the tensor
    int64_t tiles_c;        // tiles along a row
    int64_t tiles_r;        // row bands
    int64_t pitch;          // elements between the starts of consecutive rows
    int64_t fault_tile;     // test hook: the producer skips this tile's loads (-1: none)
    int* status;            // device status word (TSX_OK until a wait gives up)
    uint64_t timeout_ns;    // limit of every mbarrier wait
    int store_lag;          // a store warp's tiles between a store's issue and its stage's release
    int store_warps;        // store warp w of W takes the CTA's tiles w, w + W, ...
    int lane0_wait;         // 1: the producer and store warps wait on lane 0 alone
    int promote_shift;      // log2(tensor-map element / element): box x coordinates are in map elements
    int rows, cols;         // tensor extent (< 2^31)
    int box_rows, box_cols;
    int stages;
    int inner_elems;        // innermost box extent
    int atoms;              // boxes side by side along a tile row (rank 2)
    int rows_per_load;
    int row_chunks;         // boxes stacked along the rows
    int rank3;              // 1: one rank-3 box per row chunk covers all atoms
    uint32_t load_smem_bytes;  // shared-memory footprint of one load
    uint32_t slot_bytes;       // one operand's tile
    uint32_t stage_bytes;      // n_in slots
    uint32_t bytes_per_load;   // bytes one box delivers (out-of-bounds part zero-filled)
    uint32_t vec16_per_slot;   // 16-byte units of one slot
    // mixed variant: operand b, read by the compute threads from global memory,
    // and how many of the CTA's tiles ahead of its loads the producer asks
    // for b's boxes in L2
    const void* set_operand;
    int b_prefetch_ahead;
    uint32_t box_bytes;        // rows_per_load * inner bytes: the data part of one load
    int swizzle_mask;          // 7, 3, 1 for the 128/64/32-byte swizzle, 0 for none
    // dynamic tile order (nullptr: static, CTA c takes c, c + G, ...): {tiles
    // claimed beyond the static ones, CTAs finished}, zero at launch; the
    // launch's last CTA zeroes them again
    unsigned long long* tile_counter;
    int64_t static_tiles;   // dynamic order: tiles c, c + G, ... a CTA takes before it claims (>= 1)
    // test hook (traced kernels only): per CTA a ring of trace_cap events of
    // four 32-bit words each
    uint32_t* trace;
    int trace_cap;
};

// Event kinds of the traced kernel (test hook): what happened to tile k of
// the CTA, recorded in the order the CTA's threads counted them.
enum TraceKind {
    kTraceLoad = 1,      // producer: about to issue tile k into stage a; b = 0 prologue, 1 main loop
    kTraceReuse = 2,     // producer: stage a of tile k released (empty phase b completed)
    kTraceWait = 3,      // compute: tile k's stage a full (phase b completed)
    kTraceBody = 4,      // compute: tile k computed (thread 0's share)
    kTraceStore = 5,     // store: tile k's stores about to be issued from stage a
    kTraceRelease = 6,   // store: tile k's stage a handed back to the producer
    kTraceTile = 7,      // producer: the CTA's k-th tile is tile a | b << 16 of the tensor
};

// Kernel arguments of the cp.async and synchronous ablation kernels.
struct CopyArgs {
    int64_t rows, cols;
    int64_t pitch;            // elements between the starts of consecutive rows
    int64_t tiles, tiles_c;
    int box_rows, box_cols;
    int stages;
    int vec_bytes;            // width of one copy: 16, 8 or 4
    uint32_t tile_bytes;      // box_rows * box_cols * element size
    uint32_t slot_bytes;      // tile_bytes rounded up to 16
    uint32_t stage_bytes;
    uint32_t chunks_per_slot; // tile_bytes / vec_bytes
    uint32_t vec16_per_slot;  // slot_bytes / 16
};

// Kernel lookup and launch, one set per variant (k_tma.cu, k_ldgsts.cu,
// k_sync.cu).  `maps` holds the tensor maps of a, b, c and out.
// Instantiations of the TMA kernel: plain, mixed (b by plain loads),
// accumulate (the result reduce-added into out), and traced (a plain kernel
// that also records its schedule; fp32 copy and add only, else NULL).
// maps[0..2] are the TMA-loaded operands in slot order, maps[3] the output.
enum TmaKind { kTmaPlain = 0, kTmaMixed = 1, kTmaAccumulate = 2, kTmaSplit = 3, kTmaTraced = 4, kTmaTracedSplit = 5 };
const void* tma_kernel(int dtype, int op, int kind = kTmaPlain);
cudaError_t launch_tma(int dtype, int op, int kind, int grid, int threads, size_t smem, cudaStream_t stream,
                       const CUtensorMap* maps, const TmaArgs& args);

// Split an op argument into the op and the TSX_ACCUMULATE flag; false if it
// holds anything else.
inline bool split_op(int op_arg, int* op, bool* accumulate)
{
    *accumulate = (op_arg & TSX_ACCUMULATE) != 0;
    *op = op_arg & ~TSX_ACCUMULATE;
    return *op >= TSX_COPY && *op <= TSX_FMA;
}
// The row-reduction kernel (k_rowsum.cu): TMA ring, rows summed in fp32.
// CTA c of G streams tiles [c T / G, (c + 1) T / G) in row-major order, so a
// row band may be cut between consecutive CTAs.  Each CTA's share of a cut
// band is written to `piece` and the last CTA to count a row in `arrivals`
// adds the row's shares in CTA order.
struct RowsumScratch {
    float* piece;           // [tiles_r][pieces][box_rows] row totals of each CTA's share of a band
    uint32_t* arrivals;     // [tiles_r * box_rows] arrivals per row; zero between launches
    int64_t pieces;         // most CTAs that one band can be cut between
};
const void* rowsum_kernel(int dtype, int op);
cudaError_t launch_rowsum(int dtype, int op, int grid, int threads, size_t smem, cudaStream_t stream,
                          const CUtensorMap* maps, const TmaArgs& args, const RowsumScratch& scratch,
                          float* row_sums);
// Test hook (k_stage_image.cu): one warp stages tile `tile` of maps[0]'s
// operand and copies the slot's raw bytes to `image` (slot_bytes).
size_t stage_image_smem(const TmaArgs& args);
cudaError_t launch_stage_image(const CUtensorMap* maps, const TmaArgs& args, int64_t tile, void* image,
                               cudaStream_t stream);
const void* ldgsts_kernel(int dtype, int op);
cudaError_t launch_ldgsts(int dtype, int op, int grid, int threads, size_t smem, cudaStream_t stream,
                          const void* a, const void* b, const void* c, void* out, const CopyArgs& args);
const void* sync_kernel(int dtype, int op);
cudaError_t launch_sync(int dtype, int op, int grid, int threads, size_t smem, cudaStream_t stream,
                        const void* a, const void* b, const void* c, void* out, const CopyArgs& args);

}  // namespace tsx
