// The TMA circular-buffer elementwise kernel.
//
// A persistent CTA c of G takes tiles c, c + G, c + 2G, ... (row-major tile
// order) and streams them through S stage buffers in shared memory.  Each
// stage has one mbarrier, initialised with an arrival count of 1: the
// elected producer lane of warp 0 arrives once with expect_tx = the bytes of
// all the stage's loads, then issues the loads; the TMA unit completes the
// phase when the bytes have landed (TVM docs "copy_async -> tma",
// "Demonstration program"; nvFuser PR #2833 "Add TMA support for circular
// buffering pass", "Lowering Details").
//
// The loop structure is the one of the nvFuser page ("Loop Structure",
// "Detailed Pseudo-Code"): a pre-prologue that initialises every stage's
// barrier, a prologue that issues the loads of the first S - 1 tiles, a main
// loop whose iteration i issues the loads of tile i + S - 1 into stage
// (i + S - 1) mod S and then waits on tile i in stage i mod S with parity
// (i / S) mod 2, an epilogue that only waits, and a post-epilogue that
// invalidates the barriers.
//
// The body of an iteration is the shared-memory elementwise stage (TVM docs
// "elementwise -> smem"): every thread takes 16-byte vectors (f * threads +
// tid) of each operand's slot, applies the op, and writes the result over
// operand a's slot.  The tile then goes back to global with a TMA store from
// that slot.  Stage reuse (write after read) is guarded twice: a CTA barrier
// after the body, and, before the producer refills a stage, a wait until the
// bulk store that read it has finished reading shared memory.
//
// Every mbarrier wait is bounded in time.  If one gives up, the whole CTA
// leaves the loop together (the decision is a CTA-wide OR), the producer
// records TSX_ERR_TIMEOUT in the status word, waits (again bounded) for the
// loads it still has in flight and for its stores, and the CTA exits.

#include "tsx_device.cuh"

namespace tsx {
namespace {

using namespace dev;

struct TmaMaps {
    CUtensorMap m[4];   // a, b, c, out
};

// Origin of tile t and how many of its boxes touch the tensor: boxes that
// lie wholly past the last row or column (a ragged edge tile) are neither
// loaded nor stored.  A box that is partly outside is loaded in full (the
// outside part reads as zero) and clipped on store.
struct TileBoxes {
    int row0, col0;
    int chunks;   // row chunks with at least one row inside
    int atoms;    // innermost boxes with at least one column inside (1 for rank 3)
};

__device__ __forceinline__ TileBoxes tile_boxes(const TmaArgs& p, int64_t t)
{
    TileBoxes b;
    b.row0 = static_cast<int>((t / p.tiles_c) * p.box_rows);
    b.col0 = static_cast<int>((t % p.tiles_c) * p.box_cols);
    const int chunks_in = (p.rows - b.row0 + p.rows_per_load - 1) / p.rows_per_load;
    b.chunks = chunks_in < p.row_chunks ? chunks_in : p.row_chunks;
    if (p.rank3) {
        b.atoms = 1;
    } else {
        const int atoms_in = (p.cols - b.col0 + p.inner_elems - 1) / p.inner_elems;
        b.atoms = atoms_in < p.atoms ? atoms_in : p.atoms;
    }
    return b;
}

// expect_tx (the bytes of every load this tile issues), then the loads of
// tile t into the stage at shared address `stage` (producer lane only).
template <int NIN>
__device__ __forceinline__ void issue_tile(const TmaMaps& maps, const TmaArgs& p, uint32_t stage, uint32_t bar,
                                           int64_t t)
{
    const TileBoxes b = tile_boxes(p, t);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(NIN * b.chunks * b.atoms) * p.bytes_per_load);
    if (t == p.fault_tile)
        return;   // test hook: the announced bytes never arrive
#pragma unroll
    for (int j = 0; j < NIN; ++j) {
        const uint32_t slot = stage + j * p.slot_bytes;
        for (int r = 0; r < b.chunks; ++r) {
            const int y = b.row0 + r * p.rows_per_load;
            if (p.rank3) {
                tma_load_3d(slot + r * p.load_smem_bytes, &maps.m[j], 0, y, b.col0 / p.inner_elems, bar);
            } else {
                for (int a = 0; a < b.atoms; ++a)
                    tma_load_2d(slot + (r * p.atoms + a) * p.load_smem_bytes, &maps.m[j],
                                b.col0 + a * p.inner_elems, y, bar);
            }
        }
    }
}

// TMA store of tile t from the slot at shared address `slot` (producer lane).
__device__ __forceinline__ void store_tile(const TmaMaps& maps, const TmaArgs& p, uint32_t slot, int64_t t)
{
    const TileBoxes b = tile_boxes(p, t);
    for (int r = 0; r < b.chunks; ++r) {
        const int y = b.row0 + r * p.rows_per_load;
        if (p.rank3) {
            tma_store_3d(&maps.m[3], slot + r * p.load_smem_bytes, 0, y, b.col0 / p.inner_elems);
        } else {
            for (int a = 0; a < b.atoms; ++a)
                tma_store_2d(&maps.m[3], slot + (r * p.atoms + a) * p.load_smem_bytes, b.col0 + a * p.inner_elems,
                             y);
        }
    }
    bulk_commit();
}

// Wait on tile i (the CTA's i-th), apply the op in shared memory and store
// the result.  Returns false on every thread if any thread's wait gave up.
template <int DT, int OP, int NIN>
__device__ __forceinline__ bool consume_tile(const TmaMaps& maps, const TmaArgs& p, uint8_t* smem, uint32_t base,
                                             uint32_t bars, int64_t i, int64_t t, bool producer)
{
    const int S = p.stages;
    const int s = static_cast<int>(i % S);
    const uint32_t parity = static_cast<uint32_t>((i / S) & 1);
    const bool ok = mbar_wait(bars + 8u * s, parity, p.timeout_ns);

    if constexpr (OP != TSX_COPY) {
        if (ok) {
            uint4* A = reinterpret_cast<uint4*>(smem + static_cast<size_t>(s) * p.stage_bytes);
            const uint4* B = A + p.slot_bytes / 16;
            const uint4* C = A + 2 * (p.slot_bytes / 16);
            for (uint32_t u = threadIdx.x; u < p.vec16_per_slot; u += blockDim.x) {
                const uint4 va = A[u];
                const uint4 vb = NIN > 1 ? B[u] : va;
                const uint4 vc = NIN > 2 ? C[u] : va;
                A[u] = op_vec16<DT, OP>(va, vb, vc);
            }
            // make this thread's generic-proxy writes visible to the TMA store
            fence_proxy_async_smem();
        }
    }
    if (__syncthreads_or(!ok))
        return false;
    if (producer)
        store_tile(maps, p, base + s * p.stage_bytes, t);
    return true;
}

template <int DT, int OP>
__global__ void __launch_bounds__(kMaxThreads) tma_ewise(const __grid_constant__ TmaMaps maps, const TmaArgs p)
{
    constexpr int NIN = op_arity(OP);
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1);
    uint8_t* const smem = smem_raw + (base - raw);
    const int S = p.stages;
    const uint32_t bars = base + static_cast<uint32_t>(S) * p.stage_bytes;

    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int64_t N = cta < p.tiles ? (p.tiles - 1 - cta) / G + 1 : 0;
    const bool producer = threadIdx.x < 32 && elect_one();

    // Pre-prologue: one barrier per stage, a single arrival each.
    if (producer) {
        for (int s = 0; s < S; ++s)
            mbar_init(bars + 8u * s, 1);
        fence_proxy_async_smem();
    }
    __syncthreads();

    // Prologue: loads of the first S - 1 tiles.
    int64_t issued = 0;
    if (producer) {
        const int64_t pro = N < S - 1 ? N : S - 1;
        for (; issued < pro; ++issued)
            issue_tile<NIN>(maps, p, base + (issued % S) * p.stage_bytes, bars + 8u * (issued % S),
                            cta + issued * G);
    }

    // Main loop: issue tile i + S - 1, consume tile i.
    const int64_t main_iters = N > S - 1 ? N - (S - 1) : 0;
    int64_t i = 0;
    bool failed = false;
    for (; i < main_iters; ++i) {
        if (producer) {
            const int64_t k = i + S - 1;
            // stage k mod S last held tile i - 1: its store must be done reading
            bulk_wait_read_all();
            issue_tile<NIN>(maps, p, base + (k % S) * p.stage_bytes, bars + 8u * (k % S), cta + k * G);
            issued = k + 1;
        }
        if (!consume_tile<DT, OP, NIN>(maps, p, smem, base, bars, i, cta + i * G, producer)) {
            failed = true;
            break;
        }
    }
    // Epilogue: consume the remaining tiles.
    if (!failed) {
        for (; i < N; ++i) {
            if (!consume_tile<DT, OP, NIN>(maps, p, smem, base, bars, i, cta + i * G, producer)) {
                failed = true;
                break;
            }
        }
    }

    // Post-epilogue.
    if (producer) {
        if (failed) {
            atomicCAS(p.status, TSX_OK, TSX_ERR_TIMEOUT);
            // let loads still in flight land before the CTA's shared memory goes away
            for (int64_t k = i; k < issued; ++k)
                (void)mbar_wait(bars + 8u * (k % S), static_cast<uint32_t>((k / S) & 1), p.timeout_ns);
        }
        bulk_wait_all();
    }
    __syncthreads();
    if (producer) {
        for (int s = 0; s < S; ++s)
            mbar_inval(bars + 8u * s);
    }
}

#define TSX_ROW(DT) \
    {(const void*)tma_ewise<DT, 0>, (const void*)tma_ewise<DT, 1>, (const void*)tma_ewise<DT, 2>, \
     (const void*)tma_ewise<DT, 3>, (const void*)tma_ewise<DT, 4>, (const void*)tma_ewise<DT, 5>}
const void* const kKernels[3][6] = {TSX_ROW(TSX_F16), TSX_ROW(TSX_BF16), TSX_ROW(TSX_F32)};
#undef TSX_ROW

}  // namespace

const void* tma_kernel(int dtype, int op) { return kKernels[dtype][op]; }

cudaError_t launch_tma(int dtype, int op, int grid, int threads, size_t smem, cudaStream_t stream,
                       const CUtensorMap* maps, const TmaArgs& args)
{
    TmaMaps m;
    for (int j = 0; j < 4; ++j)
        m.m[j] = maps[j];
    TmaArgs a = args;
    void* params[] = {&m, &a};
    return cudaLaunchKernel(kKernels[dtype][op], dim3(grid), dim3(threads), params, smem, stream);
}

}  // namespace tsx
