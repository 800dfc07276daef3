// Pieces of the TMA circular-buffer kernels shared by the elementwise
// kernel (k_tma.cu) and the row-reduction kernel (k_rowsum.cu): the tensor
// maps, which boxes of a tile touch the tensor, cursors over tiles and
// stages, the producer warp's issue of a tile, the swizzle inverse and the
// bounded mbarrier wait.
#pragma once

#include "tsx_device.cuh"

namespace tsx {
namespace dev {

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

// The boxes of the tile in row band `band`, column tile `ct`.  Only an edge
// tile needs the divisions.
__device__ __forceinline__ TileBoxes boxes_at(const TmaArgs& p, int64_t band, int64_t ct)
{
    TileBoxes b;
    b.row0 = static_cast<int>(band * p.box_rows);
    b.col0 = static_cast<int>(ct * p.box_cols);
    b.chunks = p.row_chunks;
    b.atoms = p.rank3 ? 1 : p.atoms;
    if (b.row0 + p.box_rows > p.rows) {
        const int chunks_in = (p.rows - b.row0 + p.rows_per_load - 1) / p.rows_per_load;
        b.chunks = chunks_in < b.chunks ? chunks_in : b.chunks;
    }
    if (!p.rank3 && b.col0 + p.box_cols > p.cols) {
        const int atoms_in = (p.cols - b.col0 + p.inner_elems - 1) / p.inner_elems;
        b.atoms = atoms_in < b.atoms ? atoms_in : b.atoms;
    }
    return b;
}

// Walks the tiles t0, t0 + step, t0 + 2 step, ... in (row band, column tile)
// form without a division per step.
struct TileCursor {
    int64_t band, ct, step_r, step_c;
    __device__ __forceinline__ TileCursor(const TmaArgs& p, int64_t t0, int64_t step)
    {
        band = t0 / p.tiles_c;
        ct = t0 - band * p.tiles_c;
        step_r = step / p.tiles_c;
        step_c = step - step_r * p.tiles_c;
    }
    __device__ __forceinline__ void next(const TmaArgs& p)
    {
        ct += step_c;
        band += step_r;
        if (ct >= p.tiles_c) {
            ct -= p.tiles_c;
            ++band;
        }
    }
    __device__ __forceinline__ int64_t tile(const TmaArgs& p) const { return band * p.tiles_c + ct; }
    // Move to tile t (the step stays).
    __device__ __forceinline__ void seek(const TmaArgs& p, int64_t t)
    {
        if (p.tiles <= 0x7fffffff) {
            const uint32_t q = static_cast<uint32_t>(t) / static_cast<uint32_t>(p.tiles_c);
            band = q;
            ct = t - static_cast<int64_t>(q) * p.tiles_c;
        } else {
            band = t / p.tiles_c;
            ct = t - band * p.tiles_c;
        }
    }
};

// Stage s = k mod S and parity (k / S) mod 2 of a tile counter k.
struct StageCursor {
    uint32_t s = 0, phase = 0;
    __device__ __forceinline__ void next(int S)
    {
        if (++s == static_cast<uint32_t>(S)) {
            s = 0;
            phase ^= 1;
        }
    }
    // The cursor of tile counter k, and a step of w tiles (w < 2 S).
    __device__ __forceinline__ static StageCursor at(int64_t k, int S)
    {
        StageCursor c;
        c.s = static_cast<uint32_t>(k % S);
        c.phase = static_cast<uint32_t>((k / S) & 1);
        return c;
    }
    __device__ __forceinline__ void advance(int w, int S)
    {
        s += static_cast<uint32_t>(w);
        while (s >= static_cast<uint32_t>(S)) {
            s -= static_cast<uint32_t>(S);
            phase ^= 1;
        }
    }
};

// One box of a full tile's TMA loads (operand slot j) or stores: where it
// sits in the stage, its tensor map and its coordinate offsets from the
// tile's origin.  Boxes are numbered operand by operand, row chunk by row
// chunk, atom by atom, as they sit in the stage.
struct BoxRef {
    const CUtensorMap* map;
    uint32_t off;   // bytes from the start of the stage
    int r, a;       // row chunk, atom (0 for rank 3)
    int dx, dy;     // coordinate offsets (x in tensor-map elements)
};

__device__ __forceinline__ BoxRef box_ref(const TmaMaps& maps, const TmaArgs& p, int L, int first_map)
{
    const int per_op = p.rank3 ? p.row_chunks : p.row_chunks * p.atoms;
    const int j = L / per_op;
    const int rem = L - j * per_op;
    BoxRef x;
    x.map = &maps.m[first_map + j];
    x.off = static_cast<uint32_t>(j) * p.slot_bytes + static_cast<uint32_t>(rem) * p.load_smem_bytes;
    x.r = p.rank3 ? rem : rem / p.atoms;
    x.a = p.rank3 ? 0 : rem - x.r * p.atoms;
    x.dx = x.a * (p.inner_elems >> p.promote_shift);
    x.dy = x.r * p.rows_per_load;
    return x;
}

// Whether box x of a full tile touches the tensor in a tile with boxes b.
__device__ __forceinline__ bool box_in(const BoxRef& x, const TileBoxes& b) { return x.r < b.chunks && x.a < b.atoms; }

// Load box x of the tile at origin b (column tile ct) into the stage at
// shared address `stage`, completing on `bar`.
__device__ __forceinline__ void load_box(const TmaArgs& p, const BoxRef& x, const TileBoxes& b, int64_t ct,
                                         uint32_t stage, uint32_t bar)
{
    const int y = b.row0 + x.dy;
    if (p.rank3)
        tma_load_3d(stage + x.off, x.map, 0, y, static_cast<int>(ct * p.atoms), bar);
    else
        tma_load_2d(stage + x.off, x.map, (b.col0 >> p.promote_shift) + x.dx, y, bar);
}

// The producer warp's issue of one tile: lane 0 arrives on `bar` with
// expect_tx = the bytes of every load the tile issues, then each lane issues
// the loads numbered lane, lane + 32, ... (`mine` is the lane's first one,
// precomputed; n_loads those of a full tile).  The loads of one tile go out
// from one warp instruction rather than one thread's loop.
template <int NIN>
__device__ __forceinline__ void issue_tile_lanes(const TmaMaps& maps, const TmaArgs& p, const TileCursor& tc,
                                                 const BoxRef& mine, int n_loads, uint32_t stage, uint32_t bar)
{
    const int lane = static_cast<int>(threadIdx.x & 31);
    const TileBoxes b = boxes_at(p, tc.band, tc.ct);
    if (lane == 0)
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(NIN * b.chunks * b.atoms) * p.bytes_per_load);
    __syncwarp();
    if (tc.tile(p) == p.fault_tile)
        return;   // test hook: the announced bytes never arrive
    if (lane < n_loads && box_in(mine, b))
        load_box(p, mine, b, tc.ct, stage, bar);
    for (int L = lane + 32; L < n_loads; L += 32) {
        const BoxRef x = box_ref(maps, p, L, 0);
        if (box_in(x, b))
            load_box(p, x, b, tc.ct, stage, bar);
    }
}


// Offset inside one TMA box in shared memory -> offset in the box's
// row-major image.  The 128-, 64- and 32-byte swizzles exchange the 16-byte
// chunks of a 128-byte line by XOR-ing the chunk index (address bits 4..6)
// with address bits 7..9 (as many bits as the mode has), for boxes that
// start on a 1024-byte boundary, as ours do; the map is its own inverse.
__device__ __forceinline__ uint32_t unswizzle(uint32_t off, int mask)
{
    return off ^ (((off >> 7) & static_cast<uint32_t>(mask)) << 4);
}

// Bounded wait that also gives up when the CTA's abort flag is raised.  A
// wait that runs out of time raises the flag and records the timeout.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const TmaArgs& p,
                                              volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int k = 0; k < 16; ++k)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            atomicCAS(p.status, TSX_OK, TSX_ERR_TIMEOUT);
            return false;
        }
    }
}

// A wait of the producer or store warp, with one answer for the whole warp:
// every lane waits on the barrier itself, or (lane0) lane 0 waits and the
// others take its answer.  Which is faster depends on the launch (measured
// on GB300; the planner chooses, see store_schedule in plan.cpp).
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, const TmaArgs& p, volatile int* abort_flag,
                                          bool lane0)
{
    if (!lane0)
        return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p, abort_flag));
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = wait_or_abort(bar, parity, p, abort_flag);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

}  // namespace dev
}  // namespace tsx
