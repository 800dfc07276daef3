// Pieces of the TMA circular-buffer kernels shared by the elementwise
// kernel (k_tma.cu) and the row-reduction kernel (k_rowsum.cu): the tensor
// maps, which boxes of a tile touch the tensor, the producer's issue of a
// tile, the swizzle inverse and the bounded mbarrier wait.
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
// tile t into the stage at shared address `stage`.
template <int NIN>
__device__ __forceinline__ void issue_tile(const TmaMaps& maps, const TmaArgs& p, uint32_t stage, uint32_t bar,
                                           int64_t t)
{
    const TileBoxes b = tile_boxes(p, t);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(NIN * b.chunks * b.atoms) * p.bytes_per_load);
    if (t == p.fault_tile)
        return;   // test hook: the announced bytes never arrive
    // box x coordinates in tensor-map elements (wider when promoted)
    const int x0 = b.col0 >> p.promote_shift;
    const int dx = p.inner_elems >> p.promote_shift;
#pragma unroll
    for (int j = 0; j < NIN; ++j) {
        const uint32_t slot = stage + j * p.slot_bytes;
        for (int r = 0; r < b.chunks; ++r) {
            const int y = b.row0 + r * p.rows_per_load;
            if (p.rank3) {
                tma_load_3d(slot + r * p.load_smem_bytes, &maps.m[j], 0, y, b.col0 / p.inner_elems, bar);
            } else {
                for (int a = 0; a < b.atoms; ++a)
                    tma_load_2d(slot + (r * p.atoms + a) * p.load_smem_bytes, &maps.m[j], x0 + a * dx, y, bar);
            }
        }
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
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            atomicCAS(p.status, TSX_OK, TSX_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

}  // namespace dev
}  // namespace tsx
