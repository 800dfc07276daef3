// Pieces shared by the cp.async and the synchronous ablation kernels: the
// element a copy chunk stands for, and the elementwise stage that reads the
// staged tile from shared memory and writes the result straight to global
// memory with vector stores of the copy width.
#pragma once

#include "tsx_device.cuh"

namespace tsx {
namespace dev {

// Global element (row, col) of the tile byte offset `byte` (row-major tile
// of box_cols elements per row, origin row0, col0).
template <int ES>
__device__ __forceinline__ void chunk_position(const CopyArgs& p, int64_t row0, int64_t col0, uint32_t byte,
                                               int64_t& row, int64_t& col)
{
    const uint32_t e = byte / ES;
    row = row0 + e / p.box_cols;
    col = col0 + e % p.box_cols;
}

__device__ __forceinline__ void store_piece(char* dst, const uint4& r, int piece, int vec_bytes)
{
    if (vec_bytes == 16) {
        *reinterpret_cast<uint4*>(dst) = r;
    } else if (vec_bytes == 8) {
        const uint2 v = piece == 0 ? make_uint2(r.x, r.y) : make_uint2(r.z, r.w);
        *reinterpret_cast<uint2*>(dst) = v;
    } else {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
        *reinterpret_cast<uint32_t*>(dst) = w[piece];
    }
}

// The elementwise stage over one staged tile (operand slots at `stage`):
// 16-byte vectors (f * threads + tid), op applied, result stored to global
// in pieces of the copy width; out-of-bounds pieces are skipped.
template <int DT, int OP>
__device__ __forceinline__ void ewise_tile_to_global(const CopyArgs& p, const uint8_t* stage, void* out,
                                                     int64_t row0, int64_t col0)
{
    constexpr int NIN = op_arity(OP);
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
    const uint4* A = reinterpret_cast<const uint4*>(stage);
    const uint4* B = A + p.slot_bytes / 16;
    const uint4* C = A + 2 * (p.slot_bytes / 16);
    const int pieces = 16 / p.vec_bytes;
    for (uint32_t u = threadIdx.x; u < p.vec16_per_slot; u += blockDim.x) {
        const uint4 va = A[u];
        const uint4 vb = NIN > 1 ? B[u] : va;
        const uint4 vc = NIN > 2 ? C[u] : va;
        const uint4 r = op_vec16<DT, OP>(va, vb, vc);
        for (int piece = 0; piece < pieces; ++piece) {
            const uint32_t byte = u * 16 + piece * p.vec_bytes;
            if (byte >= p.tile_bytes)
                break;
            int64_t row, col;
            chunk_position<ES>(p, row0, col0, byte, row, col);
            if (row < p.rows && col < p.cols)
                store_piece(static_cast<char*>(out) + (row * p.pitch + col) * ES, r, piece, p.vec_bytes);
        }
    }
}

}  // namespace dev
}  // namespace tsx
