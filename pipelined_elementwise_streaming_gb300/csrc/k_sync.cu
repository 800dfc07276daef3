// The synchronous staged elementwise kernel: an ablation with one stage and
// no asynchronous copy.  Each thread loads its chunks q = f * threads + tid
// of a tile with plain vector loads of the copy width and stores them to
// shared memory; after a CTA barrier the elementwise stage runs and writes
// the result to global; a second barrier frees the stage for the next tile
// (the pattern of the TVM docs "elementwise -> smem" demonstration program:
// copy global -> shared, op in shared memory, copy shared -> global).

#include "tsx_copy_common.cuh"

namespace tsx {
namespace {

using namespace dev;

__device__ __forceinline__ void load_piece(uint8_t* dst, const char* src, int vec_bytes, bool in)
{
    if (vec_bytes == 16)
        *reinterpret_cast<uint4*>(dst) = in ? *reinterpret_cast<const uint4*>(src) : make_uint4(0, 0, 0, 0);
    else if (vec_bytes == 8)
        *reinterpret_cast<uint2*>(dst) = in ? *reinterpret_cast<const uint2*>(src) : make_uint2(0, 0);
    else
        *reinterpret_cast<uint32_t*>(dst) = in ? *reinterpret_cast<const uint32_t*>(src) : 0u;
}

template <int DT, int OP>
__global__ void __launch_bounds__(kMaxThreads)
    sync_ewise(const void* a, const void* b, const void* c, void* out, const CopyArgs p)
{
    constexpr int NIN = op_arity(OP);
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
    extern __shared__ __align__(16) uint8_t smem[];
    const void* const src[3] = {a, b, c};
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int64_t N = cta < p.tiles ? (p.tiles - 1 - cta) / G + 1 : 0;

    for (int64_t k = 0; k < N; ++k) {
        const int64_t t = cta + k * G;
        const int64_t row0 = (t / p.tiles_c) * p.box_rows;
        const int64_t col0 = (t % p.tiles_c) * p.box_cols;
#pragma unroll
        for (int j = 0; j < NIN; ++j) {
            const char* g = static_cast<const char*>(src[j]);
            uint8_t* slot = smem + j * p.slot_bytes;
            for (uint32_t q = threadIdx.x; q < p.chunks_per_slot; q += blockDim.x) {
                int64_t row, col;
                chunk_position<ES>(p, row0, col0, q * p.vec_bytes, row, col);
                const bool in = row < p.rows && col < p.cols;
                load_piece(slot + q * p.vec_bytes, in ? g + (row * p.pitch + col) * ES : g, p.vec_bytes, in);
            }
        }
        __syncthreads();
        ewise_tile_to_global<DT, OP>(p, smem, out, row0, col0);
        __syncthreads();
    }
}

#define TSX_ROW(DT) \
    {(const void*)sync_ewise<DT, 0>, (const void*)sync_ewise<DT, 1>, (const void*)sync_ewise<DT, 2>, \
     (const void*)sync_ewise<DT, 3>, (const void*)sync_ewise<DT, 4>, (const void*)sync_ewise<DT, 5>}
const void* const kKernels[3][6] = {TSX_ROW(TSX_F16), TSX_ROW(TSX_BF16), TSX_ROW(TSX_F32)};
#undef TSX_ROW

}  // namespace

const void* sync_kernel(int dtype, int op) { return kKernels[dtype][op]; }

cudaError_t launch_sync(int dtype, int op, int grid, int threads, size_t smem, cudaStream_t stream,
                        const void* a, const void* b, const void* c, void* out, const CopyArgs& args)
{
    CopyArgs p = args;
    void* params[] = {&a, &b, &c, &out, &p};
    return cudaLaunchKernel(kKernels[dtype][op], dim3(grid), dim3(threads), params, smem, stream);
}

}  // namespace tsx
