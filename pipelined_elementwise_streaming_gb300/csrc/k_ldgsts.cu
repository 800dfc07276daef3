// The cp.async (LDGSTS) circular-buffer elementwise kernel: an ablation of
// the TMA path with the same tiles, stages and loop trip counts.
//
// Each thread copies its share of a tile global -> shared with cp.async:
// chunk q = f * threads + tid of `vec_bytes` (16, 8 or 4) bytes, the
// [outer, threads, vec] partition of TVM docs "copy_async -> ldgsts"
// ("Algorithm" steps 1-2).  Out-of-bounds chunks of a ragged tile copy zero
// source bytes, which fills zeros.  One commit group per tile; before tile i
// is consumed each thread waits until at most min(N, i + S - 1) - i - 1 of
// its groups are pending (S - 2 in the main loop, N - 1 - i in the
// epilogue), then a CTA barrier publishes every thread's copies.  The same
// barrier marks stage (i - 1) mod S free, so the main loop's refill of it
// (tile i + S - 1) comes right after.  cp.async has no shared -> global form,
// so results go out with vector stores.  S = 1 issues, waits and consumes
// one tile at a time.

#include "tsx_copy_common.cuh"

namespace tsx {
namespace {

using namespace dev;

template <int DT, int OP>
__device__ __forceinline__ void issue_tile_cp_async(const CopyArgs& p, uint8_t* stage, const void* const* src,
                                                    int64_t row0, int64_t col0)
{
    constexpr int NIN = op_arity(OP);
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
#pragma unroll
    for (int j = 0; j < NIN; ++j) {
        const char* g = static_cast<const char*>(src[j]);
        const uint32_t slot = smem_addr(stage + j * p.slot_bytes);
        for (uint32_t q = threadIdx.x; q < p.chunks_per_slot; q += blockDim.x) {
            int64_t row, col;
            chunk_position<ES>(p, row0, col0, q * p.vec_bytes, row, col);
            const bool in = row < p.rows && col < p.cols;
            const char* gp = in ? g + (row * p.pitch + col) * ES : g;
            cp_async(slot + q * p.vec_bytes, gp, p.vec_bytes, in ? p.vec_bytes : 0u);
        }
    }
    cp_async_commit();
}

template <int DT, int OP>
__global__ void __launch_bounds__(kMaxThreads)
    ldgsts_ewise(const void* a, const void* b, const void* c, void* out, const CopyArgs p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const void* const src[3] = {a, b, c};
    const int S = p.stages;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int64_t N = cta < p.tiles ? (p.tiles - 1 - cta) / G + 1 : 0;

    auto origin = [&](int64_t k, int64_t& row0, int64_t& col0) {
        const int64_t t = cta + k * G;
        row0 = (t / p.tiles_c) * p.box_rows;
        col0 = (t % p.tiles_c) * p.box_cols;
    };
    auto issue = [&](int64_t k) {
        int64_t row0, col0;
        origin(k, row0, col0);
        issue_tile_cp_async<DT, OP>(p, smem + (k % S) * p.stage_bytes, src, row0, col0);
    };
    auto consume = [&](int64_t k) {
        int64_t row0, col0;
        origin(k, row0, col0);
        ewise_tile_to_global<DT, OP>(p, smem + (k % S) * p.stage_bytes, out, row0, col0);
    };

    if (S == 1) {
        for (int64_t i = 0; i < N; ++i) {
            issue(i);
            cp_async_wait(0);
            __syncthreads();
            consume(i);
            __syncthreads();
        }
        return;
    }
    // Prologue: the first S - 1 tiles.
    const int64_t pro = N < S - 1 ? N : S - 1;
    for (int64_t k = 0; k < pro; ++k)
        issue(k);
    // Main loop.
    const int64_t main_iters = N > S - 1 ? N - (S - 1) : 0;
    int64_t i = 0;
    for (; i < main_iters; ++i) {
        cp_async_wait(S - 2);
        __syncthreads();
        issue(i + S - 1);
        consume(i);
    }
    // Epilogue.
    for (; i < N; ++i) {
        cp_async_wait(static_cast<int>(N - 1 - i));
        __syncthreads();
        consume(i);
    }
}

#define TSX_ROW(DT) \
    {(const void*)ldgsts_ewise<DT, 0>, (const void*)ldgsts_ewise<DT, 1>, (const void*)ldgsts_ewise<DT, 2>, \
     (const void*)ldgsts_ewise<DT, 3>, (const void*)ldgsts_ewise<DT, 4>, (const void*)ldgsts_ewise<DT, 5>}
const void* const kKernels[3][6] = {TSX_ROW(TSX_F16), TSX_ROW(TSX_BF16), TSX_ROW(TSX_F32)};
#undef TSX_ROW

}  // namespace

const void* ldgsts_kernel(int dtype, int op) { return kKernels[dtype][op]; }

cudaError_t launch_ldgsts(int dtype, int op, int grid, int threads, size_t smem, cudaStream_t stream,
                          const void* a, const void* b, const void* c, void* out, const CopyArgs& args)
{
    CopyArgs p = args;
    void* params[] = {&a, &b, &c, &out, &p};
    return cudaLaunchKernel(kKernels[dtype][op], dim3(grid), dim3(threads), params, smem, stream);
}

}  // namespace tsx
