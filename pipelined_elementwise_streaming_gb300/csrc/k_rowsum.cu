// The row-reduction kernel: row_sums[r] = sum over c of op(a, b, c)[r, c].
//
// The schedule is the inner-persistent reduction of the nvFuser page
// ("Testing Setup", Reduction and InnerPersistent): a persistent CTA owns
// whole row bands (box_rows rows), and streams each band's tiles, left to
// right, through the same S-stage TMA ring as the elementwise kernel, so a
// row never needs a reduction across CTAs.
//
//   warp 0      the producer (as in the elementwise kernel): the CTA's k-th
//               tile is tile (band(k), k mod tiles_c) of its k / tiles_c-th
//               band; stage reuse waits on `empty`.
//   warps 1..   the compute warps.  Row r of a band belongs to compute warp
//               r mod W.  For each tile the warp's lanes take the row's
//               16-byte vectors (lane, lane + 32, ...), apply the op, round
//               it into the element type and add the elements into an fp32
//               lane sum in order; a fixed butterfly of shuffles adds the 32
//               lane sums; the tile's row sum is added to the row's fp32
//               accumulator in shared memory; after the band's last tile
//               the accumulator is the row's result.  Every warp then
//               releases the stage (`empty`, one arrival per warp).
//
// The order of additions is fixed by the shapes alone, so results repeat
// bit for bit from run to run.  Columns past the end of the tensor (zero
// filled, or stale when a whole box lies outside) are skipped: the column
// of a staged vector is found through the swizzle inverse.

#include "tsx_tma_common.cuh"

namespace tsx {
namespace {

using namespace dev;

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Add the elements of one 16-byte vector of op results to `part`, in order.
template <int DT>
__device__ __forceinline__ void add_vec(float& part, const uint4& r)
{
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (DT == TSX_F32) {
            part += __uint_as_float(w[k]);
        } else if constexpr (DT == TSX_F16) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
            part += f.x;
            part += f.y;
        } else {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            part += f.x;
            part += f.y;
        }
    }
}

// The op applied to one row of a staged tile, summed: this lane's share of
// the row's in-bounds 16-byte vectors, then the warp total.
template <int DT, int OP>
__device__ __forceinline__ float row_of_tile(const TmaArgs& p, const uint8_t* stage, const TileBoxes& tb, int r,
                                             int lane)
{
    constexpr int NIN = op_arity(OP);
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
    const uint32_t inner_bytes = static_cast<uint32_t>(p.inner_elems) * ES;
    const uint32_t per_atom = inner_bytes / 16;
    const uint32_t total = static_cast<uint32_t>(p.atoms) * per_atom;
    const int rc = r / p.rows_per_load;
    const uint32_t rin = static_cast<uint32_t>(r % p.rows_per_load);
    float part = 0.f;
    for (uint32_t j = lane; j < total; j += 32) {
        const uint32_t a = j / per_atom;
        const uint32_t q = j % per_atom;
        const uint32_t box = p.rank3 ? rc * p.load_smem_bytes + a * p.box_bytes
                                     : (rc * p.atoms + a) * p.load_smem_bytes;
        const uint32_t within = rin * inner_bytes + q * 16;
        const uint32_t lo = unswizzle(within, p.swizzle_mask);
        const int64_t col = tb.col0 + static_cast<int64_t>(a) * p.inner_elems + (lo % inner_bytes) / ES;
        if (col >= p.cols)
            continue;
        const uint32_t off = (box + within) / 16;
        const uint4* S = reinterpret_cast<const uint4*>(stage);
        const uint4 va = S[off];
        const uint4 vb = NIN > 1 ? S[p.slot_bytes / 16 + off] : va;
        const uint4 vc = NIN > 2 ? S[2 * (p.slot_bytes / 16) + off] : va;
        add_vec<DT>(part, op_vec16<DT, OP>(va, vb, vc));
    }
    return warp_sum(part);
}

template <int DT, int OP>
__global__ void __launch_bounds__(kMaxThreads)
    tma_rowsum(const __grid_constant__ TmaMaps maps, const TmaArgs p, float* row_sums)
{
    constexpr int NIN = op_arity(OP);
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1);
    uint8_t* const smem = smem_raw + (base - raw);
    const int S = p.stages;
    const uint32_t full = base + static_cast<uint32_t>(S) * p.stage_bytes;
    const uint32_t empty = full + 8u * S;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + (empty + 8u * S - base));
    float* acc = reinterpret_cast<float*>(smem + (empty + 8u * S + 16 - base));   // one per band row

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int compute_warps = blockDim.x / 32 - 1;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int64_t bands = cta < p.tiles_r ? (p.tiles_r - 1 - cta) / G + 1 : 0;
    const int64_t N = bands * p.tiles_c;
    // the CTA's k-th tile: column tile k mod tiles_c of its (k / tiles_c)-th band
    auto tile_of = [&](int64_t k) { return (cta + (k / p.tiles_c) * G) * p.tiles_c + k % p.tiles_c; };
    const bool elected = warp == 0 && elect_one();

    // Pre-prologue.
    if (elected) {
        for (int j = 0; j < NIN; ++j)
            prefetch_tensormap(&maps.m[j]);
        for (int s = 0; s < S; ++s) {
            mbar_init(full + 8u * s, 1);
            mbar_init(empty + 8u * s, static_cast<uint32_t>(compute_warps));
        }
        *abort_flag = 0;
        fence_proxy_async_smem();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------- producer
        if (elected) {
            int64_t issued = 0;
            const int64_t pro = N < S - 1 ? N : S - 1;
            for (; issued < pro; ++issued)
                issue_tile<NIN>(maps, p, base + (issued % S) * p.stage_bytes, full + 8u * (issued % S),
                                tile_of(issued));
            for (; issued < N; ++issued) {
                const int64_t k = issued;
                const uint32_t s = static_cast<uint32_t>(k % S);
                if (k >= S && !wait_or_abort(empty + 8u * s, static_cast<uint32_t>((k / S - 1) & 1), p, abort_flag))
                    break;
                issue_tile<NIN>(maps, p, base + s * p.stage_bytes, full + 8u * s, tile_of(k));
            }
            if (*abort_flag) {
                const int64_t first = issued > S ? issued - S : 0;
                for (int64_t k = first; k < issued; ++k)
                    (void)mbar_wait(full + 8u * (k % S), static_cast<uint32_t>((k / S) & 1), p.timeout_ns);
            }
        }
    } else {
        // ---------------------------------------------- compute warps
        const int cw = warp - 1;
        for (int64_t i = 0; i < N; ++i) {
            const uint32_t s = static_cast<uint32_t>(i % S);
            if (!wait_or_abort(full + 8u * s, static_cast<uint32_t>((i / S) & 1), p, abort_flag))
                break;
            const TileBoxes tb = tile_boxes(p, tile_of(i));
            const bool first = i % p.tiles_c == 0;
            const bool last = i % p.tiles_c == p.tiles_c - 1;
            const uint8_t* stage = smem + static_cast<size_t>(s) * p.stage_bytes;
            for (int r = cw; r < p.box_rows; r += compute_warps) {
                const int64_t row = tb.row0 + r;
                if (row >= p.rows)
                    break;   // the rows after it are past the end too
                const float t = row_of_tile<DT, OP>(p, stage, tb, r, lane);
                if (lane == 0) {
                    const float v = first ? t : acc[r] + t;
                    acc[r] = v;
                    if (last)
                        row_sums[row] = v;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty + 8u * s);
        }
    }

    // Post-epilogue.
    __syncthreads();
    if (elected) {
        for (int s = 0; s < S; ++s) {
            mbar_inval(full + 8u * s);
            mbar_inval(empty + 8u * s);
        }
    }
}

#define TSX_ROW(DT) \
    {(const void*)tma_rowsum<DT, 0>, (const void*)tma_rowsum<DT, 1>, (const void*)tma_rowsum<DT, 2>, \
     (const void*)tma_rowsum<DT, 3>, (const void*)tma_rowsum<DT, 4>, (const void*)tma_rowsum<DT, 5>}
const void* const kKernels[3][6] = {TSX_ROW(TSX_F16), TSX_ROW(TSX_BF16), TSX_ROW(TSX_F32)};
#undef TSX_ROW

}  // namespace

const void* rowsum_kernel(int dtype, int op) { return kKernels[dtype][op]; }

cudaError_t launch_rowsum(int dtype, int op, int grid, int threads, size_t smem, cudaStream_t stream,
                          const CUtensorMap* maps, const TmaArgs& args, float* row_sums)
{
    TmaMaps m;
    for (int j = 0; j < 4; ++j)
        m.m[j] = maps[j];
    TmaArgs a = args;
    void* params[] = {&m, &a, &row_sums};
    return cudaLaunchKernel(kKernels[dtype][op], dim3(grid), dim3(threads), params, smem, stream);
}

}  // namespace tsx
