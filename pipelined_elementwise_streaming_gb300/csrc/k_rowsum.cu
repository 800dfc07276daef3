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
//   warps 1..   the compute warps.  Every tile of a plan lands in shared
//               memory with the same layout, so the 16-byte unit u of a
//               staged slot holds the same (row, column within the tile) in
//               every tile.  Compute thread tid always takes units tid, tid
//               + threads, ...: it applies the op to the unit's vectors,
//               rounds into the element type, adds the elements in order and
//               adds that to the unit's fp32 partial in shared memory (set,
//               on the band's first tile).  Only a band's last, ragged tile
//               needs each unit's column, to leave out the columns past the
//               tensor's end.  Every warp then releases the stage (`empty`,
//               one arrival per warp).  After the band's last tile one
//               thread per row adds the partials of the row's units, box by
//               box in a fixed order, into the row's result.
//
// The order of additions is fixed by the shapes alone, so results repeat
// bit for bit from run to run.  Columns past the end of the tensor (zero
// filled, or stale when a whole box lies outside) are skipped: the column
// of a staged vector is found through the swizzle inverse.

#include "tsx_tma_common.cuh"

namespace tsx {
namespace {

using namespace dev;

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

// The op on the staged vectors of unit u, its elements added in order.
template <int DT, int OP>
__device__ __forceinline__ float unit_sum(const TmaArgs& p, const uint4* S, uint32_t u)
{
    constexpr int NIN = op_arity(OP);
    const uint4 va = S[u];
    const uint4 vb = NIN > 1 ? S[p.slot_bytes / 16 + u] : va;
    const uint4 vc = NIN > 2 ? S[2 * (p.slot_bytes / 16) + u] : va;
    float part = 0.f;
    add_vec<DT>(part, op_vec16<DT, OP>(va, vb, vc));
    return part;
}

// Whether unit u of a staged slot holds columns inside the tensor (a ragged
// tile's padding and the boxes skipped past its end do not).
template <int DT>
__device__ __forceinline__ bool unit_in_columns(const TmaArgs& p, const TileBoxes& tb, uint32_t u)
{
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
    const uint32_t inner_bytes = static_cast<uint32_t>(p.inner_elems) * ES;
    const uint32_t off = u * 16;
    uint32_t load = off / p.load_smem_bytes;
    uint32_t within = off - load * p.load_smem_bytes;
    uint32_t atom;
    if (p.rank3) {
        atom = within / p.box_bytes;
        within -= atom * p.box_bytes;
    } else {
        atom = load % p.atoms;
    }
    if (within >= p.box_bytes || atom >= static_cast<uint32_t>(p.atoms))
        return false;   // padding after a box
    const uint32_t lo = unswizzle(within, p.swizzle_mask);
    const int64_t col = tb.col0 + static_cast<int64_t>(atom) * p.inner_elems + (lo % inner_bytes) / ES;
    return col < p.cols;
}

// Sum of the partials of row r (of the band): its units, box by box.
template <int DT>
__device__ __forceinline__ float row_total(const TmaArgs& p, const float* partial, int r)
{
    constexpr int ES = DT == TSX_F32 ? 4 : 2;
    const uint32_t per_row = static_cast<uint32_t>(p.inner_elems) * ES / 16;   // units of one box row
    const uint32_t rc = static_cast<uint32_t>(r / p.rows_per_load);
    const uint32_t rin = static_cast<uint32_t>(r % p.rows_per_load);
    float v = 0.f;
    for (int a = 0; a < p.atoms; ++a) {
        const uint32_t box = p.rank3 ? rc * p.load_smem_bytes + a * p.box_bytes
                                     : (rc * p.atoms + a) * p.load_smem_bytes;
        const uint32_t first = (box + rin * per_row * 16) / 16;
        for (uint32_t q = 0; q < per_row; ++q)
            v += partial[first + q];
    }
    return v;
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
    // the compute warps' band barriers: partials complete / partials read
    const uint32_t band_done = empty + 8u * S;
    const uint32_t band_free = band_done + 8u;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + (band_free + 8u - base));
    float* partial = reinterpret_cast<float*>(smem + (band_free + 8u + 16 - base));   // one per item

    const int warp = threadIdx.x / 32;
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
        mbar_init(band_done, static_cast<uint32_t>(compute_warps));
        mbar_init(band_free, static_cast<uint32_t>(compute_warps));
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
        const uint32_t tid = threadIdx.x - 32;
        const uint32_t threads = blockDim.x - 32;
        // stage, phase, band and column tile advance with the tile counter
        // (no divisions in the loop)
        uint32_t s = 0, phase = 0, band_parity = 0;
        int64_t band = cta, ct = 0;
        for (int64_t i = 0; i < N; ++i) {
            if (!wait_or_abort(full + 8u * s, phase, p, abort_flag))
                break;
            TileBoxes tb;
            tb.row0 = static_cast<int>(band * p.box_rows);
            tb.col0 = static_cast<int>(ct * p.box_cols);
            tb.chunks = p.row_chunks;
            tb.atoms = p.atoms;
            const bool ragged = tb.col0 + p.box_cols > p.cols;
            const uint4* stage = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(s) * p.stage_bytes);
            if (ct == 0) {
                for (uint32_t u = tid; u < p.vec16_per_slot; u += threads)
                    partial[u] = ragged && !unit_in_columns<DT>(p, tb, u) ? 0.f : unit_sum<DT, OP>(p, stage, u);
            } else {
                for (uint32_t u = tid; u < p.vec16_per_slot; u += threads)
                    partial[u] += ragged && !unit_in_columns<DT>(p, tb, u) ? 0.f : unit_sum<DT, OP>(p, stage, u);
            }
            __syncwarp();
            if ((threadIdx.x & 31) == 0)
                mbar_arrive(empty + 8u * s);
            if (ct == p.tiles_c - 1) {
                // the band is complete once every compute warp has added its
                // last partials; then each row's partials, box by box
                if ((threadIdx.x & 31) == 0)
                    mbar_arrive(band_done);
                if (!wait_or_abort(band_done, band_parity, p, abort_flag))
                    break;
                for (uint32_t r = tid; r < static_cast<uint32_t>(p.box_rows); r += threads) {
                    const int64_t row = tb.row0 + r;
                    if (row >= p.rows)
                        break;
                    row_sums[row] = row_total<DT>(p, partial, static_cast<int>(r));
                }
                // before the next band overwrites the partials
                __syncwarp();
                if ((threadIdx.x & 31) == 0)
                    mbar_arrive(band_free);
                if (!wait_or_abort(band_free, band_parity, p, abort_flag))
                    break;
                band_parity ^= 1;
                band += G;
                ct = 0;
            } else {
                ++ct;
            }
            if (++s == static_cast<uint32_t>(S)) {
                s = 0;
                phase ^= 1;
            }
        }
    }

    // Post-epilogue.
    __syncthreads();
    if (elected) {
        for (int s = 0; s < S; ++s) {
            mbar_inval(full + 8u * s);
            mbar_inval(empty + 8u * s);
        }
        mbar_inval(band_done);
        mbar_inval(band_free);
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
