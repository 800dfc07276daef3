// The row-reduction kernel: row_sums[r] = sum over c of op(a, b, c)[r, c].
//
// The schedule is the inner-persistent reduction of the nvFuser page
// ("Testing Setup", Reduction and InnerPersistent): every tile of a row band
// streams through the same S-stage TMA ring as the elementwise kernel and is
// folded into fp32 partials.  The persistent grid splits
// the tiles, taken in row-major order (band after band, left to right), into
// G contiguous ranges of floor(T / G) or ceil(T / G) tiles: CTA c streams
// tiles [c T / G, (c + 1) T / G), so the work is even however few the bands.
//
//   warp 0      the producer (as in the elementwise kernel: one box per
//               lane); stage reuse waits on `empty`.
//   warps 1..   the compute warps.  Every tile of a plan lands in shared
//               memory with the same layout, so the 16-byte unit u of a
//               staged slot holds the same (row, column within the tile) in
//               every tile.  Compute thread tid always takes units tid, tid
//               + threads, ...: it applies the op to the unit's vectors,
//               rounds into the element type and adds the elements in order
//               to the unit's fp32 partial, kept in a register for the
//               thread's first kRegUnits units and in shared memory for any
//               further ones.  Only a band's last, ragged tile needs each
//               unit's column, to leave out the columns past the tensor's
//               end.  Every warp then releases the stage (`empty`, one
//               arrival per warp).  When the CTA's share of a band ends, the
//               register partials go to shared memory and one thread per row
//               adds the partials of the row's units, box by box in a fixed
//               order.
//
// A band the CTA streamed whole gets its row sums written directly.  A band
// cut between CTAs c0 < ... < c1 (consecutive, since the ranges are) has
// each share's row totals stored in the plan's scratch; the thread that
// stores a row's share then counts an arrival on the row, and the one that
// counts the last arrival adds the shares in CTA order into the result
// (the fence-then-count pattern of the CUDA programming guide's memory
// fence example).  No CTA waits on another.
//
// The order of additions is fixed by the shapes and the grid size, both
// fixed per plan, so results repeat bit for bit from run to run.  Columns
// past the end of the tensor (zero filled, or stale when a whole box lies
// outside) are skipped: the column of a staged vector is found through the
// swizzle inverse.

#include "tsx_tma_common.cuh"

namespace tsx {
namespace {

using namespace dev;

// Add the elements of one 16-byte vector of op results to `part`, in order.
// 16-bit elements go in through the mixed-precision add (a 16-bit operand,
// widened exactly, plus an fp32 operand, rounded once in fp32), which takes
// a half of the packed word as it is: the same sum as widening first, in
// half the instructions.
template <int DT>
__device__ __forceinline__ void add_vec(float& part, const uint4& r)
{
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (DT == TSX_F32) {
            part += __uint_as_float(w[k]);
        } else if constexpr (DT == TSX_F16) {
            asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
                "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %0, hi, %0;\n\t}"
                : "+f"(part)
                : "r"(w[k]));
        } else {
            asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
                "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %0, hi, %0;\n\t}"
                : "+f"(part)
                : "r"(w[k]));
        }
    }
}

// The op on the staged vectors of unit u, its elements added in order to `part`.
template <int DT, int OP>
__device__ __forceinline__ void add_unit(float& part, const TmaArgs& p, const uint4* S, uint32_t u)
{
    constexpr int NIN = op_arity(OP);
    const uint4 va = S[u];
    const uint4 vb = NIN > 1 ? S[p.slot_bytes / 16 + u] : va;
    const uint4 vc = NIN > 2 ? S[2 * (p.slot_bytes / 16) + u] : va;
    add_vec<DT>(part, op_vec16<DT, OP, true>(va, vb, vc));
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

// Units of a staged slot whose partials a compute thread keeps in registers
// (units tid, tid + threads, ...); any further units keep theirs in shared
// memory.
constexpr int kRegUnits = 8;

// The CTA whose tile range holds tile x: the largest c with c T / G <= x.
__device__ __forceinline__ int64_t range_owner(int64_t x, int64_t T, int64_t G)
{
    return ((x + 1) * G + T - 1) / T - 1;
}

// One row of a band cut between CTAs c0 .. c0 + shares - 1: store this
// CTA's share v as share j (shares are box_rows floats apart), count it, and
// if it is the row's last arrival add the shares in CTA order into *result.
__device__ __forceinline__ void finish_cut_row(float* share_col, uint32_t* arrivals, int64_t box_rows, int64_t j,
                                               uint32_t shares, float v, float* result)
{
    share_col[j * box_rows] = v;
    __threadfence();
    if (atomicInc(arrivals, shares - 1) == shares - 1) {
        __threadfence();
        float t = 0.f;
        for (uint32_t k = 0; k < shares; ++k)
            t += __ldcg(share_col + k * box_rows);
        *result = t;
    }
}

template <int DT, int OP>
__global__ void __launch_bounds__(kMaxThreads)
    tma_rowsum(const __grid_constant__ TmaMaps maps, const TmaArgs p, const RowsumScratch sc, float* row_sums)
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
    // the CTA's tiles: lo, lo + 1, ..., lo + N - 1
    const int64_t lo = cta * p.tiles / G;
    const int64_t N = (cta + 1) * p.tiles / G - lo;
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
        const int lane = static_cast<int>(threadIdx.x & 31);
        const int n_loads = NIN * (p.rank3 ? p.row_chunks : p.row_chunks * p.atoms);
        const BoxRef mine = box_ref(maps, p, lane < n_loads ? lane : 0, 0);
        TileCursor tc(p, lo, 1);
        StageCursor st;
        int64_t issued = 0;
        const int64_t pro = N < S - 1 ? N : S - 1;
        for (; issued < pro; ++issued) {
            issue_tile_lanes<NIN>(maps, p, tc, mine, n_loads, base + st.s * p.stage_bytes, full + 8u * st.s);
            tc.next(p);
            st.next(S);
        }
        for (; issued < N; ++issued) {
            // every lane waits (measured faster here for every op)
            if (issued >= S && !role_wait(empty + 8u * st.s, st.phase ^ 1u, p, abort_flag, false))
                break;
            issue_tile_lanes<NIN>(maps, p, tc, mine, n_loads, base + st.s * p.stage_bytes, full + 8u * st.s);
            tc.next(p);
            st.next(S);
        }
        if (*abort_flag && lane == 0) {
            const int64_t first = issued > S ? issued - S : 0;
            for (int64_t k = first; k < issued; ++k)
                (void)mbar_wait(full + 8u * (k % S), static_cast<uint32_t>((k / S) & 1), p.timeout_ns);
        }
    } else {
        // ---------------------------------------------- compute warps
        const uint32_t tid = threadIdx.x - 32;
        const uint32_t threads = blockDim.x - 32;
        // stage, phase, band and column tile advance with the tile counter
        // (no divisions in the loop); first_ct opens the CTA's share of the band
        uint32_t s = 0, phase = 0, band_parity = 0;
        // the thread's first kRegUnits units: partials in registers
        float acc[kRegUnits];
#pragma unroll
        for (int k = 0; k < kRegUnits; ++k)
            acc[k] = 0.f;
        int64_t band = lo / p.tiles_c;
        int64_t ct = lo - band * p.tiles_c, first_ct = ct;
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
            if (!ragged) {
#pragma unroll
                for (int k = 0; k < kRegUnits; ++k) {
                    const uint32_t u = tid + k * threads;
                    if (u >= p.vec16_per_slot)
                        break;
                    add_unit<DT, OP>(acc[k], p, stage, u);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kRegUnits; ++k) {
                    const uint32_t u = tid + k * threads;
                    if (u >= p.vec16_per_slot)
                        break;
                    if (unit_in_columns<DT>(p, tb, u))
                        add_unit<DT, OP>(acc[k], p, stage, u);
                }
            }
            // units past the register partials keep theirs in shared memory
            for (uint32_t u = tid + kRegUnits * threads; u < p.vec16_per_slot; u += threads) {
                float part = ct == first_ct ? 0.f : partial[u];
                if (!ragged || unit_in_columns<DT>(p, tb, u))
                    add_unit<DT, OP>(part, p, stage, u);
                partial[u] = part;
            }
            __syncwarp();
            if ((threadIdx.x & 31) == 0)
                mbar_arrive(empty + 8u * s);
            if (ct == p.tiles_c - 1 || i == N - 1) {
                // the CTA's share of the band is complete once every compute
                // warp has added its last partials; then each row's partials,
                // box by box
#pragma unroll
                for (int k = 0; k < kRegUnits; ++k) {
                    const uint32_t u = tid + k * threads;
                    if (u >= p.vec16_per_slot)
                        break;
                    partial[u] = acc[k];
                    acc[k] = 0.f;
                }
                __syncwarp();
                if ((threadIdx.x & 31) == 0)
                    mbar_arrive(band_done);
                if (!wait_or_abort(band_done, band_parity, p, abort_flag))
                    break;
                if (first_ct == 0 && ct == p.tiles_c - 1) {
                    for (uint32_t r = tid; r < static_cast<uint32_t>(p.box_rows); r += threads) {
                        const int64_t row = tb.row0 + r;
                        if (row >= p.rows)
                            break;
                        row_sums[row] = row_total<DT>(p, partial, static_cast<int>(r));
                    }
                } else {
                    const int64_t x0 = band * p.tiles_c;
                    const int64_t c0 = range_owner(x0, p.tiles, G);
                    const uint32_t shares = static_cast<uint32_t>(range_owner(x0 + p.tiles_c - 1, p.tiles, G) - c0 + 1);
                    for (uint32_t r = tid; r < static_cast<uint32_t>(p.box_rows); r += threads) {
                        const int64_t row = tb.row0 + r;
                        if (row >= p.rows)
                            break;
                        finish_cut_row(sc.piece + band * sc.pieces * p.box_rows + r, sc.arrivals + row,
                                       p.box_rows, cta - c0, shares, row_total<DT>(p, partial, static_cast<int>(r)),
                                       row_sums + row);
                    }
                }
                // before the next band overwrites the partials
                __syncwarp();
                if ((threadIdx.x & 31) == 0)
                    mbar_arrive(band_free);
                if (!wait_or_abort(band_free, band_parity, p, abort_flag))
                    break;
                band_parity ^= 1;
                ++band;
                ct = 0;
                first_ct = 0;
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
                          const CUtensorMap* maps, const TmaArgs& args, const RowsumScratch& scratch,
                          float* row_sums)
{
    TmaMaps m;
    for (int j = 0; j < 4; ++j)
        m.m[j] = maps[j];
    TmaArgs a = args;
    RowsumScratch sc = scratch;
    void* params[] = {&m, &a, &sc, &row_sums};
    return cudaLaunchKernel(kKernels[dtype][op], dim3(grid), dim3(threads), params, smem, stream);
}

}  // namespace tsx
