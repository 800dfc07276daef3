// The C ABI of libtsx (include/tsx.h): plans, tensor maps, launches and the
// device status word.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "plan.h"
#include "tsx_debug.h"

namespace tsx {

namespace {

// The last error message of the calling thread, in a fixed buffer so that
// reporting an error never allocates (longer messages are cut short).
thread_local char g_last_error[512];

void store_message(const char* a, const char* b = nullptr)
{
    std::snprintf(g_last_error, sizeof g_last_error, "%s%s%s", a ? a : "", b ? ": " : "", b ? b : "");
}

int set_error(int rc, const std::string& msg)
{
    store_message(msg.c_str());
    return rc;
}

int set_error(int rc, const char* msg)
{
    store_message(msg);
    return rc;
}

int cuda_error(cudaError_t e, const char* what)
{
    store_message(what, cudaGetErrorString(e));
    return TSX_ERR_CUDA;
}

// cuTensorMapEncodeTiled, looked up through the runtime so that the library
// does not link against the driver library (it then loads on machines
// without a GPU, where only tsx_plan_query is usable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(std::string* why)
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static std::string err;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
            err = std::string("cuTensorMapEncodeTiled is unavailable: ") + cudaGetErrorString(e);
        else
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn && why)
        *why = err;
    return fn;
}

CUtensorMapDataType map_dtype(int dtype)
{
    return dtype == TSX_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
         : dtype == TSX_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// A promoted map moves the same bytes in wider unsigned elements.
CUtensorMapDataType map_type(const Geometry& g)
{
    if (g.tma_es == g.es)
        return map_dtype(g.dtype);
    return g.tma_es == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
         : g.tma_es == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                         : CU_TENSOR_MAP_DATA_TYPE_UINT64;
}

}  // namespace

void set_last_error(const char* msg) { store_message(msg); }

}  // namespace tsx

using namespace tsx;

struct tsx_plan {
    Geometry g;
    int device = 0;
    int sm_count = 0;
    int max_smem = 0;
    int* d_status = nullptr;
    // counters of the dynamic tile order, one slot (two words) per stream the
    // plan has launched on, keyed by the stream's unique id: launches on one
    // stream run in order, and each launch's last CTA zeroes its slot
    unsigned long long* d_tile_counters = nullptr;
    std::mutex slot_mutex;
    unsigned long long slot_stream[kTileCounterSlots] = {};
    int slots_used = 0;
    // test hooks (include/tsx_debug.h): the tile whose loads the producer
    // skips, and the traced kernels' schedule record, [trace_grid][trace_cap]
    // events of 16 bytes
    int64_t fault_tile = -1;
    int trace_cap = 0;
    uint32_t* trace_buf = nullptr;
    int trace_grid = 0;

    struct OpLaunch {
        bool ready = false;
        OpGeometry og;
        int ctas_per_sm = 0;
        int grid = 0;
        RowsumScratch scratch{};   // row sums only: shares of the bands cut between CTAs
    } ops[12],   // op + 6 * accumulate
        rowsum_ops[6];

    // tensor maps, keyed by base pointer (the shape is the plan's)
    struct MapEntry {
        const void* ptr = nullptr;
        uint64_t used = 0;
        alignas(64) CUtensorMap map;
    } maps[8];
    uint64_t clock = 0;
};

namespace {

// The mixed variant runs its own instantiation only for ops with a b operand.
bool mixed_launch(int variant, int op) { return variant == TSX_TMA_MIXED && op_arity(op) >= 2; }

int tma_kind(int variant, int op, bool accumulate, bool traced, bool split)
{
    if (accumulate)
        return kTmaAccumulate;
    if (mixed_launch(variant, op))
        return kTmaMixed;
    if (split)
        return traced ? kTmaTracedSplit : kTmaSplit;
    return traced ? kTmaTraced : kTmaPlain;
}

// The reduce-store is offered by the two all-TMA variants.
bool accumulate_offered(int variant) { return variant == TSX_TMA || variant == TSX_TMA_RANK3; }

const void* kernel_of(int variant, int dtype, int op, bool accumulate, bool traced, bool split)
{
    if (variant == TSX_LDGSTS)
        return ldgsts_kernel(dtype, op);
    if (variant == TSX_SYNC)
        return sync_kernel(dtype, op);
    return tma_kernel(dtype, op, tma_kind(variant, op, accumulate, traced, split));
}

// The trace ring of the traced kernel (test hook): large enough for `grid`
// CTAs, cleared on `st` before every launch.
int prepare_trace(tsx_plan* p, int grid, cudaStream_t st)
{
    const size_t per_cta = size_t(p->trace_cap) * 16;
    if (p->trace_grid < grid) {
        cudaFree(p->trace_buf);
        p->trace_buf = nullptr;
        p->trace_grid = 0;
        if (cudaMalloc(&p->trace_buf, per_cta * size_t(grid)) != cudaSuccess) {
            (void)cudaGetLastError();
            return set_error(TSX_ERR_NOMEM, "allocating the trace ring");
        }
        p->trace_grid = grid;
    }
    const cudaError_t e = cudaMemsetAsync(p->trace_buf, 0, per_cta * size_t(grid), st);
    return e == cudaSuccess ? TSX_OK : cuda_error(e, "clearing the trace ring");
}

// Geometry, kernel attributes, occupancy and grid for one op (cached).
int prepare_op(tsx_plan* p, int op, bool accumulate, tsx_plan::OpLaunch** out)
{
    tsx_plan::OpLaunch& L = p->ops[op + (accumulate ? 6 : 0)];
    if (!L.ready) {
        std::string why;
        const int rc = make_op_geometry(p->g, op, p->max_smem, &L.og, &why);
        if (rc != TSX_OK)
            return set_error(rc, why);
        if (accumulate) {
            L.og.tile_order = 1;   // the reduce-store kernels take the static order
            L.og.dynamic_share = 0;
            L.og.compute_groups = 1;   // and store a tile at once
        }
        const void* fn = kernel_of(p->g.variant, p->g.dtype, op, accumulate, p->trace_cap > 0,
                                   L.og.compute_groups == 2);
        if (!fn)
            return set_error(TSX_ERR_UNSUPPORTED, "traced launches: only fp32 copy and add have a traced kernel");
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.og.smem_bytes));
        if (e != cudaSuccess)
            return cuda_error(e, "cudaFuncSetAttribute");
        int blocks = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, L.og.block_threads, L.og.smem_bytes);
        if (e != cudaSuccess)
            return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (blocks < 1)
            return set_error(TSX_ERR_UNSUPPORTED, "the kernel cannot be resident with this shared memory / threads");
        if (L.og.ctas_cap > 0 && blocks > L.og.ctas_cap)
            blocks = L.og.ctas_cap;
        L.ctas_per_sm = blocks;
        if (mixed_launch(p->g.variant, op))
            L.og.b_prefetch_ahead = mixed_prefetch_ahead(p->g, blocks);
        // persistent grid: every resident CTA slot once, no more CTAs than tiles
        const int64_t slots = int64_t(p->sm_count) * blocks;
        L.grid = int(p->g.tiles < slots ? p->g.tiles : slots);
        // the planner's dynamic order pays only with enough tiles per CTA
        if (L.og.tile_order == 2 && p->g.knobs.tile_order <= 0 &&
            p->g.tiles < int64_t(kDynamicMinTilesPerCta) * L.grid) {
            L.og.tile_order = 1;
            L.og.dynamic_share = 0;
        }
        L.ready = true;
    }
    *out = &L;
    return TSX_OK;
}

int encode_map(tsx_plan* p, const void* ptr, CUtensorMap* map) { return encode_tensor_map(p->g, ptr, map); }

}  // namespace

namespace tsx {

int encode_tensor_map(const Geometry& g, const void* ptr, CUtensorMap* map)
{
    std::string why;
    EncodeTiledFn fn = encode_fn(&why);
    if (!fn)
        return set_error(TSX_ERR_CUDA, why);
    TensorMapArgs m;
    tensor_map_args(g, &m);
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], estr[5];
    for (int d = 0; d < m.rank; ++d) {
        dims[d] = m.dims[d];
        box[d] = m.box[d];
        estr[d] = 1;
    }
    for (int d = 0; d + 1 < m.rank; ++d)
        strides[d] = m.strides[d];
    const CUresult r = fn(map, map_type(g), cuuint32_t(m.rank), const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, static_cast<CUtensorMapSwizzle>(m.swizzle),
                          static_cast<CUtensorMapL2promotion>(m.l2_promotion), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[96];
        std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
        return set_error(TSX_ERR_CUDA, buf);
    }
    return TSX_OK;
}

}  // namespace tsx

namespace {

// The tensor map of `ptr`, from the plan's cache or freshly encoded.
int get_map(tsx_plan* p, const void* ptr, CUtensorMap* out)
{
    tsx_plan::MapEntry* victim = &p->maps[0];
    for (auto& e : p->maps) {
        if (e.ptr == ptr) {
            e.used = ++p->clock;
            *out = e.map;
            return TSX_OK;
        }
        if (e.used < victim->used)
            victim = &e;
    }
    const int rc = encode_map(p, ptr, &victim->map);
    if (rc != TSX_OK) {
        victim->ptr = nullptr;
        victim->used = 0;
        return rc;
    }
    victim->ptr = ptr;
    victim->used = ++p->clock;
    *out = victim->map;
    return TSX_OK;
}

// Kernel arguments of the TMA kernels for plan p and one op's geometry.
void fill_tma_args(const tsx_plan* p, const OpGeometry& og, TmaArgs* args)
{
    tsx::fill_tma_args(p->g, og, p->d_status, p->fault_tile, args);
}

// The dynamic tile order's counter slot for launches on `st`, or NULL
// (static order) while the stream is being captured into a graph (a graph
// may be replayed on any stream), when the stream's id cannot be read, or
// once the plan has served kTileCounterSlots streams.
unsigned long long* tile_counter_for(tsx_plan* p, cudaStream_t st)
{
    if (!p->d_tile_counters)
        return nullptr;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &capture) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (capture != cudaStreamCaptureStatusNone)
        return nullptr;
    unsigned long long id = 0;
    if (cudaStreamGetId(st, &id) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(p->slot_mutex);
    for (int i = 0; i < p->slots_used; ++i)
        if (p->slot_stream[i] == id)
            return p->d_tile_counters + 2 * i;
    if (p->slots_used == kTileCounterSlots)
        return nullptr;
    p->slot_stream[p->slots_used] = id;
    return p->d_tile_counters + 2 * p->slots_used++;
}

int alignment_of(const void* ptr)
{
    const uintptr_t v = reinterpret_cast<uintptr_t>(ptr);
    for (int a : {16, 8, 4, 2})
        if (v % a == 0)
            return a;
    return 1;
}

size_t arrival_bytes(const Geometry& g) { return size_t(g.tiles_r) * size_t(g.box_rows) * sizeof(uint32_t); }

int read_status(tsx_plan* p, bool clear)
{
    int h = 0;
    cudaError_t e = cudaMemcpy(&h, p->d_status, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_error(e, "reading the status word");
    if (clear && h != TSX_OK) {
        e = cudaMemset(p->d_status, 0, sizeof(int));
        if (e != cudaSuccess)
            return cuda_error(e, "clearing the status word");
        // a row reduction that gave up may have left arrivals counted
        for (auto& L : p->rowsum_ops) {
            if (!L.scratch.arrivals)
                continue;
            e = cudaMemset(L.scratch.arrivals, 0, arrival_bytes(p->g));
            if (e != cudaSuccess)
                return cuda_error(e, "clearing the row arrivals");
        }
    }
    return h;
}

// Launch shape of the row reduction for one op (cached): the stages of the
// elementwise geometry, two barriers per stage, two band barriers, the
// abort flag and one fp32
// partial per 16-byte unit of a staged slot; compute warps plus the
// producer warp.
// fp32 row sums: stage bytes per SM the CTA count aims at (the
// compute-heavy sqrt and exp, the other ops).
constexpr int64_t kRowsumRingPerSmHeavy = 96 * 1024;
constexpr int64_t kRowsumRingPerSm = 128 * 1024;
// and at most this many CTAs per SM (eight CTAs of 64 threads ran fp32 copy
// row sums in 4 KB tiles at 4298 GB/s against 5666 with six)
constexpr int64_t kRowsumMaxCtas = 6;

int prepare_rowsum(tsx_plan* p, int op, tsx_plan::OpLaunch** out)
{
    tsx_plan::OpLaunch& L = p->rowsum_ops[op];
    if (!L.ready) {
        std::string why;
        int rc = make_op_geometry(p->g, op, p->max_smem, &L.og, &why);
        if (rc != TSX_OK)
            return set_error(rc, why);
        L.og.tile_order = 0;   // contiguous tile ranges per CTA, no counter
        // one fp32 partial per 16-byte unit of a staged slot
        const size_t partials = size_t(L.og.vec16_per_slot) * 4;
        const size_t smem = size_t(p->g.stages) * L.og.stage_bytes + size_t(p->g.stages) * 16 + 16 + 16 +
                            kSmemAlign + partials;
        if (smem > size_t(p->max_smem))
            return set_error(TSX_ERR_UNSUPPORTED, "the row reduction's stages do not fit in shared memory");
        L.og.smem_bytes = smem;
        // CTAs and compute threads per SM.  16-bit: about 768 threads per
        // SM, shared by every CTA that fits (a 16-bit element is half an fp32
        // one's bytes, so it needs about twice the threads per byte).  fp32:
        // enough CTAs for about 128 KB of stages per SM (96 KB for sqrt and
        // exp, which are bound by their arithmetic), at least three (as many
        // as fit) and at most six, of 384 threads in all.  Measured on GB300, [128, 2^20] in
        // 8x128 tiles at 4 stages: fp32 fma (12 KB stages) 6884 GB/s with
        // three CTAs of 192 threads against 6236 with every CTA that fits;
        // fp32 copy, exp and sqrt (4 KB stages) 5775, 4290 and 3647 with six
        // to eight CTAs of 64 threads against 3451, 3156 and 2471 with three
        // of 192.  The 128 KB target against 96 KB: fp32 add in 8x128 tiles
        // at 4 stages 5765 -> 6488, copy in 8x256 tiles 5350 -> 5981, fma at
        // 2 and 3 stages +2.6 %.  bf16 exp [16384, 16384] in 32x256 tiles at
        // 2 stages: 5942 with five CTAs of 128 threads, 5247 with three of
        // 160.
        const int fit0 = int(kSmemPerSm / (smem + kSmemPerCtaReserved));
        const int fit = fit0 < 1 ? 1 : fit0;
        const bool wide = p->g.es == 4;
        int ctas = fit;
        if (wide) {
            const int64_t ring = int64_t(p->g.stages) * int64_t(L.og.stage_bytes);
            const int64_t target = op == TSX_SQRT || op == TSX_EXP ? kRowsumRingPerSmHeavy : kRowsumRingPerSm;
            int64_t want = (target + ring / 2) / ring;
            want = want < 3 ? 3 : want > kRowsumMaxCtas ? kRowsumMaxCtas : want;
            ctas = want < fit ? int(want) : fit;
        }
        L.ctas_per_sm = ctas;   // the cap, before occupancy below
        // (fp32 CTAs that do not reach three keep 192 threads each)
        int threads = (wide ? (ctas >= 3 ? 384 : 192 * ctas) : 768) / ctas / 32 * 32;
        threads = threads < 64 ? 64 : threads > 512 ? 512 : threads;
        const int forced = p->g.knobs.threads;
        if (forced > 0) {
            if (forced > kMaxThreads - 32)
                return set_error(TSX_ERR_UNSUPPORTED, "tuning.threads: at most 992 compute threads for row sums");
            threads = forced;
        }
        L.og.threads = threads;
        L.og.block_threads = threads + 32;
        const void* fn = rowsum_kernel(p->g.dtype, op);
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess)
            return cuda_error(e, "cudaFuncSetAttribute");
        int blocks = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, L.og.block_threads, smem);
        if (e != cudaSuccess)
            return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (blocks < 1)
            return set_error(TSX_ERR_UNSUPPORTED, "the row reduction cannot be resident with this shared memory");
        const int cap = p->g.knobs.ctas_per_sm > 0 ? p->g.knobs.ctas_per_sm : L.ctas_per_sm;
        if (blocks > cap)
            blocks = cap;
        L.ctas_per_sm = blocks;
        // contiguous tile ranges, one per CTA; a band is cut between at most
        // 1 + ceil((tiles_c - 1) / floor(T / G)) consecutive CTAs
        const int64_t slots = int64_t(p->sm_count) * blocks;
        const Geometry& g = p->g;
        L.grid = int(g.tiles < slots ? g.tiles : slots);
        const int64_t shortest = g.tiles / L.grid;
        const int64_t pieces = 1 + (g.tiles_c - 1 + shortest - 1) / shortest;
        if (pieces > 1) {
            L.scratch.pieces = pieces;
            cudaError_t e1 = cudaMalloc(&L.scratch.piece, size_t(g.tiles_r) * size_t(pieces) * g.box_rows * sizeof(float));
            cudaError_t e2 = e1 == cudaSuccess ? cudaMalloc(&L.scratch.arrivals, arrival_bytes(g)) : e1;
            cudaError_t e3 = e2 == cudaSuccess ? cudaMemset(L.scratch.arrivals, 0, arrival_bytes(g)) : e2;
            if (e3 != cudaSuccess) {
                cudaFree(L.scratch.piece);
                cudaFree(L.scratch.arrivals);
                L.scratch = RowsumScratch{};
                (void)cudaGetLastError();
                return set_error(e1 == cudaErrorMemoryAllocation || e2 == cudaErrorMemoryAllocation ? TSX_ERR_NOMEM
                                                                                                      : TSX_ERR_CUDA,
                                 "allocating the row reduction's scratch");
            }
        }
        L.ready = true;
    }
    *out = &L;
    return TSX_OK;
}

}  // namespace

namespace {

// A launch candidate of tsx_plan_tune: knob values (0 / -1: the planner's).
struct TuneKnobs {
    int ctas_per_sm, threads, store_warps, store_lag;
};

// The first pass: the planner's launch, then 1..8 CTAs per SM sharing 256
// or 512 compute threads per SM (the store side as the plan's knobs say).
int shape_candidates(const Knobs& base, TuneKnobs* out)
{
    int n = 0;
    out[n++] = {0, 0, base.store_warps, base.store_lag};
    for (int ctas = 1; ctas <= 8; ++ctas)
        for (int total : {256, 512}) {
            int threads = total / ctas / 32 * 32;
            threads = threads < 32 ? 32 : threads;
            bool seen = false;
            for (int k = 1; k < n; ++k)
                seen = seen || (out[k].ctas_per_sm == ctas && out[k].threads == threads);
            if (!seen)
                out[n++] = {ctas, threads, base.store_warps, base.store_lag};
        }
    return n;
}

// Set up every candidate (one launch each, distinct launches only), time
// the distinct ones over two rounds of `reps` launches (the shortest round
// counts), and return the fastest's index in `launch` (-1 if none ran).
// The plan's knobs select a candidate while it is set up; the caller
// restores them.  Shapes that cannot be resident are skipped.
int time_candidates(tsx_plan* p, tsx_op op_arg, const void* a, const void* b, const void* c, void* out,
                    tsx_stream_t stream, int reps, const TuneKnobs* cand, int n, tsx_plan::OpLaunch* launch,
                    const Knobs& base, int* pick)
{
    tsx_plan::OpLaunch& slot = p->ops[int(op_arg)];
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    bool usable[24] = {};
    float best_ms[24];
    for (float& x : best_ms)
        x = -1.f;
    *pick = -1;
    cudaEvent_t ev[2] = {nullptr, nullptr};
    cudaError_t e = cudaEventCreate(&ev[0]);
    if (e == cudaSuccess)
        e = cudaEventCreate(&ev[1]);
    int rc = e == cudaSuccess ? TSX_OK : cuda_error(e, "cudaEventCreate");
    for (int k = 0; k < n && rc == TSX_OK; ++k) {
        p->g.knobs = base;
        p->g.knobs.ctas_per_sm = cand[k].ctas_per_sm;
        p->g.knobs.threads = cand[k].threads;
        p->g.knobs.store_warps = cand[k].store_warps;
        p->g.knobs.store_lag = cand[k].store_lag;
        slot.ready = false;
        const int r = tsx_ewise(p, op_arg, a, b, c, out, stream);
        if (r == TSX_ERR_UNSUPPORTED)
            continue;   // this shape does not fit
        if (r != TSX_OK) {
            rc = r;
            break;
        }
        bool dup = false;
        for (int j = 0; j < k; ++j)
            dup = dup || (usable[j] && launch[j].ctas_per_sm == slot.ctas_per_sm &&
                          launch[j].og.threads == slot.og.threads && launch[j].og.store_warps == slot.og.store_warps &&
                          launch[j].og.store_lag == slot.og.store_lag);
        launch[k] = slot;
        usable[k] = !dup;
    }
    for (int round = 0; round < 2 && rc == TSX_OK; ++round)
        for (int k = 0; k < n && rc == TSX_OK; ++k) {
            if (!usable[k])
                continue;
            slot = launch[k];
            e = cudaEventRecord(ev[0], st);
            for (int i = 0; i < reps && e == cudaSuccess && rc == TSX_OK; ++i)
                rc = tsx_ewise(p, op_arg, a, b, c, out, stream);
            if (e == cudaSuccess && rc == TSX_OK)
                e = cudaEventRecord(ev[1], st);
            if (e == cudaSuccess && rc == TSX_OK)
                e = cudaEventSynchronize(ev[1]);
            float ms = 0.f;
            if (e == cudaSuccess && rc == TSX_OK)
                e = cudaEventElapsedTime(&ms, ev[0], ev[1]);
            if (e != cudaSuccess && rc == TSX_OK)
                rc = cuda_error(e, "timing a candidate launch");
            if (rc == TSX_OK && (best_ms[k] < 0.f || ms < best_ms[k]))
                best_ms[k] = ms;
        }
    for (cudaEvent_t x : ev)
        if (x)
            cudaEventDestroy(x);
    for (int k = 0; k < n; ++k)
        if (usable[k] && best_ms[k] >= 0.f && (*pick < 0 || best_ms[k] < best_ms[*pick]))
            *pick = k;
    return rc;
}

// tsx_plan_tune's search: the CTA and thread shapes first, then, unless the
// plan's knobs fix it, the store side (one or two store warps, lag 0 or 1)
// on the fastest shape.  The fastest launch stays in the plan's slot.
int tune_launch(tsx_plan* p, tsx_op op_arg, const void* a, const void* b, const void* c, void* out,
                tsx_stream_t stream, int reps)
{
    tsx_plan::OpLaunch& slot = p->ops[int(op_arg)];
    const tsx_plan::OpLaunch planner = slot;
    const Knobs base = p->g.knobs;
    TuneKnobs cand[24];
    tsx_plan::OpLaunch launch[24];
    int n = shape_candidates(base, cand);
    int pick = -1;
    int rc = time_candidates(p, op_arg, a, b, c, out, stream, reps, cand, n, launch, base, &pick);
    tsx_plan::OpLaunch best = pick >= 0 ? launch[pick] : planner;
    if (rc == TSX_OK && pick >= 0 && is_tma_variant(p->g.variant) && base.store_warps <= 0 && base.store_lag < 0) {
        // the store side on the fastest shape (the shape itself first)
        const TuneKnobs shape = {best.ctas_per_sm, best.og.threads, best.og.store_warps, best.og.store_lag};
        n = 0;
        cand[n++] = shape;
        for (int w = 1; w <= 2; ++w)
            for (int lag = 0; lag <= 1; ++lag)
                if (w != shape.store_warps || lag != shape.store_lag)
                    cand[n++] = {shape.ctas_per_sm, shape.threads, w, lag};
        rc = time_candidates(p, op_arg, a, b, c, out, stream, reps, cand, n, launch, base, &pick);
        if (pick >= 0)
            best = launch[pick];
    }
    p->g.knobs = base;
    slot = best;
    slot.ready = true;
    if (rc != TSX_OK)
        return rc;
    const int s = read_status(p, true);
    if (s != TSX_OK)
        return set_error(s, "a device-side wait gave up while tuning");
    return TSX_OK;
}

}  // namespace

extern "C" {

tsx_plan_t tsx_plan_create(tsx_dtype dtype, int64_t rows, int64_t cols, int box_rows, int box_cols, int stages,
                           tsx_variant variant)
{
    return tsx_plan_create_pitched(dtype, rows, cols, cols, box_rows, box_cols, stages, variant);
}

tsx_plan_t tsx_plan_create_pitched(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                                   int box_cols, int stages, tsx_variant variant)
{
    return tsx_plan_create_tuned(dtype, rows, cols, pitch, box_rows, box_cols, stages, variant, nullptr);
}

tsx_plan_t tsx_plan_create_tuned(tsx_dtype dtype, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                                 int box_cols, int stages, tsx_variant variant, const tsx_tuning* tuning)
{
    std::string why;
    Geometry g;
    Knobs knobs;
    int rc = resolve_knobs(tuning, &knobs, &why);
    if (rc == TSX_OK)
        rc = make_geometry(dtype, rows, cols, pitch, box_rows, box_cols, stages, variant, knobs, &g, &why);
    if (rc != TSX_OK) {
        set_error(rc, why);
        return nullptr;
    }
    tsx_plan* p = new (std::nothrow) tsx_plan;
    if (!p) {
        set_error(TSX_ERR_NOMEM, "out of host memory");
        return nullptr;
    }
    p->g = g;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
    if (e == cudaSuccess) {
        e = cudaMalloc(&p->d_status, sizeof(int));
        if (e == cudaSuccess)
            e = cudaMemset(p->d_status, 0, sizeof(int));
    }
    if (e == cudaSuccess && is_tma_variant(g.variant)) {
        const size_t bytes = size_t(kTileCounterSlots) * 2 * sizeof(unsigned long long);
        e = cudaMalloc(&p->d_tile_counters, bytes);
        if (e == cudaSuccess)
            e = cudaMemset(p->d_tile_counters, 0, bytes);
    }
    if (e != cudaSuccess) {
        cuda_error(e, "tsx_plan_create");
        if (p->d_status)
            cudaFree(p->d_status);
        if (p->d_tile_counters)
            cudaFree(p->d_tile_counters);
        delete p;
        return nullptr;
    }
    set_last_error("");
    return p;
}

void tsx_plan_destroy(tsx_plan_t p)
{
    if (!p)
        return;
    if (p->d_status)
        cudaFree(p->d_status);
    cudaFree(p->d_tile_counters);
    cudaFree(p->trace_buf);
    for (auto& L : p->rowsum_ops) {
        cudaFree(L.scratch.piece);
        cudaFree(L.scratch.arrivals);
    }
    delete p;
}

int tsx_plan_status(tsx_plan_t p)
{
    if (!p)
        return set_error(TSX_ERR_INVALID, "NULL plan");
    return read_status(p, true);
}

const char* tsx_last_error(void) { return g_last_error; }

int tsx_debug_trace(tsx_plan_t p, uint32_t* events, int64_t capacity, int32_t* grid, int32_t* per_cta)
{
    if (!p || (!events && capacity > 0) || capacity < 0)
        return set_error(TSX_ERR_INVALID, "NULL plan or events");
    if (p->trace_cap <= 0 || !p->trace_buf)
        return set_error(TSX_ERR_INVALID, "the plan has no trace (tracing not enabled, or no traced launch yet)");
    const int64_t words = int64_t(p->trace_grid) * p->trace_cap * 4;
    const int64_t n = capacity < words ? capacity : words;
    if (n > 0) {
        const cudaError_t e = cudaMemcpy(events, p->trace_buf, size_t(n) * sizeof(uint32_t), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess)
            return cuda_error(e, "reading the trace");
    }
    if (grid)
        *grid = p->trace_grid;
    if (per_cta)
        *per_cta = p->trace_cap;
    set_last_error("");
    return TSX_OK;
}

int tsx_debug_stage_image(tsx_plan_t p, const void* a, int64_t tile, void* image, tsx_stream_t stream)
{
    if (!p || !a || !image)
        return set_error(TSX_ERR_INVALID, "NULL plan, operand or image");
    const Geometry& g = p->g;
    if (!is_tma_variant(g.variant))
        return set_error(TSX_ERR_UNSUPPORTED, "the staged image needs a TMA variant");
    if (tile < 0 || tile >= g.tiles)
        return set_error(TSX_ERR_INVALID, "tile outside the tensor's tiles");
    if (alignment_of(a) < 16 || alignment_of(image) < 16)
        return set_error(TSX_ERR_ALIGN, "a and image must be 16-byte aligned");
    std::string why;
    OpGeometry og;
    int rc = make_op_geometry(g, TSX_COPY, p->max_smem, &og, &why);
    if (rc != TSX_OK)
        return set_error(rc, why);
    CUtensorMap maps[4];
    std::memset(maps, 0, sizeof maps);
    rc = get_map(p, a, &maps[0]);
    if (rc != TSX_OK)
        return rc;
    TmaArgs args;
    tsx::fill_tma_args(g, og, p->d_status, -1, &args);
    if (stage_image_smem(args) > size_t(p->max_smem))
        return set_error(TSX_ERR_UNSUPPORTED, "the slot does not fit in shared memory");
    const cudaError_t e = launch_stage_image(maps, args, tile, image, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_error(e, "kernel launch");
    set_last_error("");
    return TSX_OK;
}

int tsx_debug_plan_set_fault_tile(tsx_plan_t p, int64_t tile)
{
    if (!p)
        return set_error(TSX_ERR_INVALID, "NULL plan");
    p->fault_tile = tile >= 0 ? tile : -1;
    set_last_error("");
    return TSX_OK;
}

int tsx_debug_plan_enable_trace(tsx_plan_t p, int32_t events_per_cta)
{
    if (!p)
        return set_error(TSX_ERR_INVALID, "NULL plan");
    if (events_per_cta < 0 || events_per_cta > (1 << 20))
        return set_error(TSX_ERR_INVALID, "events_per_cta must be in [0, 2^20]");
    if (events_per_cta != p->trace_cap) {
        // the elementwise launches pick their kernel again (traced or not);
        // the ring is reallocated at the next traced launch
        for (auto& L : p->ops)
            L.ready = false;
        cudaFree(p->trace_buf);
        p->trace_buf = nullptr;
        p->trace_grid = 0;
        p->trace_cap = events_per_cta;
    }
    set_last_error("");
    return TSX_OK;
}

int tsx_plan_get_info(tsx_plan_t p, tsx_op op_arg, tsx_plan_info* info)
{
    if (!p || !info)
        return set_error(TSX_ERR_INVALID, "NULL plan or info");
    const bool row_sums = (op_arg & TSX_ROW_SUMS) != 0;
    int op;
    bool accumulate;
    if (!split_op(op_arg & ~TSX_ROW_SUMS, &op, &accumulate))
        return set_error(TSX_ERR_INVALID, "unknown op");
    if (accumulate && (row_sums || !accumulate_offered(p->g.variant)))
        return set_error(row_sums ? TSX_ERR_INVALID : TSX_ERR_UNSUPPORTED,
                         row_sums ? "TSX_ACCUMULATE does not apply to row sums"
                                  : "TSX_ACCUMULATE needs TSX_TMA or TSX_TMA_RANK3");
    if (row_sums && p->g.variant != TSX_TMA && p->g.variant != TSX_TMA_RANK3)
        return set_error(TSX_ERR_UNSUPPORTED, "row sums need a TSX_TMA or TSX_TMA_RANK3 plan");
    tsx_plan::OpLaunch* L = nullptr;
    const int rc = row_sums ? prepare_rowsum(p, op, &L) : prepare_op(p, op, accumulate, &L);
    if (rc != TSX_OK)
        return rc;
    fill_info(p->g, L->og, info);
    info->ctas_per_sm = L->ctas_per_sm;
    info->grid = L->grid;
    info->sm_count = p->sm_count;
    return TSX_OK;
}

int tsx_ewise(tsx_plan_t p, tsx_op op_arg, const void* a, const void* b, const void* c, void* out,
              tsx_stream_t stream)
{
    if (!p)
        return set_error(TSX_ERR_INVALID, "NULL plan");
    int op;
    bool accumulate;
    if (!split_op(op_arg, &op, &accumulate))
        return set_error(TSX_ERR_INVALID, "unknown op");
    if (accumulate && !accumulate_offered(p->g.variant))
        return set_error(TSX_ERR_UNSUPPORTED, "TSX_ACCUMULATE needs TSX_TMA or TSX_TMA_RANK3");
    const int n_in = op_arity(op);
    const Geometry& g = p->g;
    if (g.tiles == 0) {
        set_last_error("");
        return TSX_OK;   // empty tensor: nothing to do, pointers are not examined
    }
    if (!a || !out)
        return set_error(TSX_ERR_INVALID, "a and out are required");
    if ((n_in >= 2) != (b != nullptr))
        return set_error(TSX_ERR_INVALID, n_in >= 2 ? "this op needs b" : "b must be NULL for this op");
    if ((n_in >= 3) != (c != nullptr))
        return set_error(TSX_ERR_INVALID, n_in >= 3 ? "this op needs c" : "c must be NULL for this op");
    const void* ops[4] = {a, b, c, out};
    int align = 16;
    for (int j = 0; j < 4; ++j)
        if (ops[j] && alignment_of(ops[j]) < align)
            align = alignment_of(ops[j]);

    tsx_plan::OpLaunch* L = nullptr;
    int rc = prepare_op(p, op, accumulate, &L);
    if (rc != TSX_OK)
        return rc;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (is_tma_variant(g.variant)) {
        if (align < 16)
            return set_error(TSX_ERR_ALIGN, "TMA needs 16-byte aligned base pointers");
        const bool mixed = mixed_launch(g.variant, op);
        // operands of the TMA ring in slot order; b is read directly when
        // mixed, and its map (slot 2) serves the L2 prefetch only
        const void* staged[4] = {a, b, c, out};
        if (mixed) {
            staged[1] = c;
            staged[2] = b;
        }
        CUtensorMap maps[4];
        std::memset(maps, 0, sizeof maps);
        for (int j = 0; j < 4; ++j) {
            if (!staged[j])
                continue;
            rc = get_map(p, staged[j], &maps[j]);
            if (rc != TSX_OK)
                return rc;
        }
        TmaArgs args{};
        fill_tma_args(p, L->og, &args);
        args.set_operand = mixed ? b : nullptr;
        if (L->og.tile_order == 2 && !mixed) {
            args.tile_counter = tile_counter_for(p, st);
            args.static_tiles = static_tiles_per_cta(g, L->og, L->grid);
        }
        if (p->trace_cap > 0) {
            rc = prepare_trace(p, L->grid, st);
            if (rc != TSX_OK)
                return rc;
            args.trace = p->trace_buf;
            args.trace_cap = p->trace_cap;
        }
        e = launch_tma(g.dtype, op, tma_kind(g.variant, op, accumulate, p->trace_cap > 0, L->og.compute_groups == 2),
                       L->grid, L->og.block_threads, L->og.smem_bytes, st, maps, args);
    } else {
        int vb = g.copy_vec_bytes < align ? g.copy_vec_bytes : align;
        if (vb < 4)
            return set_error(TSX_ERR_ALIGN, "cp.async / vector copies need 4-byte aligned base pointers");
        CopyArgs args{};
        args.rows = g.rows;
        args.cols = g.cols;
        args.pitch = g.pitch;
        args.tiles = g.tiles;
        args.tiles_c = g.tiles_c;
        args.box_rows = g.box_rows;
        args.box_cols = g.box_cols;
        args.stages = g.variant == TSX_SYNC ? 1 : g.stages;
        args.vec_bytes = vb;
        args.tile_bytes = uint32_t(g.box_rows) * uint32_t(g.box_cols) * uint32_t(g.es);
        args.slot_bytes = g.slot_bytes;
        args.stage_bytes = L->og.stage_bytes;
        args.chunks_per_slot = args.tile_bytes / uint32_t(vb);
        args.vec16_per_slot = L->og.vec16_per_slot;
        e = g.variant == TSX_LDGSTS
                ? launch_ldgsts(g.dtype, op, L->grid, L->og.block_threads, L->og.smem_bytes, st, a, b, c, out, args)
                : launch_sync(g.dtype, op, L->grid, L->og.block_threads, L->og.smem_bytes, st, a, b, c, out, args);
    }
    if (e != cudaSuccess)
        return cuda_error(e, "kernel launch");
    if (p->g.knobs.checked) {
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess)
            return cuda_error(e, "cudaStreamSynchronize");
        const int s = read_status(p, true);
        if (s != TSX_OK)
            return set_error(s, "a device-side wait gave up");
    }
    set_last_error("");
    return TSX_OK;
}

int tsx_plan_tune(tsx_plan_t p, tsx_op op_arg, const void* a, const void* b, const void* c, void* out,
                  tsx_stream_t stream, int32_t launches, tsx_plan_info* chosen)
{
    if (!p)
        return set_error(TSX_ERR_INVALID, "NULL plan");
    int op;
    bool accumulate;
    if (!split_op(op_arg, &op, &accumulate))
        return set_error(TSX_ERR_INVALID, "unknown op");
    if (accumulate)
        return set_error(TSX_ERR_INVALID, "tuning runs the op repeatedly: TSX_ACCUMULATE is not tuned");
    if (out && (out == a || out == b || out == c))
        return set_error(TSX_ERR_INVALID, "tuning runs the op repeatedly: out must not alias an input");
    if (p->trace_cap > 0)
        return set_error(TSX_ERR_UNSUPPORTED, "a traced plan is not tuned");
    const int reps = launches <= 0 ? 10 : launches > 1000 ? 1000 : launches;
    // the planner's launch first: it checks the arguments and sets up the op
    int rc = tsx_ewise(p, op_arg, a, b, c, out, stream);
    if (rc != TSX_OK)
        return rc;
    tsx_plan::OpLaunch& slot = p->ops[op];
    const Knobs saved = p->g.knobs;
    if (p->g.tiles > 0 && saved.threads <= 0 && saved.ctas_per_sm <= 0) {
        rc = tune_launch(p, op_arg, a, b, c, out, stream, reps);
        p->g.knobs = saved;
        if (rc != TSX_OK)
            return rc;
    }
    if (chosen) {
        fill_info(p->g, slot.og, chosen);
        chosen->ctas_per_sm = slot.ctas_per_sm;
        chosen->grid = slot.grid;
        chosen->sm_count = p->sm_count;
    }
    set_last_error("");
    return TSX_OK;
}

int tsx_reduce_rows(tsx_plan_t p, tsx_op op, const void* a, const void* b, const void* c, float* row_sums,
                    tsx_stream_t stream)
{
    if (!p)
        return set_error(TSX_ERR_INVALID, "NULL plan");
    if (op < TSX_COPY || op > TSX_FMA)
        return set_error(TSX_ERR_INVALID, "unknown op (TSX_ACCUMULATE does not apply to row sums)");
    const Geometry& g = p->g;
    if (g.variant != TSX_TMA && g.variant != TSX_TMA_RANK3)
        return set_error(TSX_ERR_UNSUPPORTED, "row sums need a TSX_TMA or TSX_TMA_RANK3 plan");
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (g.rows == 0) {
        set_last_error("");
        return TSX_OK;
    }
    if (!row_sums)
        return set_error(TSX_ERR_INVALID, "row_sums is required");
    if (reinterpret_cast<uintptr_t>(row_sums) % 4)
        return set_error(TSX_ERR_ALIGN, "row_sums must be 4-byte aligned");
    if (g.cols == 0) {
        // every row is an empty sum
        const cudaError_t e = cudaMemsetAsync(row_sums, 0, size_t(g.rows) * sizeof(float), st);
        if (e != cudaSuccess)
            return cuda_error(e, "cudaMemsetAsync");
        set_last_error("");
        return TSX_OK;
    }
    const int n_in = op_arity(op);
    if (!a)
        return set_error(TSX_ERR_INVALID, "a is required");
    if ((n_in >= 2) != (b != nullptr) || (n_in >= 3) != (c != nullptr))
        return set_error(TSX_ERR_INVALID, "b / c must be given exactly when the op uses them");
    const void* ops[3] = {a, b, c};
    for (const void* q : ops)
        if (q && alignment_of(q) < 16)
            return set_error(TSX_ERR_ALIGN, "TMA needs 16-byte aligned base pointers");
    tsx_plan::OpLaunch* L = nullptr;
    int rc = prepare_rowsum(p, op, &L);
    if (rc != TSX_OK)
        return rc;
    CUtensorMap maps[4];
    std::memset(maps, 0, sizeof maps);
    for (int j = 0; j < 3; ++j) {
        if (!ops[j])
            continue;
        rc = get_map(p, ops[j], &maps[j]);
        if (rc != TSX_OK)
            return rc;
    }
    TmaArgs args{};
    fill_tma_args(p, L->og, &args);
    cudaError_t e = launch_rowsum(g.dtype, op, L->grid, L->og.block_threads, L->og.smem_bytes, st, maps, args,
                                  L->scratch, row_sums);
    if (e != cudaSuccess)
        return cuda_error(e, "kernel launch");
    if (p->g.knobs.checked) {
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess)
            return cuda_error(e, "cudaStreamSynchronize");
        const int s = read_status(p, true);
        if (s != TSX_OK)
            return set_error(s, "a device-side wait gave up");
    }
    set_last_error("");
    return TSX_OK;
}

}  // extern "C"
