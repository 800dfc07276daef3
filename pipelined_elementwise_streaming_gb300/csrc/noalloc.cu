// tsx_ewise_noalloc: the elementwise stream for callers that may not
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or not at the moment they
// need the operation: a plugin that runs inside a host engine and may only
// use the memory the engine hands it; a framework whose pooling allocator
// has reserved the device memory it manages (allocating outside the pool
// fails or fragments it); a latency-critical loop that cannot afford the
// implicit device synchronisation that cudaMalloc and cudaFree may cause.
// tsx_plan_create allocates the plan's device status word, so it is not for
// them.  This entry point runs the same TMA kernel as tsx_ewise without a
// plan: the kernel's only scratch memory, its device status word, lives in
// the file-scope array below, which every GPU that loads the library holds
// until the process exits.  The call allocates nothing, host or device.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "plan.h"
#include "tsx_debug.h"

namespace tsx {
namespace {

// The scratch of every allocation-free call on a device.  Its size is the
// stated maximum; a call needs one 4-byte status word of it, which is
// checked here at compile time.
constexpr size_t kNoallocScratchBytes = 256;
static __device__ __align__(256) int g_noalloc_scratch[kNoallocScratchBytes / sizeof(int)];
constexpr size_t kStatusWordBytes = sizeof(int);
static_assert(kStatusWordBytes <= kNoallocScratchBytes, "the status word must fit in the scratch array");

// Device address of the scratch array, looked up once per device.
constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
int* g_scratch[kMaxDevices];
cudaError_t g_setup_error[kMaxDevices];

// Fault hook of the calling host thread (tsx_debug_noalloc_set_fault).
thread_local int64_t t_fault_tile = -1;
thread_local int t_timeout_ms = 0;

int fail(int rc, const char* msg)
{
    set_last_error(msg);
    return rc;
}

int fail(int rc, const char* what, const std::string& why)
{
    char buf[384];
    std::snprintf(buf, sizeof buf, "tsx_ewise_noalloc: %s: %s", what, why.c_str());
    set_last_error(buf);
    return rc;
}

int fail_cuda(cudaError_t e, const char* what)
{
    char buf[256];
    std::snprintf(buf, sizeof buf, "tsx_ewise_noalloc: %s: %s", what, cudaGetErrorString(e));
    set_last_error(buf);
    return TSX_ERR_CUDA;
}

// The scratch address on the current device.  The first call on a device
// takes it with cudaGetSymbolAddress (host code cannot use the array's name
// as a device address) while that device is current.
int scratch_on_current_device(int* device, int** scratch)
{
    cudaError_t e = cudaGetDevice(device);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    const int d = *device;
    if (d < 0 || d >= kMaxDevices)
        return fail(TSX_ERR_UNSUPPORTED, "tsx_ewise_noalloc: device index beyond the 64 it keeps scratch for");
    std::call_once(g_once[d], [d] {
        void* p = nullptr;
        g_setup_error[d] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        g_scratch[d] = static_cast<int*>(p);
    });
    if (g_setup_error[d] != cudaSuccess)
        return fail_cuda(g_setup_error[d], "cudaGetSymbolAddress of the scratch array");
    *scratch = g_scratch[d];
    return TSX_OK;
}

int alignment(const void* ptr)
{
    const uintptr_t v = reinterpret_cast<uintptr_t>(ptr);
    return v % 16 == 0 ? 16 : v % 8 == 0 ? 8 : v % 4 == 0 ? 4 : 1;
}

}  // namespace
}  // namespace tsx

using namespace tsx;

extern "C" void tsx_debug_noalloc_set_fault(int64_t tile, int32_t timeout_ms)
{
    t_fault_tile = tile >= 0 ? tile : -1;
    t_timeout_ms = timeout_ms > 0 ? timeout_ms : 0;
}

extern "C" int tsx_ewise_noalloc(tsx_dtype dtype, int64_t rows, int64_t cols, int box_rows, int box_cols,
                                 int stages, tsx_variant variant, tsx_op op, const void* a, const void* b,
                                 const void* c, void* out, tsx_stream_t stream, int* status_out)
{
    if (variant != TSX_TMA && variant != TSX_TMA_RANK3)
        return fail(TSX_ERR_INVALID, "tsx_ewise_noalloc: only the TMA variants (TSX_TMA, TSX_TMA_RANK3) are offered");
    if (op < TSX_COPY || op > TSX_FMA)
        return fail(TSX_ERR_INVALID, "tsx_ewise_noalloc: unknown op");
    Knobs knobs;
    knobs.timeout_ms = t_timeout_ms > 0 ? t_timeout_ms : 1000;
    Geometry g;
    std::string why;
    int rc = make_geometry(dtype, rows, cols, cols, box_rows, box_cols, stages, variant, knobs, &g, &why);
    if (rc != TSX_OK)
        return fail(rc, "no legal plan for these arguments", why);
    if (g.tiles == 0) {
        if (status_out)
            *status_out = TSX_OK;
        set_last_error("");
        return TSX_OK;   // empty tensor: nothing to do
    }
    const int n_in = op_arity(op);
    if (!a || !out)
        return fail(TSX_ERR_INVALID, "tsx_ewise_noalloc: a and out are required");
    if ((n_in >= 2) != (b != nullptr) || (n_in >= 3) != (c != nullptr))
        return fail(TSX_ERR_INVALID, "tsx_ewise_noalloc: b / c must be given exactly when the op uses them");
    const void* ptrs[4] = {a, b, c, out};
    for (const void* q : ptrs)
        if (q && alignment(q) < 16)
            return fail(TSX_ERR_ALIGN, "tsx_ewise_noalloc: TMA needs 16-byte aligned base pointers");

    int device = 0;
    int* scratch = nullptr;
    rc = scratch_on_current_device(&device, &scratch);
    if (rc != TSX_OK)
        return rc;
    int sm_count = 0, max_smem = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaDeviceGetAttribute");
    OpGeometry og;
    rc = make_op_geometry(g, op, max_smem, &og, &why);
    if (rc != TSX_OK)
        return fail(rc, "no launch for these arguments", why);
    const int kind = og.compute_groups == 2 ? kTmaSplit : kTmaPlain;
    const void* fn = tma_kernel(dtype, op, kind);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(og.smem_bytes));
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaFuncSetAttribute");
    int blocks = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, og.block_threads, og.smem_bytes);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (blocks < 1)
        return fail(TSX_ERR_UNSUPPORTED, "tsx_ewise_noalloc: the kernel cannot be resident with this shared memory");
    if (og.ctas_cap > 0 && blocks > og.ctas_cap)
        blocks = og.ctas_cap;   // the same launch as tsx_ewise
    const int64_t slots = int64_t(sm_count) * blocks;
    const int grid = int(g.tiles < slots ? g.tiles : slots);

    CUtensorMap maps[4];
    std::memset(maps, 0, sizeof maps);
    for (int j = 0; j < 4; ++j) {
        if (!ptrs[j])
            continue;
        rc = encode_tensor_map(g, ptrs[j], &maps[j]);
        if (rc != TSX_OK)
            return rc;
    }
    TmaArgs args;
    fill_tma_args(g, og, scratch, t_fault_tile, &args);

    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the status word keeps the previous call's value: start this one at zero
    e = cudaMemsetAsync(scratch, 0, kStatusWordBytes, st);
    if (e != cudaSuccess)
        return fail_cuda(e, "clearing the status word");
    e = launch_tma(dtype, op, kind, grid, og.block_threads, og.smem_bytes, st, maps, args);
    if (e != cudaSuccess)
        return fail_cuda(e, "kernel launch");
    if (status_out) {
        // read the word in stream order (no device-wide synchronisation)
        int h = 0;
        e = cudaMemcpyAsync(&h, scratch, sizeof h, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
        if (e != cudaSuccess)
            return fail_cuda(e, "reading the status word");
        *status_out = h;
    }
    set_last_error("");
    return TSX_OK;
}
