// Test hook: the raw shared-memory image of one staged tile.
//
// One warp loads tile `tile` of operand a through the plan's TMA loads, the
// same issue path as the elementwise kernel's producer (one box per lane,
// each box on its own 1024-byte boundary, the plan's swizzle), waits on the
// stage's mbarrier and copies the slot's bytes out unchanged.  Parts of the
// slot no load writes (padding after a box, boxes wholly past the tensor's
// edge) read as zero: the slot is cleared first.  This lets a test hold the
// swizzled layout itself against its definition, where the elementwise path
// only shows it end to end (TVM docs "copy_async -> tma", "Demonstration
// program": a 128-byte swizzled shared layout read back).

#include "tsx_tma_common.cuh"

namespace tsx {
namespace {

using namespace dev;

__global__ void __launch_bounds__(32)
    tma_stage_image(const __grid_constant__ TmaMaps maps, const TmaArgs p, int64_t tile, uint4* image)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1);
    uint4* const slot = reinterpret_cast<uint4*>(smem_raw + (base - raw));
    const uint32_t bar = base + p.slot_bytes;
    const uint32_t units = p.slot_bytes / 16;
    const int lane = static_cast<int>(threadIdx.x & 31);

    for (uint32_t u = lane; u < units; u += 32)
        slot[u] = make_uint4(0, 0, 0, 0);
    if (lane == 0)
        mbar_init(bar, 1);
    // the clearing writes and the barrier's initialisation come before the
    // TMA unit's writes
    fence_proxy_async_smem();
    __syncwarp();

    const int n_loads = p.rank3 ? p.row_chunks : p.row_chunks * p.atoms;
    const BoxRef mine = box_ref(maps, p, lane < n_loads ? lane : 0, 0);
    const TileCursor tc(p, tile, 1);
    issue_tile_lanes<1>(maps, p, tc, mine, n_loads, base, bar);
    bool ok = mbar_wait(bar, 0, p.timeout_ns);
    if (!ok) {
        if (lane == 0)
            atomicCAS(p.status, TSX_OK, TSX_ERR_TIMEOUT);
        (void)mbar_wait(bar, 0, p.timeout_ns);   // bounded: let loads in flight land
    }
    __syncwarp();
    for (uint32_t u = lane; u < units; u += 32)
        image[u] = ok ? slot[u] : make_uint4(0, 0, 0, 0);
    __syncwarp();
    if (lane == 0)
        mbar_inval(bar);
}

}  // namespace

size_t stage_image_smem(const TmaArgs& args) { return size_t(args.slot_bytes) + kSmemAlign + 16; }

cudaError_t launch_stage_image(const CUtensorMap* maps, const TmaArgs& args, int64_t tile, void* image,
                               cudaStream_t stream)
{
    TmaMaps m;
    for (int j = 0; j < 4; ++j)
        m.m[j] = maps[j];
    TmaArgs a = args;
    const size_t smem = stage_image_smem(args);
    cudaError_t e = cudaFuncSetAttribute((const void*)tma_stage_image, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess)
        return e;
    uint4* img = static_cast<uint4*>(image);
    void* params[] = {&m, &a, &tile, &img};
    return cudaLaunchKernel((const void*)tma_stage_image, dim3(1), dim3(32), params, smem, stream);
}

}  // namespace tsx
