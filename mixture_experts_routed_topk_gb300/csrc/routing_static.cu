// routing_static.cu -- moe_routing_static_scratch: the routing stage (histogram, scan, stable
// permutation) with its per-block scratch in a fixed device array that this library owns, for
// callers that cannot allocate a routing workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds it until
// the process exits. Host code cannot use the array's name as a device address, so every call looks
// the address up with cudaGetSymbolAddress on the current device. Nothing is cached: after a device
// reset the library's device code is loaded again and the array may sit at another address. The
// first lookup on a device may load the library's device code, which is why a caller makes its
// first call on a device before any stream capture; later lookups are plain host queries.
#include <cuda_runtime.h>

#include "moe_internal.cuh"

// [0, 64) status slot | [64, 64 + N) per-block counts | [64 + N, 64 + 2N) per-block first rows,
// N = MOE_STATIC_SCRATCH_MAX_ENTRIES (2 MiB + 256 bytes in all)
static __device__ __align__(256) int32_t g_routing_scratch[64 + 2 * MOE_STATIC_SCRATCH_MAX_ENTRIES];

namespace moe {
namespace {

constexpr int64_t kStaticEntries = MOE_STATIC_SCRATCH_MAX_ENTRIES;
constexpr int64_t kStatusSlotInts = 64;  // 256 bytes: a status word for callers that pass none

// The array's device address on the current device, looked up afresh by every call.
moe_status_t scratch_address(int32_t** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_routing_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    *out = static_cast<int32_t*>(p);
    return MOE_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_routing_static_scratch(const int32_t* topk_ids, int64_t T, int32_t E, int32_t K,
                                                   int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                                   uint32_t* device_status, moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || E <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t R = T * static_cast<int64_t>(K);
    if (T > 0 && R / K != T) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (R >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    const int64_t nblk = ceil_div(R, kRouteChunk);
    if (static_cast<int64_t>(E + 1) * nblk > kStaticEntries) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!topk_ids || !counts || !offsets || !perm || !inv) return MOE_ERR_INVALID_ARG;
    if (!aligned4(topk_ids) || !aligned4(counts) || !aligned4(offsets) || !aligned4(perm) || !aligned4(inv) ||
        !aligned4(device_status))
        return MOE_ERR_MISALIGNED;

    DeviceInfo dev;
    moe_status_t st = device_info(&dev);
    if (st != MOE_OK) return st;
    if (!dev.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
    int32_t* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != MOE_OK) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t* status = device_status ? device_status : reinterpret_cast<uint32_t*>(scratch);
    // the array keeps the previous call's contents: the status word must start at zero; the
    // per-block counts and first rows are fully rewritten by every call
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    RoutingBuffers b{};
    b.ids = topk_ids;
    b.R = R;
    b.E = E;
    b.nblk = static_cast<int>(nblk);
    b.block_counts = scratch + kStatusSlotInts;
    b.block_bases = scratch + kStatusSlotInts + kStaticEntries;
    b.counts = counts;
    b.offsets = offsets;
    b.perm = perm;
    b.inv = inv;
    b.status = status;
    return launch_routing(b, s);
}
