// route_static.cu - the routing bookkeeping (per-expert counts, group offsets, stable token
// reorder and its inverse) for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a scratch buffer: code that runs inside
// a memory allocator's own hooks, runtimes that reserve all device memory up front and forbid
// later allocations, or latency-critical loops where an allocation would synchronise the device.
// moe_route_static serves them: it needs only its inputs and outputs.  It runs the routing kernels
// of routing.cu (the ones moe_fwd runs), without the padded row layout; the per-block histograms
// and per-block starting positions they need live in a file-scope `static __device__` array of
// kStaticRouteInts 32-bit integers (256 KiB), which every GPU that loads this library holds until
// the process exits.
//
// The host never uses the array's name as an address (on the host it only names a stand-in):
// the first call on each device, with that device current, looks up the device address once with
// cudaGetSymbolAddress and caches it; that first call should therefore come before any stream
// capture.  All calls share the one array and it keeps the last call's contents; every word a
// call reads is first written by that same call, so nothing needs clearing, but two calls whose
// kernels overlap on the GPU (different streams without ordering) race on the array.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kStaticRouteInts = 65536;  // 256 KiB: hist[nb][E] followed by base[nb][E]

static __device__ __align__(256) int g_route_static_scratch[kStaticRouteInts];

// Device address of the static array on the current device, looked up once per device.
static int static_scratch_address(int** out) {
    static std::mutex mu;
    static int* addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        addr[dev] = static_cast<int*>(p);
    }
    *out = addr[dev];
    return MOE_OK;
}

}  // namespace moe

extern "C" int moe_route_static(const int32_t* topk_idx, int64_t T, int64_t k, int64_t E, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* inv, void* stream) {
    using namespace moe;
    if (T < 0 || k < 1 || E < 1 || k > E || E > kMaxExperts) return MOE_ERR_SHAPE;
    const int64_t S = T * k;
    if (S >= (int64_t)INT32_MAX / 2) return MOE_ERR_SHAPE;
    const int64_t nb = (S + kRouteChunk - 1) / kRouteChunk;
    if (2 * nb * E > kStaticRouteInts) return MOE_ERR_UNSUPPORTED;  // beyond the static array
    if (!counts || !offsets || (S > 0 && (!topk_idx || !perm || !inv))) return MOE_ERR_NULL;
    for (const void* p : {(const void*)topk_idx, (const void*)counts, (const void*)offsets, (const void*)perm,
                          (const void*)inv})
        if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return MOE_ERR_ALIGN;
    int* scratch = nullptr;
    const int rc = static_scratch_address(&scratch);
    if (rc) return rc;
    // the same kernels as moe_fwd's routing, without the padded row layout and the status word
    const RoutingBufs r{scratch, scratch + nb * E, counts, offsets, nullptr, nullptr, nullptr, perm, inv, nullptr,
                        nullptr};
    if (launch_routing_kernels(reinterpret_cast<cudaStream_t>(stream), topk_idx, (int)S, (int)E, r, nullptr) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
