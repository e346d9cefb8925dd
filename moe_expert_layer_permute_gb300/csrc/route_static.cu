// route_static.cu - the routing bookkeeping (per-expert counts, group offsets, stable token
// reorder and its inverse) for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a scratch buffer: code that runs inside
// a memory allocator's own hooks, runtimes that reserve all device memory up front and forbid
// later allocations, or latency-critical loops where an allocation would synchronise the device.
// moe_route_static serves them: it needs only its inputs and outputs.  The per-block histograms
// and per-block starting positions that the routing kernels need live in a file-scope
// `static __device__` array of kStaticRouteInts 32-bit integers (256 KiB), which every GPU that
// loads this library holds until the process exits.
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
constexpr int kStaticThreads = 256;
constexpr int kStaticChunk = 2048;       // slots per block

static __device__ __align__(256) int g_route_static_scratch[kStaticRouteInts];

__global__ void __launch_bounds__(kStaticThreads) route_static_hist(const int32_t* __restrict__ idx, int S, int E,
                                                                     int* __restrict__ hist) {
    extern __shared__ int sh_cnt[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh_cnt[e] = 0;
    __syncthreads();
    const int s0 = blockIdx.x * kStaticChunk, s1 = min(S, s0 + kStaticChunk);
    for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
        const int e = idx[s];
        if ((unsigned)e < (unsigned)E) atomicAdd(&sh_cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh_cnt[e];
}

// one block of 1024 threads, thread e owns expert e
__global__ void __launch_bounds__(1024) route_static_scan(const int* __restrict__ hist, int nb, int E,
                                                           int* __restrict__ cnt, int* __restrict__ off,
                                                           int* __restrict__ base) {
    __shared__ int sh_warp[32];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    int c = 0;
    if (e < E)
        for (int b = 0; b < nb; ++b) c += hist[(size_t)b * E + e];
    int v = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) sh_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = sh_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        sh_warp[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += sh_warp[warp - 1];
    if (e < E) {
        cnt[e] = c;
        off[e] = v - c;
        if (e == E - 1) off[E] = v;
        int run = v - c;
        for (int b = 0; b < nb; ++b) {
            base[(size_t)b * E + e] = run;
            run += hist[(size_t)b * E + e];
        }
    }
}

__global__ void __launch_bounds__(kStaticThreads) route_static_place(const int32_t* __restrict__ idx, int S, int E,
                                                                      const int* __restrict__ base,
                                                                      int* __restrict__ perm, int* __restrict__ inv) {
    constexpr int kWarps = kStaticThreads / 32;
    extern __shared__ int sh[];
    int* ctr = sh;
    int* wc = sh + E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < E; e += kStaticThreads) ctr[e] = base[(size_t)blockIdx.x * E + e];
    for (int i = tid; i < kWarps * E; i += kStaticThreads) wc[i] = 0;
    __syncthreads();
    const int s0 = blockIdx.x * kStaticChunk, s1 = min(S, s0 + kStaticChunk);
    for (int r0 = s0; r0 < s1; r0 += kStaticThreads) {
        const int s = r0 + tid;
        const bool valid = s < s1;
        const int e = valid ? idx[s] : -1;
        const bool ok = valid && (unsigned)e < (unsigned)E;
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (ok && lane == __ffs(peers) - 1) wc[warp * E + e] = __popc(peers);
        __syncthreads();
        if (ok) {
            int before = 0;
            for (int w = 0; w < warp; ++w) before += wc[w * E + e];
            const int p = ctr[e] + before + rank;
            perm[p] = s;
            inv[s] = p;
        } else if (valid) {
            inv[s] = -1;
        }
        __syncthreads();
        for (int f = tid; f < E; f += kStaticThreads) {
            int add = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                add += wc[w * E + f];
                wc[w * E + f] = 0;
            }
            ctr[f] += add;
        }
        __syncthreads();
    }
}

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
    const int64_t nb = (S + kStaticChunk - 1) / kStaticChunk;
    if (2 * nb * E > kStaticRouteInts) return MOE_ERR_UNSUPPORTED;  // beyond the static array
    if (!counts || !offsets || (S > 0 && (!topk_idx || !perm || !inv))) return MOE_ERR_NULL;
    for (const void* p : {(const void*)topk_idx, (const void*)counts, (const void*)offsets, (const void*)perm,
                          (const void*)inv})
        if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return MOE_ERR_ALIGN;
    int* scratch = nullptr;
    const int rc = static_scratch_address(&scratch);
    if (rc) return rc;
    int* hist = scratch;
    int* base = scratch + nb * E;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (nb > 0) route_static_hist<<<(int)nb, kStaticThreads, E * sizeof(int), st>>>(topk_idx, (int)S, (int)E, hist);
    route_static_scan<<<1, 1024, 0, st>>>(hist, (int)nb, (int)E, counts, offsets, base);
    if (nb > 0)
        route_static_place<<<(int)nb, kStaticThreads, (size_t)9 * E * sizeof(int), st>>>(topk_idx, (int)S, (int)E,
                                                                                        base, perm, inv);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
