// routing.cu - routing bookkeeping of the MoE layer: per-expert token counts, the exclusive
// prefix of the counts (group offsets), and a stable token reorder with its inverse.
//
// Grouping the routed tokens by expert and indexing every group by its offset is the grouped-GEMM
// set-up the pages describe (kongchang.com, "Prime Intellect推出Prime Mega MoE", section
// "为什么 MoE 训练特别需要融合内核": group offsets, routing index, token reorder).  The order inside
// a group is slot order s = t*k + j, which makes the reorder unique.
//
// Three launches, no host synchronisation:
//   route_hist  : block b counts the experts of its chunk of slots into hist[b][e];
//   route_scan  : one block sums hist over b (counts), scans them into offsets, padded offsets
//                 (each group rounded up to a 128-row GEMM tile), the m-tile prefix and the
//                 per-block starting positions base[b][e]; it also ranks the experts by count;
//   route_place : block b walks its chunk in slot order and places every slot at
//                 base[b][e] + (slots of e earlier in the chunk), ranking ties inside a warp with
//                 __match_any_sync and across the block's warps with per-warp counts.
// Expert ids outside [0, E) are never used as an index: they are counted nowhere, recorded as
// MOE_DEV_BAD_EXPERT in the status word (when there is one), their slots get inv = pos = -1, and
// the sorted positions they leave free, [offsets[E], T*k), hold perm = -1.
// The padded-layout outputs (pad_off, mtile, order, pos, row_slot) and the status word are
// optional: the allocation-free entry point (route_static.cu) runs the same kernels without them.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRouteThreads = 256;   // route_hist
constexpr int kPlaceThreads = 512;   // route_place: a 2048-slot chunk in four rounds

__global__ void __launch_bounds__(kRouteThreads) route_hist_kernel(const int32_t* __restrict__ idx, int S, int E,
                                                                    int* __restrict__ hist, int* status) {
    grid_dep_wait();
    extern __shared__ int sh_cnt[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh_cnt[e] = 0;
    __syncthreads();
    const int s0 = blockIdx.x * kRouteChunk, s1 = min(S, s0 + kRouteChunk);
    for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
        const int e = idx[s];
        if ((unsigned)e < (unsigned)E)
            atomicAdd(&sh_cnt[e], 1);
        else
            set_status(status, MOE_DEV_BAD_EXPERT);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh_cnt[e];
}

// Inclusive scan over the 1024 threads of a block (value per thread).
__device__ int block_inclusive_scan(int v, int* sh_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
    __syncthreads();
    return v;
}

__global__ void __launch_bounds__(1024) route_scan_kernel(const int* __restrict__ hist, int nb, int E,
                                                           int* __restrict__ cnt, int* __restrict__ off,
                                                           int* __restrict__ pad_off, int* __restrict__ mtile,
                                                           int* __restrict__ order, int* __restrict__ base) {
    grid_dep_wait();
    __shared__ int sh_cnt[kMaxExperts];
    __shared__ int sh_warp[32];
    const int e = threadIdx.x;
    int c = 0;
    if (e < E)
        for (int b = 0; b < nb; ++b) c += hist[(size_t)b * E + e];
    sh_cnt[e] = c;
    const int tiles = (c + kBM - 1) / kBM;
    const int c_incl = block_inclusive_scan(c, sh_warp);
    const int t_incl = block_inclusive_scan(tiles, sh_warp);
    if (e < E) {
        cnt[e] = c;
        off[e] = c_incl - c;
        if (e == E - 1) off[E] = c_incl;
        if (pad_off) {
            mtile[e] = t_incl - tiles;
            pad_off[e] = (t_incl - tiles) * kBM;
            if (e == E - 1) {
                mtile[E] = t_incl;
                pad_off[E] = t_incl * kBM;
            }
        }
        int run = c_incl - c;
        for (int b = 0; b < nb; ++b) {
            base[(size_t)b * E + e] = run;
            run += hist[(size_t)b * E + e];
        }
        if (order) {
            // rank by count, largest first, ties by expert id (used to order weight-gradient tiles)
            int rank = 0;
            for (int f = 0; f < E; ++f) {
                const int cf = sh_cnt[f];
                rank += (cf > c) || (cf == c && f < e);
            }
            order[rank] = e;
        }
    }
}

__global__ void __launch_bounds__(kPlaceThreads) route_place_kernel(
    const int32_t* __restrict__ idx, int S, int E, const int* __restrict__ base, const int* __restrict__ off,
    const int* __restrict__ pad_off, const int* __restrict__ cnt, int* __restrict__ perm, int* __restrict__ inv,
    int* __restrict__ pos, int* __restrict__ row_slot) {
    grid_dep_wait();
    constexpr int kWarps = kPlaceThreads / 32;
    extern __shared__ int sh[];
    int* ctr = sh;          // [E]   next sorted position of each expert for this block
    int* wc = sh + E;       // [kWarps][E] per-warp counts of the current round
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < E; e += kPlaceThreads) ctr[e] = base[(size_t)blockIdx.x * E + e];
    for (int i = tid; i < kWarps * E; i += kPlaceThreads) wc[i] = 0;
    __syncthreads();
    const int s0 = blockIdx.x * kRouteChunk, s1 = min(S, s0 + kRouteChunk);
    for (int r0 = s0; r0 < s1; r0 += kPlaceThreads) {
        const int s = r0 + tid;
        const bool valid = s < s1;
        const int e = valid ? idx[s] : -1;
        const bool ok = valid && (unsigned)e < (unsigned)E;
        const int key = ok ? e : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (ok && lane == __ffs(peers) - 1) wc[warp * E + e] = __popc(peers);
        __syncthreads();
        if (ok) {
            int before = 0;
            for (int w = 0; w < warp; ++w) before += wc[w * E + e];
            const int p = ctr[e] + before + rank;
            perm[p] = s;
            inv[s] = p;
            if (pos) {
                const int pp = p - off[e] + pad_off[e];
                pos[s] = pp;
                row_slot[pp] = s;
            }
        } else if (valid) {
            inv[s] = -1;
            if (pos) pos[s] = -1;
        }
        __syncthreads();
        for (int f = tid; f < E; f += kPlaceThreads) {
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
    // sorted positions left free by dropped slots (none for valid ids)
    for (int p = off[E] + blockIdx.x * kPlaceThreads + tid; p < S; p += gridDim.x * kPlaceThreads) perm[p] = -1;
    // padding rows of the groups this block owns
    if (row_slot) {
        for (int f = blockIdx.x; f < E; f += gridDim.x) {
            const int lo = pad_off[f] + cnt[f], hi = pad_off[f + 1];
            for (int r = lo + tid; r < hi; r += kPlaceThreads) row_slot[r] = -1;
        }
    }
}

cudaError_t launch_routing_kernels(cudaStream_t st, const int32_t* topk_idx, int S, int E, const RoutingBufs& r,
                                   int* status) {
    const int nb = (S + kRouteChunk - 1) / kRouteChunk;
    cudaError_t err = cudaSuccess;
    if (nb > 0) {
        trace_begin(st, kTraceRouteHist);
        err = launch_pdl(route_hist_kernel, nb, kRouteThreads, E * sizeof(int), st, topk_idx, S, E, r.hist, status);
        trace_end(st, kTraceRouteHist);
    }
    if (err != cudaSuccess) return err;
    trace_begin(st, kTraceRouteScan);
    err = launch_pdl(route_scan_kernel, 1, 1024, 0, st, (const int*)r.hist, nb, E, r.cnt, r.off, r.pad_off, r.mtile,
                     r.order, r.base);
    trace_end(st, kTraceRouteScan);
    if (err != cudaSuccess) return err;
    if (nb > 0) {
        trace_begin(st, kTraceRoutePlace);
        const size_t sm = (size_t)(E + (kPlaceThreads / 32) * E) * sizeof(int);
        static std::once_flag once;
        static cudaError_t attr_err = cudaSuccess;
        std::call_once(once, [] {
            attr_err = cudaFuncSetAttribute(route_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)((kMaxExperts + (kPlaceThreads / 32) * kMaxExperts) * sizeof(int)));
        });
        if (attr_err != cudaSuccess) return attr_err;
        err = launch_pdl(route_place_kernel, nb, kPlaceThreads, sm, st, topk_idx, S, E, (const int*)r.base,
                         (const int*)r.off, (const int*)r.pad_off, (const int*)r.cnt, r.perm, r.inv, r.pos, r.row_slot);
        trace_end(st, kTraceRoutePlace);
    }
    return err;
}

cudaError_t launch_routing(const Ctx& c, const int32_t* topk_idx) {
    const Layout& L = *c.L;
    auto at = [&](size_t off) { return reinterpret_cast<int*>(c.base + off); };
    const RoutingBufs r{at(L.hist), at(L.base), at(L.cnt), at(L.off), at(L.pad_off), at(L.mtile),
                        at(L.order),  at(L.perm), at(L.inv), at(L.pos), at(L.row_slot)};
    return launch_routing_kernels(c.st, topk_idx, (int)L.S, (int)L.E, r, c.status);
}

}  // namespace moe
