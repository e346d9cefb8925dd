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
// MOE_DEV_BAD_EXPERT in the status word, and their slots get inv = pos = -1.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRouteThreads = 256;

__global__ void __launch_bounds__(kRouteThreads) route_hist_kernel(const int32_t* __restrict__ idx, int S, int E,
                                                                    int* __restrict__ hist, int* status) {
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
        mtile[e] = t_incl - tiles;
        pad_off[e] = (t_incl - tiles) * kBM;
        if (e == E - 1) {
            off[E] = c_incl;
            mtile[E] = t_incl;
            pad_off[E] = t_incl * kBM;
        }
        int run = c_incl - c;
        for (int b = 0; b < nb; ++b) {
            base[(size_t)b * E + e] = run;
            run += hist[(size_t)b * E + e];
        }
        // rank by count, largest first, ties by expert id (used to order weight-gradient tiles)
        int rank = 0;
        for (int f = 0; f < E; ++f) {
            const int cf = sh_cnt[f];
            rank += (cf > c) || (cf == c && f < e);
        }
        order[rank] = e;
    }
}

__global__ void __launch_bounds__(kRouteThreads) route_place_kernel(
    const int32_t* __restrict__ idx, int S, int E, const int* __restrict__ base, const int* __restrict__ off,
    const int* __restrict__ pad_off, const int* __restrict__ cnt, int* __restrict__ perm, int* __restrict__ inv,
    int* __restrict__ pos, int* __restrict__ row_slot) {
    constexpr int kWarps = kRouteThreads / 32;
    extern __shared__ int sh[];
    int* ctr = sh;          // [E]   next sorted position of each expert for this block
    int* wc = sh + E;       // [kWarps][E] per-warp counts of the current round
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < E; e += kRouteThreads) ctr[e] = base[(size_t)blockIdx.x * E + e];
    for (int i = tid; i < kWarps * E; i += kRouteThreads) wc[i] = 0;
    __syncthreads();
    const int s0 = blockIdx.x * kRouteChunk, s1 = min(S, s0 + kRouteChunk);
    for (int r0 = s0; r0 < s1; r0 += kRouteThreads) {
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
            const int pp = p - off[e] + pad_off[e];
            perm[p] = s;
            inv[s] = p;
            pos[s] = pp;
            row_slot[pp] = s;
        } else if (valid) {
            inv[s] = -1;
            pos[s] = -1;
        }
        __syncthreads();
        for (int f = tid; f < E; f += kRouteThreads) {
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
    // padding rows of the groups this block owns
    for (int f = blockIdx.x; f < E; f += gridDim.x) {
        const int lo = pad_off[f] + cnt[f], hi = pad_off[f + 1];
        for (int r = lo + tid; r < hi; r += kRouteThreads) row_slot[r] = -1;
    }
}

cudaError_t launch_routing(const Ctx& c, const int32_t* topk_idx) {
    const Layout& L = *c.L;
    int* hist = reinterpret_cast<int*>(c.base + L.hist);
    int* cnt = reinterpret_cast<int*>(c.base + L.cnt);
    int* off = reinterpret_cast<int*>(c.base + L.off);
    int* pad_off = reinterpret_cast<int*>(c.base + L.pad_off);
    int* mtile = reinterpret_cast<int*>(c.base + L.mtile);
    int* order = reinterpret_cast<int*>(c.base + L.order);
    int* base = reinterpret_cast<int*>(c.base + L.base);
    const int S = (int)L.S, E = (int)L.E, nb = (int)L.nb_route;
    if (nb > 0) {
        trace_begin(c.st, kTraceRouteHist);
        route_hist_kernel<<<nb, kRouteThreads, E * sizeof(int), c.st>>>(topk_idx, S, E, hist, c.status);
        trace_end(c.st, kTraceRouteHist);
    }
    trace_begin(c.st, kTraceRouteScan);
    route_scan_kernel<<<1, 1024, 0, c.st>>>(hist, nb, E, cnt, off, pad_off, mtile, order, base);
    trace_end(c.st, kTraceRouteScan);
    if (nb > 0) {
        trace_begin(c.st, kTraceRoutePlace);
        const size_t sm = (size_t)(E + 8 * E) * sizeof(int);
        route_place_kernel<<<nb, kRouteThreads, sm, c.st>>>(
            topk_idx, S, E, base, off, pad_off, cnt, reinterpret_cast<int*>(c.base + L.perm),
            reinterpret_cast<int*>(c.base + L.inv), reinterpret_cast<int*>(c.base + L.pos),
            reinterpret_cast<int*>(c.base + L.row_slot));
        trace_end(c.st, kTraceRoutePlace);
    }
    return cudaGetLastError();
}

}  // namespace moe
