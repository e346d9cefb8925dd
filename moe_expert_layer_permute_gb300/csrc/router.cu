// router.cu - the top-k router that precedes the MoE layer, forward and backward.
//
// The pages' single-layer benchmark leaves the router out (ic.work analysis, section
// "跑分背后的理想假设与闭源软肋"); its output is what the layer consumes, each token's k experts and
// the routing weights that aggregate their outputs (kongchang.com, "Prime Intellect推出Prime Mega
// MoE", section "为什么 MoE 训练特别需要融合内核").  Readings where the pages are silent: the k
// largest logits are selected, ties to the lower expert index, listed in descending order; the
// weights are the softmax over the selected logits; the backward reaches the selected logits only:
//   dlogits[t, e_j] = w_j (dw_j - sum_i w_i dw_i), zero elsewhere.
//
// One warp per token.  The forward holds the token's logits as order-preserving integer keys,
// ceil(E / 32) per lane, and runs k rounds of two warp reductions: the largest remaining key
// (__reduce_max_sync), then the lowest expert index holding it (__reduce_min_sync).  The winners
// end on lanes 0..k-1, which form the softmax in fp32 and write the outputs.  Every comparison is
// exact, so the indices match any exact implementation bit for bit.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRouterWarps = 8;   // tokens per block

// float -> uint32 whose unsigned order is the float order (finite values and infinities); -0.0
// and +0.0 are equal logits and get the same key
__device__ __forceinline__ uint32_t ordered_key(float v) {
    if (v == 0.f) v = 0.f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// C: logits per lane, E <= 32 C
template <int C>
__global__ void __launch_bounds__(32 * kRouterWarps) router_fwd_kernel(const float* __restrict__ logits, int T, int E,
                                                                       int k, int* __restrict__ topk_idx,
                                                                       float* __restrict__ topk_w) {
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const long long t = (long long)blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + t * E;
    uint32_t key[C];
    uint32_t taken = 0;   // bit c: expert lane + 32 c is selected or does not exist
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int e = lane + 32 * c;
        key[c] = e < E ? ordered_key(__ldg(row + e)) : 0u;
        if (e >= E) taken |= 1u << c;
    }
    int sel_e = 0;
    float sel_v = 0.f;
    for (int r = 0; r < k; ++r) {
        // this lane's largest untaken key, at its lowest index (c ascends with the expert index)
        uint32_t bk = 0;
        int bc = -1;
#pragma unroll
        for (int c = 0; c < C; ++c)
            if (!((taken >> c) & 1u) && (bc < 0 || key[c] > bk)) {
                bk = key[c];
                bc = c;
            }
        // the warp's largest key, then the lowest expert holding it (k <= E: some lane has one)
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bc >= 0 ? bk : 0u);
        const uint32_t e = __reduce_min_sync(0xffffffffu, (bc >= 0 && bk == kmax) ? (uint32_t)(lane + 32 * bc) : 0xffffffffu);
        if ((int)(e & 31) == lane) taken |= 1u << (e >> 5);
        if (lane == r) {
            sel_e = (int)e;
            sel_v = key_value(kmax);
        }
    }
    const float m = __shfl_sync(0xffffffffu, sel_v, 0);   // the largest selected logit
    const float z = lane < k ? expf(sel_v - m) : 0.f;
    const float s = warp_sum(z);
    if (lane < k) {
        topk_idx[t * k + lane] = sel_e;
        topk_w[t * k + lane] = z / s;
    }
}

__global__ void __launch_bounds__(32 * kRouterWarps) router_bwd_kernel(const int* __restrict__ topk_idx,
                                                                       const float* __restrict__ topk_w,
                                                                       const float* __restrict__ dtopk_w, int T, int E,
                                                                       int k, float* __restrict__ dlogits) {
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const long long t = (long long)blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int e = -1;
    float w = 0.f, dw = 0.f;
    if (lane < k) {
        e = __ldg(topk_idx + t * k + lane);
        w = __ldg(topk_w + t * k + lane);
        dw = __ldg(dtopk_w + t * k + lane);
    }
    const float dot = warp_sum(w * dw);
    float* row = dlogits + t * E;
    for (int c = lane; c < E; c += 32) row[c] = 0.f;
    __syncwarp();   // the zeros are ordered before the selected experts' values
    if (lane < k && e >= 0 && e < E) row[e] = w * (dw - dot);
}

template <int C>
static cudaError_t fwd_c(cudaStream_t st, const float* logits, int T, int E, int k, int* idx, float* w) {
    const int blocks = (T + kRouterWarps - 1) / kRouterWarps;
    return launch_pdl(router_fwd_kernel<C>, blocks, 32 * kRouterWarps, 0, st, logits, T, E, k, idx, w);
}

cudaError_t launch_router_fwd(cudaStream_t st, const float* logits, int T, int E, int k, int* topk_idx,
                              float* topk_w) {
    if (T == 0) return cudaSuccess;
    const int c = (E + 31) / 32;
    if (c <= 1) return fwd_c<1>(st, logits, T, E, k, topk_idx, topk_w);
    if (c <= 2) return fwd_c<2>(st, logits, T, E, k, topk_idx, topk_w);
    if (c <= 4) return fwd_c<4>(st, logits, T, E, k, topk_idx, topk_w);
    if (c <= 8) return fwd_c<8>(st, logits, T, E, k, topk_idx, topk_w);
    if (c <= 16) return fwd_c<16>(st, logits, T, E, k, topk_idx, topk_w);
    return fwd_c<32>(st, logits, T, E, k, topk_idx, topk_w);
}

cudaError_t launch_router_bwd(cudaStream_t st, const int* topk_idx, const float* topk_w, const float* dtopk_w, int T,
                              int E, int k, float* dlogits) {
    if (T == 0) return cudaSuccess;
    const int blocks = (T + kRouterWarps - 1) / kRouterWarps;
    return launch_pdl(router_bwd_kernel, blocks, 32 * kRouterWarps, 0, st, topk_idx, topk_w, dtopk_w, T, E, k,
                      dlogits);
}

}  // namespace moe
