// rows.cu - the two HBM-bound row movers of the MoE layer.
//
// Dispatch and combine are the expert-parallel exchange steps of the fused layer (MarkTechPost,
// "Prime Intellect Releases Prime Mega MoE", section "How does the fused kernel work?").  With
// every expert on one GPU they reduce to
//   gather  : dst[r] = src[row_slot[r] / k] for each padded routed row r (zero on padding rows),
//   combine : out[t] = sum_j part[pos[t*k + j]], summed in fp32 in the fixed order j = 0..k-1,
// where the routing weight has already been applied to `part` by the down-projection epilogue
// (aggregation by routing weight: kongchang.com, "Prime Intellect推出Prime Mega MoE", section
// "为什么 MoE 训练特别需要融合内核").  One warp moves one row with 16-byte accesses.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) gather_rows_kernel(const uint4* __restrict__ src0, uint4* __restrict__ dst0,
                                                                   const uint4* __restrict__ src1, uint4* __restrict__ dst1,
                                                                   const int* __restrict__ row_slot,
                                                                   const int* __restrict__ mtile_total, int k,
                                                                   int row_vecs) {
    grid_dep_wait();
    const int nrows = (*mtile_total) * kBM;
    const int wpb = kRowThreads / 32;
    const int lane = threadIdx.x & 31;
    const int stride = gridDim.x * wpb;
    for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < nrows; r += stride) {
        const int slot = row_slot[r];
        uint4* d0 = dst0 + (size_t)r * row_vecs;
        uint4* d1 = dst1 ? dst1 + (size_t)r * row_vecs : nullptr;
        if (slot >= 0) {
            const size_t t = (size_t)(slot / k);
            const uint4* s0 = src0 + t * row_vecs;
            const uint4* s1 = src1 ? src1 + t * row_vecs : nullptr;
            int v = lane;
            for (; v + 96 < row_vecs; v += 128) {
                const uint4 a = __ldg(s0 + v), b = __ldg(s0 + v + 32), c = __ldg(s0 + v + 64), d = __ldg(s0 + v + 96);
                d0[v] = a; d0[v + 32] = b; d0[v + 64] = c; d0[v + 96] = d;
            }
            for (; v < row_vecs; v += 32) d0[v] = __ldg(s0 + v);
            if (s1) {
                v = lane;
                for (; v + 96 < row_vecs; v += 128) {
                    const uint4 a = __ldg(s1 + v), b = __ldg(s1 + v + 32), c = __ldg(s1 + v + 64), d = __ldg(s1 + v + 96);
                    d1[v] = a; d1[v + 32] = b; d1[v + 64] = c; d1[v + 96] = d;
                }
                for (; v < row_vecs; v += 32) d1[v] = __ldg(s1 + v);
            }
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int v = lane; v < row_vecs; v += 32) d0[v] = z;
            if (d1)
                for (int v = lane; v < row_vecs; v += 32) d1[v] = z;
        }
    }
}

// One warp per token.  Each lane owns 8 consecutive columns of every 256-column chunk and takes
// two such chunks at a time, loading four routed rows of both before summing them (8 loads of 16
// bytes in flight per lane, at 64 registers so that 64 warps stay resident: the kernel is bound
// by memory latency).  Each output sums its k rows in the fixed order j = 0..k-1 in fp32.
__device__ __forceinline__ void add_bf16x8(float* acc, uint4 w) {
    const float2 a = unpack_bf16x2(w.x), b = unpack_bf16x2(w.y), c = unpack_bf16x2(w.z), d = unpack_bf16x2(w.w);
    acc[0] += a.x; acc[1] += a.y; acc[2] += b.x; acc[3] += b.y;
    acc[4] += c.x; acc[5] += c.y; acc[6] += d.x; acc[7] += d.y;
}
__device__ __forceinline__ uint4 pack_bf16x8(const float* acc) {
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    return o;
}

__global__ void __launch_bounds__(kRowThreads, 4) combine_rows_kernel(const uint4* __restrict__ part, uint4* __restrict__ out,
                                                                    const int* __restrict__ pos, int T, int k,
                                                                    int row_vecs, const float* __restrict__ dtw,
                                                                    int n_dtw, float* __restrict__ dtopk_w) {
    grid_dep_wait();
    constexpr int kBatch = 4;   // routed rows loaded per batch (for each of the two chunks)
    const int wpb = kRowThreads / 32;
    const int lane = threadIdx.x & 31;
    const int stride = gridDim.x * wpb;
    for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += stride) {
        const int* pt = pos + (size_t)t * k;
        for (int v0 = lane; v0 < row_vecs; v0 += 64) {
            const int v1 = v0 + 32;
            const bool two = v1 < row_vecs;
            float acc0[8], acc1[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc0[q] = acc1[q] = 0.f;
            for (int j0 = 0; j0 < k; j0 += kBatch) {
                uint4 w0[kBatch], w1[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int p = j0 + u < k ? pt[j0 + u] : -1;
                    const uint4* r = part + (size_t)(p >= 0 ? p : 0) * row_vecs;
                    w0[u] = p >= 0 ? __ldg(r + v0) : make_uint4(0, 0, 0, 0);
                    w1[u] = (p >= 0 && two) ? __ldg(r + v1) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (j0 + u < k) {
                        add_bf16x8(acc0, w0[u]);
                        add_bf16x8(acc1, w1[u]);
                    }
                }
            }
            out[(size_t)t * row_vecs + v0] = pack_bf16x8(acc0);
            if (two) out[(size_t)t * row_vecs + v1] = pack_bf16x8(acc1);
        }
        if (dtopk_w) {
            for (int j = lane; j < k; j += 32) {
                const int p = pt[j];
                float s = 0.f;
                if (p >= 0)
                    for (int n = 0; n < n_dtw; ++n) s += dtw[(size_t)p * n_dtw + n];
                dtopk_w[(size_t)t * k + j] = s;
            }
        }
    }
}

// y = bf16(acc) over the fused combine's fp32 [T, H] accumulator, 8 values per thread and step
__global__ void __launch_bounds__(kRowThreads) reduce_finish_kernel(const float4* __restrict__ acc,
                                                                     uint4* __restrict__ out, long long n8) {
    grid_dep_wait();
    for (long long i = (long long)blockIdx.x * kRowThreads + threadIdx.x; i < n8;
         i += (long long)gridDim.x * kRowThreads) {
        const float4 a = __ldg(acc + 2 * i), b = __ldg(acc + 2 * i + 1);
        out[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                            pack_bf16x2(b.z, b.w));
    }
}

static int row_grid(const Ctx& c) { return c.num_sms * 8; }

cudaError_t launch_reduce_zero(const Ctx& c) {
    const Layout& L = *c.L;
    return cudaMemsetAsync(c.base + L.ypart, 0, (size_t)L.T * L.H * 4, c.st);
}

cudaError_t launch_reduce_finish(const Ctx& c, void* y) {
    const Layout& L = *c.L;
    trace_begin(c.st, kTraceReduceFinish);
    const cudaError_t err = launch_pdl(reduce_finish_kernel, row_grid(c), kRowThreads, 0, c.st,
                                       reinterpret_cast<const float4*>(c.base + L.ypart), reinterpret_cast<uint4*>(y),
                                       (long long)(L.T * L.H / 8));
    trace_end(c.st, kTraceReduceFinish);
    return err;
}

cudaError_t launch_gather(const Ctx& c, const void* src0, void* dst0, const void* src1, void* dst1) {
    const Layout& L = *c.L;
    const int row_vecs = (int)(L.H * 2 / 16);
    trace_begin(c.st, kTraceGather);
    const cudaError_t err = launch_pdl(
        gather_rows_kernel, row_grid(c), kRowThreads, 0, c.st, reinterpret_cast<const uint4*>(src0),
        reinterpret_cast<uint4*>(dst0), reinterpret_cast<const uint4*>(src1), reinterpret_cast<uint4*>(dst1),
        reinterpret_cast<const int*>(c.base + L.row_slot), reinterpret_cast<const int*>(c.base + L.mtile) + L.E,
        (int)L.k, row_vecs);
    trace_end(c.st, kTraceGather);
    return err;
}

cudaError_t launch_combine(const Ctx& c, const void* part, void* out, float* dtopk_w) {
    const Layout& L = *c.L;
    const int row_vecs = (int)(L.H * 2 / 16);
    trace_begin(c.st, kTraceCombine);
    const cudaError_t err = launch_pdl(
        combine_rows_kernel, row_grid(c), kRowThreads, 0, c.st, reinterpret_cast<const uint4*>(part),
        reinterpret_cast<uint4*>(out), reinterpret_cast<const int*>(c.base + L.pos), (int)L.T, (int)L.k, row_vecs,
        reinterpret_cast<const float*>(c.base + L.dtw), (int)L.n_dtw, dtopk_w);
    trace_end(c.st, kTraceCombine);
    return err;
}

}  // namespace moe
