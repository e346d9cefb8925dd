// rows.cu - the two HBM-bound row movers of the MoE layer.
//
// Dispatch and combine are the expert-parallel exchange steps of the fused layer (MarkTechPost,
// "Prime Intellect Releases Prime Mega MoE", section "How does the fused kernel work?").  With
// every expert on one GPU they reduce to
//   gather  : dst[pos[t*k + j]] = src[t] for each token t and choice j, zero on the padding rows,
//   combine : out[t] = sum_j part[pos[t*k + j]], summed in fp32 in the fixed order j = 0..k-1,
// where `part` already carries the routing weight (aggregation by routing weight: kongchang.com,
// "Prime Intellect推出Prime Mega MoE", section "为什么 MoE 训练特别需要融合内核"): applied to h by the
// BF16 gate/up epilogue, to the down product's output by the MXFP8 one.  The gather moves two
// token rows per warp, the combine one token per warp, both with 16-byte accesses.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRowThreads = 256;

// The gather runs token-major: one warp reads two token rows once and stores each to its k
// dispatched rows (pos), so x is read from HBM exactly once, in order, and the stores stream out
// at the write rate.  Walking the dispatched rows in order instead reads each token row k times
// at scattered moments, and the 0.5 GB of stores streaming through L2 evict those rows between
// uses: on GB300 that walk takes 0.14 ms at the 30B size where this one takes 0.10 ms.  Units
// past the token pairs zero the padding rows (row_slot < 0), 32 rows a unit.  With a second
// source (dy beside x) the token units run once per source.
constexpr int kGatherTokens = 2;

__global__ void __launch_bounds__(kRowThreads) gather_rows_kernel(const uint4* __restrict__ src0, uint4* __restrict__ dst0,
                                                                   const uint4* __restrict__ src1, uint4* __restrict__ dst1,
                                                                   const int* __restrict__ row_slot,
                                                                   const int* __restrict__ pos,
                                                                   const int* __restrict__ mtile_total, int T, int k,
                                                                   int row_vecs) {
    grid_dep_wait();
    const int nrows = (*mtile_total) * kBM;
    const int lane = threadIdx.x & 31;
    const int wpb = kRowThreads / 32;
    const int stride = gridDim.x * wpb;
    const int tgroups = (T + kGatherTokens - 1) / kGatherTokens;
    const int tok_units = src1 ? 2 * tgroups : tgroups;
    const int units = tok_units + (nrows + 31) / 32;
    for (int u = blockIdx.x * wpb + (threadIdx.x >> 5); u < units; u += stride) {
        if (u < tok_units) {
            const bool second = u >= tgroups;
            const uint4* src = second ? src1 : src0;
            uint4* dst = second ? dst1 : dst0;
            const int t0 = (second ? u - tgroups : u) * kGatherTokens;
            int p[kGatherTokens];   // the first 32 destinations of each token, one per lane
#pragma unroll
            for (int a = 0; a < kGatherTokens; ++a)
                p[a] = (t0 + a < T && lane < k) ? pos[(size_t)(t0 + a) * k + lane] : -1;
            for (int v0 = 0; v0 < row_vecs; v0 += 256) {
                uint4 w[kGatherTokens][8];
#pragma unroll
                for (int a = 0; a < kGatherTokens; ++a) {
                    const uint4* s = src + (size_t)(t0 + a < T ? t0 + a : 0) * row_vecs;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int v = v0 + lane + 32 * q;
                        w[a][q] = (t0 + a < T && v < row_vecs) ? __ldg(s + v) : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int a = 0; a < kGatherTokens; ++a) {
                    if (t0 + a >= T) break;
                    for (int j0 = 0; j0 < k; j0 += 32) {
                        const int pj = j0 == 0 ? p[a] : (j0 + lane < k ? pos[(size_t)(t0 + a) * k + j0 + lane] : -1);
                        const int nj = min(32, k - j0);
                        for (int j = 0; j < nj; ++j) {
                            const int r = __shfl_sync(0xffffffffu, pj, j);
                            if (r < 0) continue;   // a slot with an out-of-range expert id is not dispatched
                            uint4* d = dst + (size_t)r * row_vecs;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const int v = v0 + lane + 32 * q;
                                if (v < row_vecs) __stcs(d + v, w[a][q]);
                            }
                        }
                    }
                }
            }
        } else {
            const int row0 = (u - tok_units) * 32;
            const bool pad = row0 + lane < nrows && row_slot[row0 + lane] < 0;
            unsigned m = __ballot_sync(0xffffffffu, pad);
            const uint4 z = make_uint4(0, 0, 0, 0);
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1;
                uint4* d0 = dst0 + (size_t)(row0 + b) * row_vecs;
                for (int v = lane; v < row_vecs; v += 32) d0[v] = z;
                if (dst1) {
                    uint4* d1 = dst1 + (size_t)(row0 + b) * row_vecs;
                    for (int v = lane; v < row_vecs; v += 32) d1[v] = z;
                }
            }
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
        reinterpret_cast<const int*>(c.base + L.row_slot), reinterpret_cast<const int*>(c.base + L.pos),
        reinterpret_cast<const int*>(c.base + L.mtile) + L.E, (int)L.T, (int)L.k, row_vecs);
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
