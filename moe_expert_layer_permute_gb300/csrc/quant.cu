// quant.cu - MXFP8 quantiser: bf16 [R, C] -> E4M3 values with one E8M0 scale per 32 elements.
//
// MXFP8 operands (Blackwell only, per ic.work analysis, section "算子下沉时代的硬件死锁暗礁") follow
// the OCP Microscaling v1.0 rule: a block of 32 values shares the exponent
// floor(log2(amax)) - 8 (8 = the largest E4M3 exponent), stored biased by 127 in one byte; each
// value is divided by 2^exp, rounded to the nearest E4M3 value (ties to even) and saturated to
// +-448.  A block whose amax is 0 gets scale byte 0 and zero values.
//
// One pass reads a 32 x 128 tile of bf16 and can emit both blockings:
//   row blocks: 32 consecutive columns of a row (the contraction axis of a K-major operand);
//   col blocks: 32 consecutive rows of a column (the contraction axis of an MN-major operand,
//               e.g. weight-gradient operands whose contraction runs over an expert's rows).
// Values keep the source layout [R, C] (1 byte each).  Scales are written in the layout the
// block-scaled tensor-core MMA reads from tensor memory after a 32x128b.warpx4 copy: atoms of
// 128 MN-rows x 4 K-blocks (512 bytes), MN-row m / K-block b at byte
// 16*(m % 32) + 4*((m / 32) % 4) + (b % 4); atom (mn / 128, kb / 4) at
// ((mn / 128) * (K / 128) + kb / 4) * 512.  For row blocks MN = rows, K = C; for col blocks
// MN = columns, K = R.
// Optionally the row-blocked output permutes rows within each expert's [2I, H] gate/up matrix so
// that every 128-row block holds 64 gate rows followed by the 64 up rows of the same I columns.
// With a row map (row_slot, k) the quantiser is also the dispatch: output row r takes source row
// row_slot[r] / k, or zeros where row_slot[r] < 0 (padding), so the bf16 dispatched rows are
// never written.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kQRows = 32, kQCols = 128, kQThreads = 128;

// grid: (C / 128, R_max / 32).  rows_dev (optional): device count of valid 128-row tiles.
__global__ void __launch_bounds__(kQThreads) mx_quant_kernel(const __nv_bfloat16* __restrict__ src, long long R_max,
                                                             int C, const int* __restrict__ tiles_dev,
                                                             uint8_t* __restrict__ q_row, uint8_t* __restrict__ sf_row,
                                                             uint8_t* __restrict__ q_col, uint8_t* __restrict__ sf_col,
                                                             int gate_up_I, const int* __restrict__ row_slot, int k) {
    __shared__ __align__(16) __nv_bfloat16 tile[kQRows][kQCols + 8];
    __shared__ __align__(16) uint8_t qt[kQRows][kQCols + 16];
    const long long r0 = (long long)blockIdx.y * kQRows;
    const long long R = tiles_dev ? (long long)(*tiles_dev) * kBM : R_max;
    if (r0 >= R) return;
    const int c0 = blockIdx.x * kQCols;
    const int t = threadIdx.x;
    // load 32 x 128 bf16 with 16-byte accesses
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rr = it * 8 + (t >> 4), cc = (t & 15) * 8;
        long long sr = r0 + rr;
        if (row_slot) {
            const int slot = row_slot[sr];
            sr = slot >= 0 ? slot / k : -1;
        }
        *reinterpret_cast<uint4*>(&tile[rr][cc]) =
            sr >= 0 ? __ldg(reinterpret_cast<const uint4*>(src + sr * C + c0 + cc)) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (q_row) {
        // thread -> (row t/4, block t%4)
        const int rr = t >> 2, b = t & 3;
        float v[32];
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            v[j] = __bfloat162float(tile[rr][32 * b + j]);
            amax = fmaxf(amax, fabsf(v[j]));
        }
        uint8_t sf;
        float inv;
        mx_scale(amax, &sf, &inv);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            w[j] = (uint32_t)to_e4m3x2(v[4 * j] * inv, v[4 * j + 1] * inv) |
                   ((uint32_t)to_e4m3x2(v[4 * j + 2] * inv, v[4 * j + 3] * inv) << 16);
        long long r = r0 + rr;
        if (gate_up_I > 0) {  // 128-row blocks of [64 gate rows | 64 up rows] per expert
            const long long e = r / (2 * gate_up_I), j = r % (2 * gate_up_I);
            const long long jj = j < gate_up_I ? j : j - gate_up_I;
            r = e * 2 * gate_up_I + 128 * (jj / 64) + (j < gate_up_I ? 0 : 64) + jj % 64;
        }
        uint4* dst = reinterpret_cast<uint4*>(q_row + r * C + c0 + 32 * b);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        sf_row[sf_index(r, (c0 >> 5) + b, C / 128)] = sf;
    }
    if (q_col) {
        // thread -> column t, 32 rows
        float v[32];
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            v[j] = __bfloat162float(tile[j][t]);
            amax = fmaxf(amax, fabsf(v[j]));
        }
        uint8_t sf;
        float inv;
        mx_scale(amax, &sf, &inv);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const uint16_t p = to_e4m3x2(v[j] * inv, v[j + 1] * inv);
            qt[j][t] = (uint8_t)(p & 0xFF);
            qt[j + 1][t] = (uint8_t)(p >> 8);
        }
        sf_col[sf_index(c0 + t, r0 >> 5, R_max / 128)] = sf;
        __syncthreads();
        const int rr = t >> 2, q = t & 3;
        const uint4* s = reinterpret_cast<const uint4*>(&qt[rr][32 * q]);
        uint4* dst = reinterpret_cast<uint4*>(q_col + (r0 + rr) * C + c0 + 32 * q);
        dst[0] = s[0];
        dst[1] = s[1];
    }
}

cudaError_t launch_mx_quant(const Ctx& c, const void* src, long long R_max, int C, const int* tiles_dev, void* q_row,
                            void* sf_row, void* q_col, void* sf_col, int gate_up_I, const int* row_slot) {
    if (R_max <= 0) return cudaSuccess;
    dim3 grid(C / kQCols, (unsigned)(R_max / kQRows));
    trace_begin(c.st, kTraceQuant);
    mx_quant_kernel<<<grid, kQThreads, 0, c.st>>>(
        reinterpret_cast<const __nv_bfloat16*>(src), R_max, C, tiles_dev, reinterpret_cast<uint8_t*>(q_row),
        reinterpret_cast<uint8_t*>(sf_row), reinterpret_cast<uint8_t*>(q_col), reinterpret_cast<uint8_t*>(sf_col),
        gate_up_I, row_slot, (int)c.L->k);
    trace_end(c.st, kTraceQuant);
    return cudaGetLastError();
}

}  // namespace moe
