// quant.cu - MX quantiser: bf16 [R, C] -> E4M3 (or E2M1) values with one E8M0 scale per 32 elements.
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
// FP4 (row blocks only, weights of the FP8 x FP4 forward): E2M1 values with the block exponent
// floor(log2(amax)) - 2, rounded to nearest even and saturated to +-6, two per byte (the even
// column in the low nibble), rows of C / 2 bytes; the scales are laid out as above.
// Optionally the row-blocked output permutes rows within each expert's [2I, H] gate/up matrix so
// that every 128-row block holds 64 gate rows followed by the 64 up rows of the same I columns.
// With a row map (row_slot, k) the quantiser is also the dispatch: output row r takes source row
// row_slot[r] / k, or zeros where row_slot[r] < 0 (padding), so the bf16 dispatched rows are
// never written.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kQRows = 32, kQCols = 128, kQThreads = 128;

// Staged-tile layout: a row holds 16 chunks of 8 bf16 (16 bytes) at a 272-byte pitch, chunk j at
// position j ^ 2 * ((j >> 3) & 1).  The row-blocked pass has four lanes per row reading chunks
// 4b + q (b = the lane's 32-column block): without the swap chunks q and q + 8 share banks; with it
// eight lanes (two rows) read eight distinct bank groups.  Loads into the tile (16 consecutive
// chunks per row) and the column pass (32-bit words of one row) stay conflict-free.
__device__ __forceinline__ int tile_chunk(int j) { return j ^ (((j >> 3) & 1) << 1); }

// Maximum |x| of packed bf16 pairs: |bf16| bit patterns order like unsigned 16-bit integers, so a
// per-halfword unsigned max of the sign-cleared words gives both halves' maxima at once.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) { return __vmaxu2(acc, w & 0x7FFF7FFFu); }
__device__ __forceinline__ uint32_t absmax_to_f32_bits(uint32_t m2) {
    return max(m2 & 0xFFFFu, m2 >> 16) << 16;   // the larger half, as fp32 bits
}
// 8 bf16 (one uint4) scaled by inv into 8 E4M3 bytes (two 32-bit words)
__device__ __forceinline__ uint2 e4m3x8(uint4 w, float inv) {
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p[i] = to_e4m3x2(__uint_as_float(in[i] << 16) * inv, __uint_as_float(in[i] & 0xFFFF0000u) * inv);
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// 8 bf16 (one uint4) scaled by inv into 8 E2M1 nibbles (one 32-bit word, element 0 lowest)
__device__ __forceinline__ uint32_t e2m1x8(uint4 w, float inv) {
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t p = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p |= to_e2m1x2(__uint_as_float(in[i] << 16) * inv, __uint_as_float(in[i] & 0xFFFF0000u) * inv) << (8 * i);
    return p;
}

// grid: (C / 128, R_max / 128); one block quantises a 128 x 128 tile in four passes of 32 rows.
// Its row-blocked scales (128 rows x 4 column blocks) and column-blocked scales (128 columns x 4
// row blocks) are each exactly one 512-byte atom: staged in shared memory and written with 16-byte
// stores.  tiles_dev (optional): device count of valid 128-row tiles.
template <bool FP4>
__global__ void __launch_bounds__(kQThreads) mx_quant_kernel(const __nv_bfloat16* __restrict__ src, long long R_max,
                                                             int C, const int* __restrict__ tiles_dev,
                                                             uint8_t* __restrict__ q_row, uint8_t* __restrict__ sf_row,
                                                             uint8_t* __restrict__ q_col, uint8_t* __restrict__ sf_col,
                                                             int gate_up_I, const int* __restrict__ row_slot, int k) {
    grid_dep_wait();
    __shared__ __align__(16) __nv_bfloat16 tile[kQRows][kQCols + 8];
    __shared__ __align__(16) uint8_t qt[kQRows][kQCols + 16];
    __shared__ __align__(16) uint8_t s_sfr[512];
    __shared__ __align__(16) uint8_t s_sfc[512];
    __shared__ uint2 s_cmax[4][32];     // column-quad maxima of the four row quarters (column blocks)
    __shared__ long long s_src[128];   // source row of each tile row (-1: a zero padding row)
    const long long rt = (long long)blockIdx.y * 128;
    const long long R = tiles_dev ? (long long)(*tiles_dev) * kBM : R_max;
    if (rt >= R) return;
    const int c0 = blockIdx.x * kQCols;
    const int t = threadIdx.x;
    if (row_slot) {
        const int slot = __ldg(row_slot + rt + t);
        s_src[t] = slot >= 0 ? slot / k : -1;
    } else {
        s_src[t] = rt + t;
    }
    __syncthreads();
    // row blocks: thread -> (row 32 sub + t/4 of the tile, block t%4), the row's 32 values in w
    const int rr = t >> 2, b = t & 3;
    auto emit_row = [&](const uint4* w, int sub) {
        uint32_t m2 = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            m2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(m2, w[q].x), w[q].y), w[q].z), w[q].w);
        uint8_t sf;
        float inv;
        if constexpr (FP4) mx_scale_bits_e2m1(absmax_to_f32_bits(m2), &sf, &inv);
        else mx_scale_bits(absmax_to_f32_bits(m2), &sf, &inv);
        long long r = rt + 32 * sub + rr;
        if (gate_up_I > 0) {  // 128-row blocks of [64 gate rows | 64 up rows] per expert
            const long long e = r / (2 * gate_up_I), j = r % (2 * gate_up_I);
            const long long jj = j < gate_up_I ? j : j - gate_up_I;
            r = e * 2 * gate_up_I + 128 * (jj / 64) + (j < gate_up_I ? 0 : 64) + jj % 64;
        }
        s_sfr[16 * rr + 4 * sub + b] = sf;                      // tile row 32 sub + rr
        if constexpr (FP4) {
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = e2m1x8(w[q], inv);
            *reinterpret_cast<uint4*>(q_row + r * (C / 2) + (c0 + 32 * b) / 2) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            uint2 o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = e4m3x8(w[q], inv);
            uint4* dst = reinterpret_cast<uint4*>(q_row + r * C + c0 + 32 * b);
            dst[0] = make_uint4(o[0].x, o[0].y, o[1].x, o[1].y);
            dst[1] = make_uint4(o[2].x, o[2].y, o[3].x, o[3].y);
        }
    };
    // the gate/up copy's scales (threads 0..63, after the passes): the tile (128 rows, all gate or
    // all up, as 128 divides I) fills one half of two destination atoms, its rows [0, 64) the half
    // at row 64 * up of block jb / 64 and rows [64, 128) that of the next block; atom row p's four
    // bytes sit at 16 (p % 32) + 4 ((p / 32) % 4), so each half is 8 contiguous bytes per p % 32
    auto store_gate_up_scales = [&]() {
        if (t >= 64) return;
        const long long e = rt / (2 * gate_up_I), j = rt % (2 * gate_up_I);
        const bool up = j >= gate_up_I;
        const long long jb = up ? j - gate_up_I : j;                         // a multiple of 128
        const int half = t >> 5, m = t & 31;
        const long long blk = e * 2 * gate_up_I + 128 * (jb / 64 + half);   // destination block's first row
        uint8_t* dst = sf_row + sf_index(blk, c0 >> 5, C / 128) + 16 * m + (up ? 8 : 0);
        *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(s_sfr + 16 * m + 8 * half);
    };
    if (!q_col) {
        if (!q_row) return;
        // row blocks only: each thread reads its 64 bytes of the row straight from global memory
        // (no staging, no barriers), the next pass's loads in flight while this one is quantised
        auto load_row = [&](int sub, uint4* w) {
            const long long sr = s_src[32 * sub + rr];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                w[q] = sr >= 0 ? __ldg(reinterpret_cast<const uint4*>(src + sr * C + c0 + 32 * b) + q)
                               : make_uint4(0, 0, 0, 0);
        };
        uint4 cur[4], nx[4];
        load_row(0, cur);
#pragma unroll 1
        for (int sub = 0; sub < 4; ++sub) {
            if (sub < 3) load_row(sub + 1, nx);
            emit_row(cur, sub);
#pragma unroll
            for (int q = 0; q < 4; ++q) cur[q] = nx[q];
        }
        __syncthreads();
        if (gate_up_I <= 0 && t < 32)
            reinterpret_cast<uint4*>(sf_row + sf_index(rt, c0 >> 5, C / 128))[t] = reinterpret_cast<const uint4*>(s_sfr)[t];
        if (gate_up_I > 0) store_gate_up_scales();
        return;
    }
    // with a column-blocked copy: the 32 x 128 bf16 of pass `sub` staged in shared memory with
    // 16-byte accesses; thread t loads rows it*8 + t/16, columns 8 (t % 16) .. + 7 (through the
    // row map when dispatching)
    const int lr = t >> 4, lc = (t & 15) * 8;
    auto load_pass = [&](int sub, uint4* w) {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const long long sr = s_src[32 * sub + it * 8 + lr];
            w[it] = sr >= 0 ? __ldg(reinterpret_cast<const uint4*>(src + sr * C + c0 + lc)) : make_uint4(0, 0, 0, 0);
        }
    };
    uint4 nxt[4];
    load_pass(0, nxt);
    for (int sub = 0; sub < 4; ++sub) {
        const long long r0 = rt + 32 * sub;
#pragma unroll
        for (int it = 0; it < 4; ++it)
            *reinterpret_cast<uint4*>(&tile[it * 8 + lr][8 * tile_chunk(lc >> 3)]) = nxt[it];
        __syncthreads();
        if (sub < 3) load_pass(sub + 1, nxt);   // in flight while this pass is quantised
        if (q_row) {
            uint4 w[4];
            const uint4* row4 = reinterpret_cast<const uint4*>(&tile[rr][0]);
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = row4[tile_chunk(4 * b + q)];
            emit_row(w, sub);
        }
        if (!FP4 && q_col) {
            // thread -> columns 4 cq .. 4 cq + 3 (cq = lane) over rows 8 rq .. 8 rq + 7 (rq = warp): one
            // 8-byte shared load holds the four columns of a row, two packed unsigned maxima track
            // their |value| maxima, the four row quarters' maxima meet in shared memory (8 bytes a
            // thread), and each row's four codes leave as one 4-byte store
            const int cq = t & 31, rq = t >> 5;
            uint2 w[8];
            uint32_t ma = 0, mb = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                w[j] = reinterpret_cast<const uint2*>(&tile[8 * rq + j][0])[2 * tile_chunk(cq >> 1) + (cq & 1)];
                ma = absmax_bf16x2(ma, w[j].x);
                mb = absmax_bf16x2(mb, w[j].y);
            }
            s_cmax[rq][cq] = make_uint2(ma, mb);
            __syncthreads();
#pragma unroll
            for (int o = 1; o < 4; ++o) {
                const uint2 m = s_cmax[(rq + o) & 3][cq];
                ma = __vmaxu2(ma, m.x);
                mb = __vmaxu2(mb, m.y);
            }
            uint8_t sf[4];
            float inv[4];
            mx_scale_bits((ma & 0xFFFFu) << 16, &sf[0], &inv[0]);   // column 4 cq
            mx_scale_bits(ma & 0xFFFF0000u, &sf[1], &inv[1]);       // column 4 cq + 1
            mx_scale_bits((mb & 0xFFFFu) << 16, &sf[2], &inv[2]);   // column 4 cq + 2
            mx_scale_bits(mb & 0xFFFF0000u, &sf[3], &inv[3]);       // column 4 cq + 3
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint32_t*>(&qt[8 * rq + j][4 * cq]) =
                    (uint32_t)to_e4m3x2(__uint_as_float(w[j].x << 16) * inv[0],
                                        __uint_as_float(w[j].x & 0xFFFF0000u) * inv[1]) |
                    ((uint32_t)to_e4m3x2(__uint_as_float(w[j].y << 16) * inv[2],
                                         __uint_as_float(w[j].y & 0xFFFF0000u) * inv[3])
                     << 16);
            if (rq == 0) {   // columns 4 cq .. 4 cq + 3, row block sub
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int col = 4 * cq + i;
                    s_sfc[16 * (col & 31) + 4 * (col >> 5) + sub] = sf[i];
                }
            }
            __syncthreads();
            // the 32 x 128 codes out, thread -> (row t/4, 32 columns at 32 (t%4))
            const uint4* s4 = reinterpret_cast<const uint4*>(&qt[rr][32 * b]);
            uint4* dst = reinterpret_cast<uint4*>(q_col + (r0 + rr) * C + c0 + 32 * b);
            dst[0] = s4[0];
            dst[1] = s4[1];
        }
        __syncthreads();
    }
    // the tile's two scale atoms, 16 bytes per thread
    if (q_row && gate_up_I <= 0 && t < 32)
        reinterpret_cast<uint4*>(sf_row + sf_index(rt, c0 >> 5, C / 128))[t] = reinterpret_cast<const uint4*>(s_sfr)[t];
    if (q_row && gate_up_I > 0) store_gate_up_scales();
    if (!FP4 && q_col && t >= 32 && t < 64)
        reinterpret_cast<uint4*>(sf_col + sf_index(c0, rt >> 5, R_max / 128))[t - 32] =
            reinterpret_cast<const uint4*>(s_sfc)[t - 32];
}

// The row-blocked E4M3 copy of the dispatched rows, token-major.  A row block (32 consecutive
// columns of one row) does not depend on where the row is dispatched, so one warp quantises each
// token row once and stores its codes and scale bytes to every one of the token's k dispatched
// rows (pos); units past the tokens write the padding rows' zero codes and zero scales, 32 rows
// a unit.  This reads x from HBM once, in order, where the dispatched-row walk of mx_quant_kernel
// reads each token row k times from L2 while its stores stream past.
// Lane l holds the 16-byte vectors l + 32 q (q < 8) of each 2048-column chunk, so block
// l / 4 + 8 q of the chunk lives in lanes 4 (l / 4) .. + 3 and its maximum takes two shuffles.
// The scale bytes of four consecutive blocks form one 4-byte word of the atom layout above;
// lane g < 16 ends up holding the chunk's word g and stores it for each destination row.
constexpr int kTokThreads = 256;

__global__ void __launch_bounds__(kTokThreads) mx_rows_token_kernel(const uint4* __restrict__ src, int T, int C, int k,
                                                                    const int* __restrict__ pos,
                                                                    const int* __restrict__ row_slot,
                                                                    const int* __restrict__ tiles_dev,
                                                                    uint8_t* __restrict__ q_row,
                                                                    uint8_t* __restrict__ sf_row) {
    grid_dep_wait();
    const int nrows = (*tiles_dev) * kBM;
    const int lane = threadIdx.x & 31;
    const int wpb = kTokThreads / 32;
    const int stride = gridDim.x * wpb;
    const int rv = C / 8;              // 16-byte bf16 vectors in a row
    const long long k_atoms = C / 128;
    const int units = T + (nrows + 31) / 32;
    for (int u = blockIdx.x * wpb + (threadIdx.x >> 5); u < units; u += stride) {
        if (u < T) {
            const int p0 = lane < k ? pos[(size_t)u * k + lane] : -1;
            for (int v0 = 0; v0 < rv; v0 += 256) {
                const int nq = min(256, rv - v0) / 32;   // C % 256 == 0: whole 32-vector steps
                const uint4* s = src + (size_t)u * rv + v0;
                uint4 w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) w[q] = q < nq ? __ldg(s + lane + 32 * q) : make_uint4(0, 0, 0, 0);
                uint2 code[8];
                uint32_t word = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    code[q] = make_uint2(0, 0);
                    if (q >= nq) continue;   // warp-uniform
                    uint32_t m2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(0u, w[q].x), w[q].y), w[q].z), w[q].w);
                    m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 1));
                    m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 2));
                    uint8_t sf;
                    float inv;
                    mx_scale_bits(absmax_to_f32_bits(m2), &sf, &inv);
                    code[q] = e4m3x8(w[q], inv);
                    // the word of blocks 8 q + 4 h .. + 3 (h = lane / 16) in every lane of half h
                    uint32_t pk = (uint32_t)sf << (8 * ((lane >> 2) & 3));
                    pk |= __shfl_xor_sync(0xffffffffu, pk, 4);
                    pk |= __shfl_xor_sync(0xffffffffu, pk, 8);
                    const uint32_t from = __shfl_sync(0xffffffffu, pk, (lane & 1) << 4);
                    if (((lane & 15) >> 1) == q) word = from;   // lane g < 16: word g = 2 q + (g & 1)
                }
                for (int j0 = 0; j0 < k; j0 += 32) {
                    const int pj = j0 == 0 ? p0 : (j0 + lane < k ? pos[(size_t)u * k + j0 + lane] : -1);
                    const int nj = min(32, k - j0);
                    for (int j = 0; j < nj; ++j) {
                        const int r = __shfl_sync(0xffffffffu, pj, j);
                        if (r < 0) continue;   // a slot with an out-of-range expert id is not dispatched
                        uint8_t* d = q_row + (size_t)r * C + (size_t)v0 * 8;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            if (q < nq) *reinterpret_cast<uint2*>(d + 8 * (lane + 32 * q)) = code[q];
                        if (lane < 2 * nq)
                            *reinterpret_cast<uint32_t*>(sf_row + sf_index(r, v0 / 4 + 4 * lane, k_atoms)) = word;
                    }
                }
            }
        } else {
            const int row0 = (u - T) * 32;
            const bool pad = row0 + lane < nrows && row_slot[row0 + lane] < 0;
            unsigned m = __ballot_sync(0xffffffffu, pad);
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1;
                const long long r = row0 + b;
                uint4* d = reinterpret_cast<uint4*>(q_row + r * C);
                for (int v = lane; v < C / 16; v += 32) d[v] = make_uint4(0, 0, 0, 0);
                for (int g = lane; g < C / 128; g += 32)
                    *reinterpret_cast<uint32_t*>(sf_row + sf_index(r, 4 * g, k_atoms)) = 0u;
            }
        }
    }
}

cudaError_t launch_mx_rows_token(const Ctx& c, const void* src, const int* pos, const int* row_slot,
                                 const int* tiles_dev, void* q_row, void* sf_row) {
    const Layout& L = *c.L;
    trace_begin(c.st, kTraceQuantRows);
    const cudaError_t err = launch_pdl(mx_rows_token_kernel, c.num_sms * 8, kTokThreads, 0, c.st,
                                       reinterpret_cast<const uint4*>(src), (int)L.T, (int)L.H, (int)L.k, pos,
                                       row_slot, tiles_dev, reinterpret_cast<uint8_t*>(q_row),
                                       reinterpret_cast<uint8_t*>(sf_row));
    trace_end(c.st, kTraceQuantRows);
    return err;
}

cudaError_t launch_mx_quant(const Ctx& c, const void* src, long long R_max, int C, const int* tiles_dev, void* q_row,
                            void* sf_row, void* q_col, void* sf_col, int gate_up_I, const int* row_slot, bool fp4) {
    if (R_max <= 0) return cudaSuccess;
    if (fp4 && (q_col || !q_row)) return cudaErrorInvalidValue;   // MXFP4 copies are row-blocked only
    dim3 grid(C / kQCols, (unsigned)(R_max / 128));
    auto kern = fp4 ? mx_quant_kernel<true> : mx_quant_kernel<false>;
    trace_begin(c.st, kTraceQuant);
    const cudaError_t err = launch_pdl(
        kern, grid, kQThreads, 0, c.st, reinterpret_cast<const __nv_bfloat16*>(src), R_max, C, tiles_dev,
        reinterpret_cast<uint8_t*>(q_row), reinterpret_cast<uint8_t*>(sf_row), reinterpret_cast<uint8_t*>(q_col),
        reinterpret_cast<uint8_t*>(sf_col), gate_up_I, row_slot, (int)c.L->k);
    trace_end(c.st, kTraceQuant);
    return err;
}

}  // namespace moe
