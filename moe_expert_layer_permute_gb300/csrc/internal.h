// internal.h - scratch layout and kernel launchers of the MoE layer (host side, C++).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_layer.h"

namespace moe {

// Launches `kern` with programmatic stream serialization (see grid_dep_wait in common.cuh): the
// launch may begin while the previous kernel on `st` finishes; the kernel itself waits for it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kBM = 128;          // rows of a GEMM tile; each expert's rows are padded to a multiple
constexpr int kBK = 64;           // bf16 elements of K per pipeline stage (one 128-byte row)
constexpr int kRouteChunk = 2048; // slots per block of the routing kernels
constexpr int kMaxExperts = 1024;

// MX operand copies (E4M3 values + E8M0 scale atoms, see quant.cu): "_r" blocked along the
// row (K-major use), "_c" blocked along the column (MN-major use).  In the FP8 x FP4 forward the
// weights' _r copies hold packed E2M1 values instead.
struct MxLayout {
    size_t x_r, x_r_sf, x_c, x_c_sf;      // dispatched x rows [rows, H]
    size_t h_r, h_r_sf;                   // h [rows, I]
    size_t dy_r, dy_r_sf, dy_c, dy_c_sf;  // dispatched dy rows [rows, H]
    size_t dg_r, dg_r_sf, dg_c, dg_c_sf;  // [dg|du] [rows, 2I]
    size_t hw_c, hw_c_sf;                 // w h [rows, I]
    size_t w13_r, w13_r_sf, w13_c, w13_c_sf;  // W13 [E*2I, H] (the _r copy in [64 gate|64 up] blocks)
    size_t w2_r, w2_r_sf, w2_c, w2_c_sf;      // W2 [E*H, I]
};

// Byte offsets of every region of the scratch buffer for one desc.  The routed rows of expert e
// occupy padded rows [pad_off[e], pad_off[e+1]) with pad_off[e] a multiple of 128, so a GEMM
// tile never straddles two experts; padding rows hold zeros.  `rows` bounds the padded count.
struct Layout {
    int64_t T, H, I, E, k, S, rows, nb_route, n_dtw;
    size_t ctrl, hist, cnt, off, pad_off, mtile, order, base, perm, inv, pos, row_slot;
    size_t xperm, hid, gu, ypart, dyperm, dg, hw, dtw;   // ypart also holds the fused combine's fp32 [T, H]
    bool mx_fwd, mx_bwd, mx_on;   // forward / backward GEMMs in MXFP8; either (MXFP8 regions exist)
    bool fp4w;                    // FP8 x FP4 forward: w13_r / w2_r hold MXFP4 (packed E2M1)
    MxLayout mx;
    size_t mx_bytes[24];          // byte size of each MxLayout region, in field order (0: absent)
    size_t total;
};

bool make_layout(const moe_desc* d, Layout* L);

// ---- launchers (all asynchronous on `st`) ---------------------------------------------------
struct Ctx {
    cudaStream_t st;
    char* base;        // scratch base
    const Layout* L;
    int* status;       // device status word
    int num_sms;
    const float* topk_w;  // routing weights [T*k] (caller's tensor)
    long long wait_limit = 0;   // pipeline wait limit in cycles (0: the default)
    uint32_t test_flags = 0;    // MOE_TEST_* (moe_set_wait_limit)
};

// routing: counts, offsets, padded offsets, m-tile prefix, expert order, perm / inv / pos / row_slot
cudaError_t launch_routing(const Ctx& c, const int32_t* topk_idx);
// The routing kernels on explicit buffers: hist and base hold 2 * ceil(S / kRouteChunk) * E ints of
// working memory; pad_off, mtile, order, pos, row_slot (the padded row layout) and status may all
// be null together, in which case only counts, offsets, perm and inv are produced.
struct RoutingBufs {
    int *hist, *base, *cnt, *off, *pad_off, *mtile, *order, *perm, *inv, *pos, *row_slot;
};
cudaError_t launch_routing_kernels(cudaStream_t st, const int32_t* topk_idx, int S, int E, const RoutingBufs& r,
                                   int* status);
// dst[r] = src[row_slot[r] / k] for every padded row r (zeros on padding rows); up to two pairs
cudaError_t launch_gather(const Ctx& c, const void* src0, void* dst0, const void* src1, void* dst1);
// out[t] = sum_j part[pos[t*k+j]] (fixed j order); optionally dtopk_w[s] = sum_n dtw[pos[s], n]
cudaError_t launch_combine(const Ctx& c, const void* part, void* out, float* dtopk_w);
// fused combine: zero the fp32 [T, H] accumulator (before FwdDownReduce), and round it to bf16 y
cudaError_t launch_reduce_zero(const Ctx& c);
cudaError_t launch_reduce_finish(const Ctx& c, void* y);

// router (the step before the layer): top-k of fp32 logits with the softmax over the selected,
// and its backward; T = 0 launches nothing
cudaError_t launch_router_fwd(cudaStream_t st, const float* logits, int T, int E, int k, int* topk_idx, float* topk_w);
cudaError_t launch_router_bwd(cudaStream_t st, const int* topk_idx, const float* topk_w, const float* dtopk_w, int T,
                              int E, int k, float* dlogits);

// grouped GEMMs (persistent, TMA + tcgen05)
enum class GemmKind : int {
    FwdGateUp = 0,     // [g|u] = X_perm W13[e]^T, epilogue w h = w silu(g) u (MXFP8: h, unweighted)
                       // (optionally saves [g|u])
    FwdGateUpSaveOnly, // same GEMM, epilogue stores [g|u] only (MXFP8 backward recompute)
    FwdDown,           // Ypart = (w h) W2[e]^T (MXFP8: o = h W2[e]^T, epilogue Ypart = w o)
    BwdDown,           // dA = dY_perm W2[e], epilogue SwiGLU backward -> [dg|du], <dA, h> (MXFP8: and w h)
    BwdGateUp,         // dXpart = [dg|du] W13[e]
    WgradDown,         // dW2[e] = dY_perm^T (w h) over the expert's rows
    WgradGateUp,       // dW13[e] = [dg|du]^T X_perm over the expert's rows
    FwdDownReduce,     // (w h) W2[e]^T, added by the epilogue into the fp32 [T, H] accumulator (fused combine)
};
constexpr int kGemmKinds = 8;
cudaError_t launch_gemm(const Ctx& c, GemmKind kind, const void* W, void* out, bool out_f32, bool save_gu);
// N tile of the backward down-projection product (and so the number of <dA, h> partials per row)
int bwd_down_bn(int64_t I);

// MX quantiser over a bf16 [R_max, C] array (R_max % 32 == 0, C % 128 == 0); with tiles_dev only
// the first tiles_dev[0] * 128 rows.  Any of the outputs may be null.  gate_up_I > 0 stores the
// row-blocked copy of a [E*2I, H] gate/up weight in [64 gate | 64 up] row blocks.
// With row_slot (padded rows only) source row r is row_slot[r] / k, zero where row_slot[r] < 0.
// fp4: the row-blocked copy holds MXFP4 (packed E2M1, C / 2 bytes a row) and q_col must be null.
// the row-blocked E4M3 copy of the dispatched rows of src [T, H], token-major (quant.cu)
cudaError_t launch_mx_rows_token(const Ctx& c, const void* src, const int* pos, const int* row_slot,
                                 const int* tiles_dev, void* q_row, void* sf_row);
cudaError_t launch_mx_quant(const Ctx& c, const void* src, long long R_max, int C, const int* tiles_dev, void* q_row,
                            void* sf_row, void* q_col, void* sf_col, int gate_up_I, const int* row_slot = nullptr,
                            bool fp4 = false);

// tracing ids: one per kernel kind; the GEMM kinds follow kTraceGemm (BF16) and kTraceGemmMx
enum TraceId : int {
    kTraceRouteHist = 0, kTraceRouteScan, kTraceRoutePlace, kTraceGather, kTraceCombine, kTraceQuant,
    kTraceReduceFinish, kTraceQuantRows, kTraceGemm, kTraceGemmMx = kTraceGemm + kGemmKinds, kTraceKinds = kTraceGemmMx + kGemmKinds
};

// tracing hooks used by the launch sequence
void trace_begin(cudaStream_t st, int kind_id);
void trace_end(cudaStream_t st, int kind_id);

}  // namespace moe
