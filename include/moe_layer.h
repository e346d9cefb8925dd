/*
 * moe_layer.h - C ABI of the GB300 fused MoE expert layer (forward and backward).
 *
 * The layer (MarkTechPost, "Prime Intellect Releases Prime Mega MoE", section "How does the fused
 * kernel work?"): every token is dispatched to k of E experts, each expert applies two linear
 * layers with SwiGLU between them, and the expert outputs are combined back per token by routing
 * weight; the fused call keeps its intermediates in GPU-only scratch buffers instead of tensors.
 * Grouping tokens by expert (counts, group offsets, token reorder) and the weighted aggregation
 * follow kongchang.com, "Prime Intellect推出Prime Mega MoE", section "为什么 MoE 训练特别需要融合内核".
 * The experts are gated and bias-free, H % 256 == 0 and I % 128 == 0, in BF16 or MXFP8 on
 * Blackwell (ic.work analysis, section "算子下沉时代的硬件死锁暗礁").  One call per direction:
 * moe_fwd and moe_bwd (the backward was added for training: MarkTechPost, same section).
 *
 * With every expert on one GPU, the expert-parallel dispatch is a gather of token rows into
 * expert order and the combine is a weighted, fixed-order sum back to token order.
 *
 * Shapes (row-major, element strides; the innermost stride must be 1 and rows contiguous):
 *   x, dy, y, dx : [T, H]  bf16          topk_idx : [T, k] int32 (expert ids, distinct per token)
 *   topk_w       : [T, k]  fp32          dtopk_w  : [T, k] fp32
 *   W13, dW13    : [E, 2I, H]            rows [0, I) = gate projection, rows [I, 2I) = up projection
 *   W2,  dW2     : [E, H, I]             W13 / W2 are bf16; dW13 / dW2 are bf16 or fp32
 *   y[t] = sum_j topk_w[t,j] * W2[e] (silu(W13[e,:I] x[t]) * (W13[e,I:] x[t])),  e = topk_idx[t,j]
 *   moe_bwd returns the gradients of <dy, y> with respect to x, W13, W2 and topk_w.
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller owns every buffer, the scratch buffer included.  The library never
 *     allocates or frees device memory and keeps no pointer after a call returns.
 *   - Asynchrony: moe_fwd / moe_bwd only enqueue work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronise.  Outputs are overwritten, not accumulated.
 *   - Errors: arguments are validated on the host before anything is launched; a negative
 *     MOE_ERR_* code is returned and nothing is enqueued.  A launch failure returns MOE_ERR_CUDA.
 *     Device-side problems (an expert id outside [0, E), a pipeline wait that timed out) never
 *     trap: the kernels record a code in the scratch status word, which moe_read_device_status
 *     returns.  Out-of-range expert ids are always checked on the device and such slots are
 *     dropped (they contribute nothing; their dtopk_w is 0).
 *   - Alignment: every device pointer must be 16-byte aligned (TMA); the scratch pointer 256-byte.
 *   - T == 0 is a valid no-op (dW13 / dW2 are zeroed by moe_bwd).
 *   - Calls that share one scratch buffer must be ordered on one stream.
 *   - moe_bwd runs its final combine (dx) on a side stream of the device, forked from and joined
 *     back to `stream` by events inside the call, so that it overlaps the weight-gradient products;
 *     work enqueued on `stream` after the call is ordered after all of it.  The side stream and its
 *     events are created on the first moe_bwd on a device and shared by all calls on that device:
 *     host threads that call moe_bwd concurrently on one device must serialise those calls.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- types ------------------------------------------------------------------------------- */
/* MOE_FP8_BWD: the forward in BF16 and the backward in MXFP8 (the pages' fp8_bwd precision, a BF16
 * forward with an FP8 backward: MarkTechPost, "Prime Intellect Releases Prime Mega MoE", section
 * "How does the fused kernel work?"); y is bit-identical to MOE_BF16's. */
/* MOE_FP8_FP4: a forward-only layer whose GEMMs take MXFP8 activations (E4M3) times MXFP4 weights
 * (E2M1 values, grid 0, 0.5, 1, 1.5, 2, 3, 4, 6, one E8M0 scale per 32 values with exponent
 * floor(log2(amax)) - 2, ties to even, saturating at 6), each blocked along its GEMM's contraction
 * (the FP8xFP4 data type the comparison table lists for DeepGEMM's Mega MoE: wire.sakhanda.co,
 * "Prime Intellect пусна Prime Mega MoE", section "Как се сравнява с други слети MoE опции?", data
 * types row; the English copy of that table drops the row).  Forward only, like DeepGEMM's kernel:
 * moe_bwd returns MOE_ERR_UNSUPPORTED for it. */
typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1, MOE_FP8_BWD = 2, MOE_FP8_FP4 = 3 } moe_precision;
typedef enum { MOE_DT_BF16 = 0, MOE_DT_F32 = 1, MOE_DT_I32 = 2 } moe_dtype;

/* A view of a caller-owned buffer: `data` is a device pointer for the layer calls. */
typedef struct {
    void*   data;
    int32_t dtype;      /* moe_dtype */
    int32_t ndim;       /* 1..3 */
    int64_t shape[3];
    int64_t stride[3];  /* in elements */
} moe_tensor;

/* Problem description.  precision is a moe_precision; flags a set of MOE_FLAG_*. */
typedef struct {
    int64_t  T, H, I, E, k;
    int32_t  precision;
    uint32_t flags;
} moe_desc;

/* moe_fwd also stores the gate/up pre-activations [g|u] (bf16, 2I per routed row) in scratch, so
 * that a following moe_bwd with MOE_FLAG_REUSE_FWD skips recomputing the first GEMM (the second
 * forward of an activation-checkpointed layer is that recompute). */
#define MOE_FLAG_SAVE_GU     0x1u
/* moe_bwd reuses the routing, the dispatched rows and [g|u] left in scratch by the latest moe_fwd
 * that had MOE_FLAG_SAVE_GU and the same x, topk_idx, topk_w, W13, W2 pointers, desc and epoch;
 * returns MOE_ERR_STATE (before any launch) if the scratch handle does not record such a forward. */
#define MOE_FLAG_REUSE_FWD   0x2u
/* Block-scaled precisions only (MOE_MXFP8, MOE_FP8_BWD, MOE_FP8_FP4): W13 and W2 hold the same
 * values as when an earlier call on this scratch (same pointers, same epoch) quantised them, so
 * their E4M3 / E2M1 copies in scratch are reused instead of being made again (a training step
 * quantises its weights once: forward, recompute and backward share them; a forward-only layer
 * keeps them).  Returns MOE_ERR_STATE (before any launch) if the scratch handle records no
 * quantisation of these pointers at the current epoch. */
#define MOE_FLAG_REUSE_WEIGHTS 0x4u
/* moe_fwd only, BF16 forward (MOE_BF16, MOE_FP8_BWD; MOE_ERR_UNSUPPORTED for the others): the
 * combine is fused into the down projection, one call with no intermediate Ypart rows (the pages'
 * single fused layer: MarkTechPost, "Prime Intellect Releases Prime Mega MoE", section "How does
 * the fused kernel work?").  The down GEMM's epilogue adds w * o of every routed row into an fp32
 * [T, H] accumulator in scratch by vector atomic reductions, and a final pass rounds it to y.  y is
 * then not bitwise reproducible: the fp32 additions follow the tiles' timing, so runs may differ in
 * the last bit of an element; without the flag the combine sums in a fixed order. */
#define MOE_FLAG_FUSED_COMBINE 0x8u

/* Host-side handle of a caller-owned device scratch buffer of at least moe_scratch_bytes(desc)
 * bytes.  `epoch` is the caller's: a counter it advances whenever x, W13 or W2 may have changed in
 * place at the same addresses (an optimizer step updates the weights in place), so that the reuse
 * flags refuse results made before the change.  `state` is written by the library (which forward's
 * results and which weight copies the buffer holds, and the wait settings of
 * moe_set_wait_limit); zero `epoch` and `state` when the handle is created. */
typedef struct {
    void*    data;
    uint64_t bytes;
    moe_desc desc;
    uint64_t epoch;
    uint64_t state[4];
} moe_scratch;

/* ---- status codes ------------------------------------------------------------------------ */
#define MOE_OK                0
#define MOE_ERR_NULL         -1   /* a required pointer is NULL */
#define MOE_ERR_SHAPE        -2   /* shape rules: H % 256, I % 128, 1 <= k <= E, tensor shapes */
#define MOE_ERR_DTYPE        -3   /* a tensor has the wrong element type */
#define MOE_ERR_LAYOUT       -4   /* rows not contiguous / innermost stride != 1 */
#define MOE_ERR_ALIGN        -5   /* a pointer or row pitch is not 16-byte aligned */
#define MOE_ERR_SCRATCH      -6   /* scratch missing, too small, misaligned or made for another desc */
#define MOE_ERR_STATE        -7   /* MOE_FLAG_REUSE_FWD without a matching saved forward */
#define MOE_ERR_UNSUPPORTED  -8   /* precision or size outside what this build supports */
#define MOE_ERR_CUDA         -9   /* a CUDA runtime call or kernel launch failed */
#define MOE_ERR_DEVICE       -10  /* the device status word holds a MOE_DEV_* code */

/* device status word codes (moe_read_device_status) */
#define MOE_DEV_OK            0
#define MOE_DEV_BAD_EXPERT    1   /* an expert id outside [0, E) was dropped */
#define MOE_DEV_TIMEOUT       2   /* a pipeline wait gave up; the kernel exited early */

/* ---- sizes -------------------------------------------------------------------------------- */
/* Bytes of scratch moe_fwd / moe_bwd need for `desc` (0 if desc breaks the shape rules).
 * It grows linearly in T*k (routed rows, each padded per expert to a multiple of 128). */
size_t moe_scratch_bytes(const moe_desc* desc);

/* ---- the layer ---------------------------------------------------------------------------- */
/* Forward: y = the layer applied to x.  Scratch receives the routing bookkeeping, the dispatched
 * rows, the hidden activations and (with MOE_FLAG_SAVE_GU) [g|u]. */
int moe_fwd(const moe_tensor* x, const moe_tensor* topk_idx, const moe_tensor* topk_w,
            const moe_tensor* W13, const moe_tensor* W2, moe_tensor* y,
            moe_scratch* scratch, void* stream);

/* Backward of <dy, y>: dx, dW13, dW2 and dtopk_w (all overwritten).  Without
 * MOE_FLAG_REUSE_FWD it recomputes the routing and the first GEMM itself.  MOE_FP8_FP4 scratch:
 * MOE_ERR_UNSUPPORTED (forward only). */
int moe_bwd(const moe_tensor* dy, const moe_tensor* x, const moe_tensor* topk_idx,
            const moe_tensor* topk_w, const moe_tensor* W13, const moe_tensor* W2,
            moe_tensor* dx, moe_tensor* dW13, moe_tensor* dW2, moe_tensor* dtopk_w,
            moe_scratch* scratch, void* stream);

/* Synchronises `stream`, returns the device status word in *status (a MOE_DEV_* code) and
 * clears it.  Returns MOE_OK, or MOE_ERR_CUDA if the synchronisation itself failed. */
int moe_read_device_status(moe_scratch* scratch, void* stream, int* status);

/* Every wait of the grouped GEMMs' pipelines is bounded: a wait that lasts longer than the limit
 * gives up, the kernel records MOE_DEV_TIMEOUT in the status word, drains what it has in flight,
 * frees its tensor memory and returns (it never traps or hangs: a lesson the pages draw from a
 * persistent kernel that deadlocked, ic.work analysis, section "算子下沉时代的硬件死锁暗礁").
 * moe_set_wait_limit sets, for later calls on this scratch handle, the limit in SM clock cycles
 * (0 restores the default, 4e9 cycles, about 2 s at the maximum SM clock) and test flags:
 * MOE_TEST_WITHHOLD_LOADS makes the grouped GEMMs issue no operand loads, so that their waits run
 * out with no copy in flight, which tests this path (outputs are then unspecified).  Host-side
 * only (stored in scratch->state); returns MOE_ERR_NULL for a NULL handle, MOE_ERR_SHAPE for a
 * negative limit. */
#define MOE_TEST_WITHHOLD_LOADS 0x1u
int moe_set_wait_limit(moe_scratch* scratch, int64_t wait_cycles, uint32_t test_flags);

/* Static message for a MOE_ERR_* code. */
const char* moe_strerror(int code);

/* ---- the router that precedes the layer ----------------------------------------------------- */
/* The pages' single-layer benchmark leaves the router out (ic.work analysis, section
 * "跑分背后的理想假设与闭源软肋"); its outputs are the layer's topk_idx and topk_w, the routing
 * weights that aggregate each token's expert outputs (kongchang.com, "Prime Intellect推出Prime Mega
 * MoE", section "为什么 MoE 训练特别需要融合内核").  Where the pages are silent: the k largest
 * logits of each token are selected (ties to the lower expert index), listed in descending
 * order, and weighted by the softmax over the selected logits.
 *
 * moe_router_fwd: logits fp32 [T, E] -> topk_idx int32 [T, k], topk_w fp32 [T, k] (overwritten).
 * moe_router_bwd: dlogits fp32 [T, E] (overwritten) of sum_j dtopk_w[t,j] * topk_w[t,j]:
 *   dlogits[t, topk_idx[t,j]] = w_j (dw_j - sum_i w_i dw_i), zero for experts a token did not
 *   select; topk_idx and topk_w as moe_router_fwd wrote them (distinct experts per token).
 * All tensors are row-contiguous device buffers, 16-byte aligned, owned by the caller; T and E are
 * the logits' / dlogits' shape and k the second dimension of topk_idx.  1 <= k <= 32,
 * k <= E <= 1024, T >= 0 (T = 0 launches nothing).  Returns MOE_ERR_* before any launch on bad
 * arguments, MOE_ERR_UNSUPPORTED for k or E outside those bounds, MOE_ERR_CUDA on a launch error.
 * Asynchronous on `stream`.  Logits must be finite: NaN logits give unspecified experts (always
 * in [0, E)) and NaN weights; expert ids outside [0, E) given to moe_router_bwd are skipped. */
int moe_router_fwd(const moe_tensor* logits, moe_tensor* topk_idx, moe_tensor* topk_w, void* stream);
int moe_router_bwd(const moe_tensor* topk_idx, const moe_tensor* topk_w, const moe_tensor* dtopk_w,
                   moe_tensor* dlogits, void* stream);

/* ---- routing without caller-provided scratch ---------------------------------------------- */
/* The pages have no counterpart to this entry point; it exists for callers that cannot allocate
 * device memory or hand over a scratch buffer (code running inside an allocator's hooks, runtimes
 * that reserve all device memory up front and forbid later allocations, loops where an allocation
 * would synchronise the device).  It computes the same routing bookkeeping as moe_fwd:
 *   counts  int32[E]     tokens routed to each expert
 *   offsets int32[E+1]   exclusive prefix of counts
 *   perm    int32[T*k]   slot at each sorted position, stable in slot order s = t*k + j; slots
 *                        whose id is outside [0, E) are dropped, and the positions they leave free,
 *                        [offsets[E], T*k), hold -1
 *   inv     int32[T*k]   sorted position of each slot (-1 for a slot whose id is outside [0, E))
 * from topk_idx int32[T, k] (all device pointers, 4-byte aligned, caller-owned), asynchronously on
 * `stream`.  It allocates nothing: its working memory is a file-scope static device array of
 * 65536 int32 (256 KiB) that every GPU loading the library holds until exit.  Sizes with
 * 2 * ceil(T*k / 2048) * E > 65536 are rejected with MOE_ERR_UNSUPPORTED before any launch.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) and caches
 * it; make that first call before any stream capture.  Calls share the array: calls whose kernels
 * may overlap on the GPU (unordered streams) race on it and must not be issued. */
int moe_route_static(const int32_t* topk_idx, int64_t T, int64_t k, int64_t E, int32_t* counts,
                     int32_t* offsets, int32_t* perm, int32_t* inv, void* stream);

/* ---- introspection (tests, tracing) ------------------------------------------------------- */
/* Named regions of the scratch buffer, valid after a call on that scratch.  Layouts:
 *   MOE_VIEW_COUNTS   int32[E]        tokens routed to each expert
 *   MOE_VIEW_OFFSETS  int32[E+1]      exclusive prefix of the counts (group offsets)
 *   MOE_VIEW_PERM     int32[T*k]      slot (t*k+j) at each sorted position, stable in slot order
 *                                     (-1 in the positions [OFFSETS[E], T*k) that dropped slots free)
 *   MOE_VIEW_INV      int32[T*k]      sorted position of each slot (-1 for a dropped slot)
 *   MOE_VIEW_PAD_OFFSETS int32[E+1]   start row of each expert in the padded row layout
 *   MOE_VIEW_XPERM    bf16 [rows, H]  dispatched x rows (padded layout: expert e's rows start at
 *                                     PAD_OFFSETS[e], padding rows are zero)
 *   MOE_VIEW_HID      bf16 [rows, I]  w * silu(g) * u of every routed row, w the row's routing
 *                                     weight (BF16 forward: the down product then applies no
 *                                     weight, and the backward reuses these rows)
 *   MOE_VIEW_GU       bf16 [rows, 2I] [g | u] pre-activations
 *   MOE_VIEW_YPART    bf16 [rows, H]  w * expert output per routed row (forward, before combine)
 *   MOE_VIEW_DG       bf16 [rows, 2I] [dg | du] (backward)
 *   MOE_VIEW_HW       bf16 [rows, I]  w * h: the same region as MOE_VIEW_HID
 *   MOE_VIEW_DYPERM   bf16 [rows, H]  dispatched dy rows (backward)
 * `rows` is T*k + 128*E, the largest padded row count.  Returns MOE_ERR_SHAPE for an unknown id. */
enum {
    MOE_VIEW_COUNTS = 0, MOE_VIEW_OFFSETS, MOE_VIEW_PERM, MOE_VIEW_INV, MOE_VIEW_PAD_OFFSETS,
    MOE_VIEW_XPERM, MOE_VIEW_HID, MOE_VIEW_GU, MOE_VIEW_YPART, MOE_VIEW_DG, MOE_VIEW_HW,
    MOE_VIEW_DYPERM, MOE_VIEW_COUNT_
};
/* MX operand copies (MOE_MXFP8; MOE_FP8_BWD has only the backward's: X_C, DY_R, DY_C, DG_R, DG_C,
 * HW_C, W13_C, W2_C; MOE_FP8_FP4 only the forward's: X_R, H_R, W13_R, W2_R; absent ones are 0
 * bytes): for each operand a uint8 E4M3 value array in
 * the source's layout, then its E8M0 scales (one byte per 32 values) in tensor-core atoms of 128
 * MN-rows x 4 K-blocks (512 bytes: MN-row m, K-block b at byte 16*(m%32) + 4*((m/32)%4) + b%4;
 * atom (m/128, b/4) at ((m/128) * (K/128) + b/4) * 512).  "_R" copies are blocked along the row
 * (MN = rows, K = columns), "_C" copies along the column (MN = columns, K = rows).
 * W13_R stores each expert's rows in 128-row blocks of [64 gate rows | 64 up rows].  Under
 * MOE_FP8_FP4, W13_R and W2_R hold packed E2M1 values, two per byte (the even column in the low
 * nibble), half the bytes of a row; their scale arrays keep the layout above. */
enum {
    MOE_VIEW_MX_X_R = 32, MOE_VIEW_MX_X_R_SF, MOE_VIEW_MX_X_C, MOE_VIEW_MX_X_C_SF,
    MOE_VIEW_MX_H_R, MOE_VIEW_MX_H_R_SF,
    MOE_VIEW_MX_DY_R, MOE_VIEW_MX_DY_R_SF, MOE_VIEW_MX_DY_C, MOE_VIEW_MX_DY_C_SF,
    MOE_VIEW_MX_DG_R, MOE_VIEW_MX_DG_R_SF, MOE_VIEW_MX_DG_C, MOE_VIEW_MX_DG_C_SF,
    MOE_VIEW_MX_HW_C, MOE_VIEW_MX_HW_C_SF,
    MOE_VIEW_MX_W13_R, MOE_VIEW_MX_W13_R_SF, MOE_VIEW_MX_W13_C, MOE_VIEW_MX_W13_C_SF,
    MOE_VIEW_MX_W2_R, MOE_VIEW_MX_W2_R_SF, MOE_VIEW_MX_W2_C, MOE_VIEW_MX_W2_C_SF,
    MOE_VIEW_MX_END_
};
int moe_scratch_view(const moe_desc* desc, int view, uint64_t* offset, uint64_t* bytes);

/* Per-kernel timing.  With tracing on, every launch made by moe_fwd / moe_bwd is bracketed by a
 * pair of CUDA events recorded on the caller's stream (so the times are those of the launches as
 * they run in the step).  moe_trace_read synchronises on the recorded events, and for each kernel
 * kind i < *n fills names[i] (static strings), launches[i] and total_ms[i]; *n is set to the number
 * of kinds seen.  moe_trace_reset clears the counters.  Not thread-safe. */
int moe_trace_enable(int on);
int moe_trace_reset(void);
int moe_trace_read(const char** names, int64_t* launches, double* total_ms, int* n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LAYER_H */
