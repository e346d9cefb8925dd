// moe_api.cu - the C ABI of the MoE layer: argument checks, scratch layout, the forward and
// backward launch sequences, device status, per-kernel tracing.
//
// Forward (one call, all on the caller's stream, no host synchronisation):
//   routing -> gather x -> [g|u] = X W13^T, w h = w silu(g) u -> Ypart = (w h) W2^T -> y = combine
//   (MXFP8: h is quantised unweighted and the down epilogue applies w)
// Backward of <dy, y>:
//   [routing -> gather x -> [g|u] (and w h) recompute]  (skipped under MOE_FLAG_REUSE_FWD)
//   gather dy -> dA = dY W2 with the SwiGLU backward in the epilogue ([dg|du], <dA, h>; MXFP8
//   also the E4M3 copy of w h) -> dXpart = [dg|du] W13 -> dW2 = dY^T (w h) -> dW13 = [dg|du]^T X
//   -> dx = combine(dXpart), dtopk_w = sum of the <dA, h> partials.
// The single call per direction and the GPU-only scratch in place of intermediate tensors follow
// MarkTechPost, "Prime Intellect Releases Prime Mega MoE", section "How does the fused kernel
// work?"; the shape rules follow ic.work analysis, section "算子下沉时代的硬件死锁暗礁".
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace moe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
static_assert(sizeof(MxLayout) == 24 * sizeof(size_t), "MxLayout: 12 operands of (values, scales) offsets");

bool make_layout(const moe_desc* d, Layout* L) {
    if (!d) return false;
    if (d->T < 0 || d->H <= 0 || d->I <= 0 || d->E <= 0 || d->k <= 0) return false;
    if (d->H % 256 != 0 || d->I % 128 != 0 || d->k > d->E || d->E > kMaxExperts) return false;
    const int64_t S = d->T * d->k;
    const int64_t rows = (S + kBM - 1) / kBM * kBM + (int64_t)kBM * d->E;  // a multiple of 128
    if (rows >= (int64_t)INT32_MAX / 2) return false;
    L->T = d->T; L->H = d->H; L->I = d->I; L->E = d->E; L->k = d->k; L->S = S; L->rows = rows;
    L->nb_route = (S + kRouteChunk - 1) / kRouteChunk;
    L->fp4w = d->precision == MOE_FP8_FP4;
    L->mx_fwd = d->precision == MOE_MXFP8 || L->fp4w;
    L->mx_bwd = d->precision == MOE_MXFP8 || d->precision == MOE_FP8_BWD;
    L->mx_on = L->mx_fwd || L->mx_bwd;
    L->n_dtw = 2 * (d->I / (L->mx_bwd ? 128 : bwd_down_bn(d->I)));  // two column halves per n-tile
    const size_t A = 4096;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes, A); return at; };
    L->ctrl = take(256);
    L->hist = take((size_t)std::max<int64_t>(L->nb_route, 1) * d->E * 4);
    L->cnt = take((size_t)d->E * 4);
    L->off = take((size_t)(d->E + 1) * 4);
    L->pad_off = take((size_t)(d->E + 1) * 4);
    L->mtile = take((size_t)(d->E + 1) * 4);
    L->order = take((size_t)d->E * 4);
    L->base = take((size_t)std::max<int64_t>(L->nb_route, 1) * d->E * 4);
    L->perm = take((size_t)S * 4);
    L->inv = take((size_t)S * 4);
    L->pos = take((size_t)S * 4);
    L->row_slot = take((size_t)rows * 4);
    L->xperm = take((size_t)rows * d->H * 2);
    L->hid = take((size_t)rows * d->I * 2);
    L->gu = take((size_t)rows * 2 * d->I * 2);
    // also dXpart in the backward, and the fused combine's fp32 [T, H] accumulator
    L->ypart = take(std::max((size_t)rows * d->H * 2, (size_t)d->T * d->H * 4));
    L->dyperm = take((size_t)rows * d->H * 2);
    L->dg = take((size_t)rows * 2 * d->I * 2);
    L->hw = L->hid;   // BF16: the gate/up epilogue stores w h there, and the backward reads it
    L->dtw = take((size_t)rows * L->n_dtw * 4);
    L->mx = MxLayout{};
    for (size_t& v : L->mx_bytes) v = 0;
    if (L->mx_on) {
        MxLayout& M = L->mx;
        const size_t H = d->H, I = d->I, E = d->E, R = rows;
        // regions in MxLayout field order: the values (vbits bits each), then one scale byte per 32
        int n = 0;
        auto q = [&](size_t elems, int vbits, size_t* data, size_t* sf) {
            L->mx_bytes[n++] = elems * vbits / 8;
            L->mx_bytes[n++] = elems / 32;
            *data = take(elems * vbits / 8);
            *sf = take(elems / 32);
        };
        const size_t F = L->mx_fwd ? 1 : 0;   // forward-only copies: empty without an MX forward
        const size_t B = L->mx_bwd ? 1 : 0;   // backward copies: empty without an MXFP8 backward
        const int wb = L->fp4w ? 4 : 8;       // bits of the forward weights' values
        q(F * R * H, 8, &M.x_r, &M.x_r_sf);
        q(B * R * H, 8, &M.x_c, &M.x_c_sf);
        q(F * R * I, 8, &M.h_r, &M.h_r_sf);
        q(B * R * H, 8, &M.dy_r, &M.dy_r_sf);
        q(B * R * H, 8, &M.dy_c, &M.dy_c_sf);
        q(B * R * 2 * I, 8, &M.dg_r, &M.dg_r_sf);
        q(B * R * 2 * I, 8, &M.dg_c, &M.dg_c_sf);
        q(B * R * I, 8, &M.hw_c, &M.hw_c_sf);
        q(F * E * 2 * I * H, wb, &M.w13_r, &M.w13_r_sf);
        q(B * E * 2 * I * H, 8, &M.w13_c, &M.w13_c_sf);
        q(F * E * H * I, wb, &M.w2_r, &M.w2_r_sf);
        q(B * E * H * I, 8, &M.w2_c, &M.w2_c_sf);
    }
    L->total = o;
    return true;
}

// ------------------------------------------------------------------------------------------
// tracing
// ------------------------------------------------------------------------------------------
static const char* kTraceNames[kTraceKinds] = {
    "route_hist", "route_scan", "route_place", "gather_rows", "combine_rows", "mx_quant", "reduce_finish", "mx_quant_rows",
    "gemm_fwd_gate_up_swiglu", "gemm_fwd_gate_up_save", "gemm_fwd_down_weighted", "gemm_bwd_down_swiglu_bwd",
    "gemm_bwd_gate_up", "gemm_wgrad_down", "gemm_wgrad_gate_up", "gemm_fwd_down_reduce",
    "gemm_mx_fwd_gate_up_swiglu", "gemm_mx_fwd_gate_up_save", "gemm_mx_fwd_down_weighted",
    "gemm_mx_bwd_down_swiglu_bwd", "gemm_mx_bwd_gate_up", "gemm_mx_wgrad_down", "gemm_mx_wgrad_gate_up",
    "gemm_mx_fwd_down_reduce",
};

struct TraceRec {
    int kind;
    cudaEvent_t a, b;
};
static bool g_trace_on = false;
static std::vector<TraceRec> g_trace;
static int64_t g_trace_launches[kTraceKinds];
static double g_trace_ms[kTraceKinds];
static cudaEvent_t g_pending_begin = nullptr;

void trace_begin(cudaStream_t st, int kind) {
    if (!g_trace_on) return;
    cudaEventCreate(&g_pending_begin);
    cudaEventRecord(g_pending_begin, st);
}
void trace_end(cudaStream_t st, int kind) {
    if (!g_trace_on || !g_pending_begin) return;
    cudaEvent_t e;
    cudaEventCreate(&e);
    cudaEventRecord(e, st);
    g_trace.push_back({kind, g_pending_begin, e});
    g_pending_begin = nullptr;
}
static void trace_flush() {
    for (auto& r : g_trace) {
        float ms = 0.f;
        cudaEventSynchronize(r.b);
        if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess && r.kind >= 0 && r.kind < kTraceKinds) {
            g_trace_launches[r.kind] += 1;
            g_trace_ms[r.kind] += ms;
        }
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_trace.clear();
}

// ------------------------------------------------------------------------------------------
// argument checks
// ------------------------------------------------------------------------------------------
static int num_sms_current() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        cached[dev] = n;
    }
    return cached[dev];
}

static int check_tensor(const moe_tensor* t, int dtype, int ndim, int64_t s0, int64_t s1, int64_t s2) {
    if (!t) return MOE_ERR_NULL;
    if (t->ndim != ndim) return MOE_ERR_SHAPE;
    const int64_t want[3] = {s0, s1, s2};
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] != want[i]) return MOE_ERR_SHAPE;
    if (t->dtype != dtype) return MOE_ERR_DTYPE;
    int64_t numel = 1;
    for (int i = 0; i < ndim; ++i) numel *= t->shape[i];
    if (numel == 0) return MOE_OK;  // an empty tensor is never dereferenced
    int64_t expect = 1;
    for (int i = ndim - 1; i >= 0; --i) {
        if (t->shape[i] > 1 && t->stride[i] != expect) return MOE_ERR_LAYOUT;
        expect *= t->shape[i];
    }
    if (!t->data) return MOE_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0) return MOE_ERR_ALIGN;
    return MOE_OK;
}

static int check_weight_grad(const moe_tensor* t, int ndim, int64_t a, int64_t b, int64_t c, bool* f32) {
    if (!t) return MOE_ERR_NULL;
    *f32 = t->dtype == MOE_DT_F32;
    return check_tensor(t, *f32 ? MOE_DT_F32 : MOE_DT_BF16, ndim, a, b, c);
}

static int check_desc_scratch(moe_scratch* s, Layout* L) {
    if (!s) return MOE_ERR_NULL;
    const moe_desc* d = &s->desc;
    if (d->precision != MOE_BF16 && d->precision != MOE_MXFP8 && d->precision != MOE_FP8_BWD &&
        d->precision != MOE_FP8_FP4)
        return MOE_ERR_UNSUPPORTED;
    if (!make_layout(d, L)) return MOE_ERR_SHAPE;
    if (!s->data) return MOE_ERR_SCRATCH;
    if (reinterpret_cast<uintptr_t>(s->data) % 256 != 0) return MOE_ERR_SCRATCH;
    if (s->bytes < L->total) return MOE_ERR_SCRATCH;
    return MOE_OK;
}

// Combines v into the hash h; the splitmix64 finaliser spreads every input bit over the whole
// word, so that a change in any input (an epoch advanced by one included) changes the high bits.
static uint64_t mix(uint64_t h, uint64_t v) {
    uint64_t z = h ^ (v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2));
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
// Tags of what a scratch buffer holds: the inputs' addresses and the caller's epoch (advanced
// whenever those buffers may have changed in place), never the device data itself.
static uint64_t fwd_tag(const moe_scratch* s, const void* x, const void* idx, const void* w, const void* w13,
                        const void* w2) {
    const moe_desc* d = &s->desc;
    uint64_t h = 0x6D6F655F66776400ull;
    for (uint64_t v : {(uint64_t)d->T, (uint64_t)d->H, (uint64_t)d->I, (uint64_t)d->E, (uint64_t)d->k,
                       (uint64_t)d->precision, (uint64_t)(uintptr_t)x, (uint64_t)(uintptr_t)idx,
                       (uint64_t)(uintptr_t)w, (uint64_t)(uintptr_t)w13, (uint64_t)(uintptr_t)w2, s->epoch})
        h = mix(h, v);
    return h | 1ull;  // never 0 (0 = no saved forward)
}

static uint64_t weights_tag(const moe_scratch* s, const void* w13, const void* w2) {
    const moe_desc* d = &s->desc;
    uint64_t h = 0x6D6F655F77717500ull;
    for (uint64_t v : {(uint64_t)d->H, (uint64_t)d->I, (uint64_t)d->E, (uint64_t)d->precision,
                       (uint64_t)(uintptr_t)w13, (uint64_t)(uintptr_t)w2, s->epoch})
        h = mix(h, v);
    return h | 1ull;
}

// MOE_FLAG_REUSE_WEIGHTS is honoured only if this scratch holds copies of these weights made at
// the current epoch; checked before anything is launched.
static int check_weight_reuse(const moe_scratch* s, bool needs_copies, const void* w13, const void* w2) {
    if (!needs_copies || !(s->desc.flags & MOE_FLAG_REUSE_WEIGHTS)) return MOE_OK;
    return s->state[1] == weights_tag(s, w13, w2) ? MOE_OK : MOE_ERR_STATE;
}

// One side stream per device (non-blocking) with a fork and a join event, created on first use
// and kept until exit; null if they cannot be created (the work then stays on the caller's stream).
// Calls on the same device share them, so, as for a shared scratch buffer, calls on one device must
// be ordered on one stream.
struct SideStream {
    cudaStream_t st;
    cudaEvent_t fork, join;
};
static SideStream* side_stream() {
    static std::mutex mu;
    static SideStream streams[64];
    static int state[64] = {0};   // 0: not tried, 1: ready, -1: unavailable
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (state[dev] == 0) {
        SideStream& s = streams[dev];
        const bool ok = cudaStreamCreateWithFlags(&s.st, cudaStreamNonBlocking) == cudaSuccess &&
                        cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) == cudaSuccess &&
                        cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) == cudaSuccess;
        state[dev] = ok ? 1 : -1;
    }
    return state[dev] == 1 ? &streams[dev] : nullptr;
}

static Ctx make_ctx(cudaStream_t st, moe_scratch* s, const Layout* L, int nsm, const void* topk_w) {
    char* base = reinterpret_cast<char*>(s->data);
    Ctx c{st, base, L, reinterpret_cast<int*>(base + L->ctrl), nsm, reinterpret_cast<const float*>(topk_w)};
    c.wait_limit = (long long)s->state[2];
    c.test_flags = (uint32_t)s->state[3];
    return c;
}

// MX copies of the weights: for an MX forward W13 blocked along H (gate/up row blocks) and W2
// along I, in E4M3 or, for the FP8 x FP4 forward, in E2M1; for an MXFP8 backward W13 blocked
// along 2I and W2 along H.  Skipped when the caller
// states the weights are unchanged since the call that made these copies on this scratch
// (MOE_FLAG_REUSE_WEIGHTS).
static int mx_weights(const Ctx& c, moe_scratch* s, const void* W13, const void* W2) {
    const Layout& L = *c.L;
    const MxLayout& M = L.mx;
    const moe_desc* d = &s->desc;
    const uint64_t tag = weights_tag(s, W13, W2);
    if (d->flags & MOE_FLAG_REUSE_WEIGHTS) return s->state[1] == tag ? MOE_OK : MOE_ERR_STATE;
    char* b = c.base;
    auto fw = [&](size_t off) { return L.mx_fwd ? b + off : nullptr; };
    auto bw = [&](size_t off) { return L.mx_bwd ? b + off : nullptr; };
    if (launch_mx_quant(c, W13, L.E * 2 * L.I, (int)L.H, nullptr, fw(M.w13_r), fw(M.w13_r_sf), bw(M.w13_c),
                        bw(M.w13_c_sf), (int)L.I, nullptr, L.fp4w) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_mx_quant(c, W2, L.E * L.H, (int)L.I, nullptr, fw(M.w2_r), fw(M.w2_r_sf), bw(M.w2_c), bw(M.w2_c_sf), 0,
                        nullptr, L.fp4w) != cudaSuccess)
        return MOE_ERR_CUDA;
    s->state[1] = tag;
    return MOE_OK;
}

// activation quantisation over the padded routed rows (count read on the device); with `gather`
// the source is the caller's [T, C] tensor, dispatched on the fly through row_slot
static cudaError_t mx_rows(const Ctx& c, const void* src, bool gather, int C, size_t qr, size_t qr_sf, size_t qc,
                           size_t qc_sf) {
    const Layout& L = *c.L;
    char* b = c.base;
    const int* tiles = reinterpret_cast<const int*>(b + L.mtile) + L.E;
    if (gather && qr && !qc) {
        // the row-blocked copy alone runs token-major; with the token-blocked copy (which needs the
        // dispatched order) one dispatched-order pass makes both, which measured faster on GB300
        // than the token-major row pass plus a column-only pass (0.19 against 0.07 + 0.10 ms)
        return launch_mx_rows_token(c, src, reinterpret_cast<const int*>(b + L.pos),
                                    reinterpret_cast<const int*>(b + L.row_slot), tiles, b + qr, b + qr_sf);
    }
    return launch_mx_quant(c, src, L.rows, C, tiles, qr ? b + qr : nullptr, qr ? b + qr_sf : nullptr,
                           qc ? b + qc : nullptr, qc ? b + qc_sf : nullptr, 0,
                           gather ? reinterpret_cast<const int*>(b + L.row_slot) : nullptr);
}

}  // namespace moe

using namespace moe;

#define MOE_TRY_CUDA(expr)                              \
    do {                                                \
        if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
    } while (0)

extern "C" {

size_t moe_scratch_bytes(const moe_desc* desc) {
    Layout L;
    return make_layout(desc, &L) ? L.total : 0;
}

int moe_fwd(const moe_tensor* x, const moe_tensor* topk_idx, const moe_tensor* topk_w, const moe_tensor* W13,
            const moe_tensor* W2, moe_tensor* y, moe_scratch* scratch, void* stream) {
    Layout L;
    int rc = check_desc_scratch(scratch, &L);
    if (rc) return rc;
    const moe_desc* d = &scratch->desc;
    const int64_t T = d->T, H = d->H, I = d->I, E = d->E, k = d->k;
    if ((rc = check_tensor(x, MOE_DT_BF16, 2, T, H, 0))) return rc;
    if ((rc = check_tensor(topk_idx, MOE_DT_I32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(topk_w, MOE_DT_F32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(W13, MOE_DT_BF16, 3, E, 2 * I, H))) return rc;
    if ((rc = check_tensor(W2, MOE_DT_BF16, 3, E, H, I))) return rc;
    if ((rc = check_tensor(y, MOE_DT_BF16, 2, T, H, 0))) return rc;
    if (T > 0 && (rc = check_weight_reuse(scratch, L.mx_fwd, W13->data, W2->data))) return rc;
    const uint64_t tag = fwd_tag(scratch, x->data, topk_idx->data, topk_w->data, W13->data, W2->data);
    const bool save = (d->flags & MOE_FLAG_SAVE_GU) != 0;
    const bool fused = (d->flags & MOE_FLAG_FUSED_COMBINE) != 0;
    if (fused && L.mx_fwd) return MOE_ERR_UNSUPPORTED;   // the fused combine has a BF16 epilogue only
    if (T == 0) {
        scratch->state[0] = save ? tag : 0;
        return MOE_OK;
    }
    const int nsm = num_sms_current();
    if (nsm <= 0) return MOE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* base = reinterpret_cast<char*>(scratch->data);
    const Ctx c = make_ctx(st, scratch, &L, nsm, topk_w->data);
    MOE_TRY_CUDA(launch_routing(c, reinterpret_cast<const int32_t*>(topk_idx->data)));
    if (L.mx_fwd) {
        // dispatch and quantise in one pass; a forward that saves for the backward also makes the
        // token-blocked copy the weight gradient of W13 reads
        const MxLayout& M = L.mx;
        if ((rc = mx_weights(c, scratch, W13->data, W2->data))) return rc;
        const bool xc = save && L.mx_bwd;
        MOE_TRY_CUDA(mx_rows(c, x->data, true, (int)H, M.x_r, M.x_r_sf, xc ? M.x_c : 0, xc ? M.x_c_sf : 0));
    } else {
        MOE_TRY_CUDA(launch_gather(c, x->data, base + L.xperm, nullptr, nullptr));
    }
    MOE_TRY_CUDA(launch_gemm(c, GemmKind::FwdGateUp, W13->data, nullptr, false, save));  // MXFP8: emits E4M3 h
    if (fused) {
        // the down product's epilogue adds w o into an fp32 accumulator by token; no Ypart rows
        MOE_TRY_CUDA(launch_reduce_zero(c));
        MOE_TRY_CUDA(launch_gemm(c, GemmKind::FwdDownReduce, W2->data, nullptr, false, false));
        MOE_TRY_CUDA(launch_reduce_finish(c, y->data));
    } else {
        MOE_TRY_CUDA(launch_gemm(c, GemmKind::FwdDown, W2->data, nullptr, false, false));
        MOE_TRY_CUDA(launch_combine(c, base + L.ypart, y->data, nullptr));
    }
    // routing and dispatched rows are rewritten identically for the same inputs, so an earlier
    // saved [g|u] of these inputs stays valid; anything else invalidates it
    if (save)
        scratch->state[0] = tag;
    else if (scratch->state[0] != tag)
        scratch->state[0] = 0;
    return MOE_OK;
}

int moe_bwd(const moe_tensor* dy, const moe_tensor* x, const moe_tensor* topk_idx, const moe_tensor* topk_w,
            const moe_tensor* W13, const moe_tensor* W2, moe_tensor* dx, moe_tensor* dW13, moe_tensor* dW2,
            moe_tensor* dtopk_w, moe_scratch* scratch, void* stream) {
    Layout L;
    int rc = check_desc_scratch(scratch, &L);
    if (rc) return rc;
    if (L.fp4w) return MOE_ERR_UNSUPPORTED;   // the FP8 x FP4 layer is forward only
    const moe_desc* d = &scratch->desc;
    const int64_t T = d->T, H = d->H, I = d->I, E = d->E, k = d->k;
    bool f32_13 = false, f32_2 = false;
    if ((rc = check_tensor(dy, MOE_DT_BF16, 2, T, H, 0))) return rc;
    if ((rc = check_tensor(x, MOE_DT_BF16, 2, T, H, 0))) return rc;
    if ((rc = check_tensor(topk_idx, MOE_DT_I32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(topk_w, MOE_DT_F32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(W13, MOE_DT_BF16, 3, E, 2 * I, H))) return rc;
    if ((rc = check_tensor(W2, MOE_DT_BF16, 3, E, H, I))) return rc;
    if ((rc = check_tensor(dx, MOE_DT_BF16, 2, T, H, 0))) return rc;
    if ((rc = check_weight_grad(dW13, 3, E, 2 * I, H, &f32_13))) return rc;
    if ((rc = check_weight_grad(dW2, 3, E, H, I, &f32_2))) return rc;
    if ((rc = check_tensor(dtopk_w, MOE_DT_F32, 2, T, k, 0))) return rc;
    const uint64_t tag = fwd_tag(scratch, x->data, topk_idx->data, topk_w->data, W13->data, W2->data);
    const bool reuse = (d->flags & MOE_FLAG_REUSE_FWD) != 0;
    if (reuse && scratch->state[0] != tag) return MOE_ERR_STATE;
    if (T > 0 && (rc = check_weight_reuse(scratch, L.mx_on, W13->data, W2->data))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {
        MOE_TRY_CUDA(cudaMemsetAsync(dW13->data, 0, (size_t)E * 2 * I * H * (f32_13 ? 4 : 2), st));
        MOE_TRY_CUDA(cudaMemsetAsync(dW2->data, 0, (size_t)E * H * I * (f32_2 ? 4 : 2), st));
        return MOE_OK;
    }
    const int nsm = num_sms_current();
    if (nsm <= 0) return MOE_ERR_CUDA;
    char* base = reinterpret_cast<char*>(scratch->data);
    const Ctx c = make_ctx(st, scratch, &L, nsm, topk_w->data);
    const MxLayout& M = L.mx;
    if (L.mx_on && (rc = mx_weights(c, scratch, W13->data, W2->data))) return rc;
    if (!reuse) {
        MOE_TRY_CUDA(launch_routing(c, reinterpret_cast<const int32_t*>(topk_idx->data)));
        if (L.mx_fwd)
            MOE_TRY_CUDA(mx_rows(c, x->data, true, (int)H, M.x_r, M.x_r_sf, M.x_c, M.x_c_sf));
        else if (L.mx_bwd)
            MOE_TRY_CUDA(launch_gather(c, x->data, base + L.xperm, nullptr, nullptr));
        else
            MOE_TRY_CUDA(launch_gather(c, x->data, base + L.xperm, dy->data, base + L.dyperm));
        // a BF16 backward also needs the forward's w h (its W2 weight-gradient operand); with an
        // MXFP8 backward the SwiGLU-backward epilogue makes that operand's E4M3 copy itself
        MOE_TRY_CUDA(launch_gemm(c, L.mx_on ? GemmKind::FwdGateUpSaveOnly : GemmKind::FwdGateUp, W13->data,
                                 nullptr, false, true));
    } else if (!L.mx_bwd) {
        MOE_TRY_CUDA(launch_gather(c, dy->data, base + L.dyperm, nullptr, nullptr));
    }
    if (L.mx_bwd) {
        // a BF16 forward (fp8_bwd) made no MXFP8 copy of x: the W13 weight gradient's comes here
        if (!L.mx_fwd) MOE_TRY_CUDA(mx_rows(c, x->data, true, (int)H, 0, 0, M.x_c, M.x_c_sf));
        MOE_TRY_CUDA(mx_rows(c, dy->data, true, (int)H, M.dy_r, M.dy_r_sf, M.dy_c, M.dy_c_sf));
    }
    // MXFP8: the SwiGLU-backward epilogue emits the E4M3 copies of [dg|du] and w h directly
    MOE_TRY_CUDA(launch_gemm(c, GemmKind::BwdDown, W2->data, nullptr, false, false));
    MOE_TRY_CUDA(launch_gemm(c, GemmKind::BwdGateUp, W13->data, nullptr, false, false));
    // dx = combine(dXpart) needs only the product above, and the two weight gradients do not read
    // what it reads or writes: it runs on the device's side stream (forked and joined by events,
    // so the caller's stream orders everything after this call as before), where its HBM-bound
    // sum overlaps the tensor-bound weight-gradient products
    SideStream* side = side_stream();
    if (side) {
        Ctx cs = c;
        cs.st = side->st;
        MOE_TRY_CUDA(cudaEventRecord(side->fork, st));
        MOE_TRY_CUDA(cudaStreamWaitEvent(side->st, side->fork, 0));
        MOE_TRY_CUDA(launch_combine(cs, base + L.ypart, dx->data, reinterpret_cast<float*>(dtopk_w->data)));
        MOE_TRY_CUDA(cudaEventRecord(side->join, side->st));
    }
    MOE_TRY_CUDA(launch_gemm(c, GemmKind::WgradDown, nullptr, dW2->data, f32_2, false));
    MOE_TRY_CUDA(launch_gemm(c, GemmKind::WgradGateUp, nullptr, dW13->data, f32_13, false));
    if (side)
        MOE_TRY_CUDA(cudaStreamWaitEvent(st, side->join, 0));
    else
        MOE_TRY_CUDA(launch_combine(c, base + L.ypart, dx->data, reinterpret_cast<float*>(dtopk_w->data)));
    scratch->state[0] = tag;  // routing, dispatched x and [g|u] now describe these inputs
    return MOE_OK;
}

int moe_read_device_status(moe_scratch* scratch, void* stream, int* status) {
    if (!scratch || !scratch->data || !status) return MOE_ERR_NULL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    MOE_TRY_CUDA(cudaMemcpyAsync(&v, scratch->data, sizeof(int), cudaMemcpyDeviceToHost, st));
    MOE_TRY_CUDA(cudaMemsetAsync(scratch->data, 0, sizeof(int), st));
    MOE_TRY_CUDA(cudaStreamSynchronize(st));
    *status = v;
    return MOE_OK;
}

int moe_set_wait_limit(moe_scratch* scratch, int64_t wait_cycles, uint32_t test_flags) {
    if (!scratch) return MOE_ERR_NULL;
    if (wait_cycles < 0) return MOE_ERR_SHAPE;
    scratch->state[2] = (uint64_t)wait_cycles;
    scratch->state[3] = test_flags & MOE_TEST_WITHHOLD_LOADS;
    return MOE_OK;
}

static int router_shape(const moe_tensor* logits_like, const moe_tensor* idx, int64_t* T, int64_t* E, int64_t* k) {
    if (!logits_like || !idx) return MOE_ERR_NULL;
    if (logits_like->ndim != 2 || idx->ndim != 2) return MOE_ERR_SHAPE;
    *T = logits_like->shape[0];
    *E = logits_like->shape[1];
    *k = idx->shape[1];
    if (*T < 0 || *T >= (int64_t)INT32_MAX / 32 || idx->shape[0] != *T) return MOE_ERR_SHAPE;
    if (*k < 1 || *k > 32 || *E < *k || *E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int moe_router_fwd(const moe_tensor* logits, moe_tensor* topk_idx, moe_tensor* topk_w, void* stream) {
    int64_t T, E, k;
    int rc = router_shape(logits, topk_idx, &T, &E, &k);
    if (rc) return rc;
    if ((rc = check_tensor(logits, MOE_DT_F32, 2, T, E, 0))) return rc;
    if ((rc = check_tensor(topk_idx, MOE_DT_I32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(topk_w, MOE_DT_F32, 2, T, k, 0))) return rc;
    MOE_TRY_CUDA(launch_router_fwd(reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<const float*>(logits->data),
                                   (int)T, (int)E, (int)k, reinterpret_cast<int*>(topk_idx->data),
                                   reinterpret_cast<float*>(topk_w->data)));
    return MOE_OK;
}

int moe_router_bwd(const moe_tensor* topk_idx, const moe_tensor* topk_w, const moe_tensor* dtopk_w, moe_tensor* dlogits,
                   void* stream) {
    int64_t T, E, k;
    int rc = router_shape(dlogits, topk_idx, &T, &E, &k);
    if (rc) return rc;
    if ((rc = check_tensor(topk_idx, MOE_DT_I32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(topk_w, MOE_DT_F32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(dtopk_w, MOE_DT_F32, 2, T, k, 0))) return rc;
    if ((rc = check_tensor(dlogits, MOE_DT_F32, 2, T, E, 0))) return rc;
    MOE_TRY_CUDA(launch_router_bwd(reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<const int*>(topk_idx->data),
                                   reinterpret_cast<const float*>(topk_w->data),
                                   reinterpret_cast<const float*>(dtopk_w->data), (int)T, (int)E, (int)k,
                                   reinterpret_cast<float*>(dlogits->data)));
    return MOE_OK;
}

const char* moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL: return "a required pointer is NULL";
        case MOE_ERR_SHAPE: return "shape rules broken (H % 256, I % 128, 1 <= k <= E <= 1024, tensor shapes)";
        case MOE_ERR_DTYPE: return "a tensor has the wrong element type";
        case MOE_ERR_LAYOUT: return "a tensor is not contiguous row-major";
        case MOE_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case MOE_ERR_SCRATCH: return "scratch missing, misaligned or smaller than moe_scratch_bytes";
        case MOE_ERR_STATE: return "MOE_FLAG_REUSE_FWD without a matching forward saved in scratch";
        case MOE_ERR_UNSUPPORTED: return "precision or size not supported";
        case MOE_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case MOE_ERR_DEVICE: return "the device status word reports an error";
        default: return "unknown status code";
    }
}

int moe_scratch_view(const moe_desc* desc, int view, uint64_t* offset, uint64_t* bytes) {
    Layout L;
    if (!offset || !bytes) return MOE_ERR_NULL;
    if (!make_layout(desc, &L)) return MOE_ERR_SHAPE;
    const uint64_t R = L.rows, S = L.S, E = L.E, H = L.H, I = L.I;
    switch (view) {
        case MOE_VIEW_COUNTS: *offset = L.cnt; *bytes = E * 4; break;
        case MOE_VIEW_OFFSETS: *offset = L.off; *bytes = (E + 1) * 4; break;
        case MOE_VIEW_PERM: *offset = L.perm; *bytes = S * 4; break;
        case MOE_VIEW_INV: *offset = L.inv; *bytes = S * 4; break;
        case MOE_VIEW_PAD_OFFSETS: *offset = L.pad_off; *bytes = (E + 1) * 4; break;
        case MOE_VIEW_XPERM: *offset = L.xperm; *bytes = R * H * 2; break;
        case MOE_VIEW_HID: *offset = L.hid; *bytes = R * I * 2; break;
        case MOE_VIEW_GU: *offset = L.gu; *bytes = R * 2 * I * 2; break;
        case MOE_VIEW_YPART: *offset = L.ypart; *bytes = R * H * 2; break;
        case MOE_VIEW_DG: *offset = L.dg; *bytes = R * 2 * I * 2; break;
        case MOE_VIEW_HW: *offset = L.hw; *bytes = R * I * 2; break;
        case MOE_VIEW_DYPERM: *offset = L.dyperm; *bytes = R * H * 2; break;
        default: {
            if (!L.mx_on || view < MOE_VIEW_MX_X_R || view >= MOE_VIEW_MX_END_) return MOE_ERR_SHAPE;
            // MxLayout lists the regions in view order: value array then scales, per operand
            const int i = view - MOE_VIEW_MX_X_R;
            *offset = reinterpret_cast<const size_t*>(&L.mx)[i];
            *bytes = L.mx_bytes[i];
        }
    }
    return MOE_OK;
}

int moe_trace_enable(int on) {
    g_trace_on = on != 0;
    return MOE_OK;
}

int moe_trace_reset(void) {
    trace_flush();
    for (int i = 0; i < kTraceKinds; ++i) {
        g_trace_launches[i] = 0;
        g_trace_ms[i] = 0.0;
    }
    return MOE_OK;
}

int moe_trace_read(const char** names, int64_t* launches, double* total_ms, int* n) {
    if (!n) return MOE_ERR_NULL;
    trace_flush();
    int cap = *n, out = 0;
    for (int i = 0; i < kTraceKinds; ++i) {
        if (!g_trace_launches[i]) continue;
        if (out < cap) {
            if (names) names[out] = kTraceNames[i];
            if (launches) launches[out] = g_trace_launches[i];
            if (total_ms) total_ms[out] = g_trace_ms[i];
        }
        ++out;
    }
    *n = out;
    return MOE_OK;
}

}  // extern "C"
