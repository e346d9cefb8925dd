// gemm.cu - persistent grouped GEMMs of the MoE layer on the 5th-generation tensor cores.
//
// The pages' fused layer runs the two expert linear layers with SwiGLU between them and combines
// by routing weight (MarkTechPost, "Prime Intellect Releases Prime Mega MoE", section "How does
// the fused kernel work?"); a grouped GEMM packs many differently sized per-expert products into
// one launch indexed by group offsets (kongchang.com, "Prime Intellect推出Prime Mega MoE", section
// "为什么 MoE 训练特别需要融合内核").  The backward adds the activation- and weight-gradient
// products (ic.work analysis, section "从 3.11 倍到 1.32 倍的性能漏斗").
//
// One kernel template serves all seven products.  Each CTA is persistent (one per SM) and walks a
// static list of 128 x BN output tiles; its warps are specialised:
//   warp 0      TMA producer: loads 64-deep K slices of A and B into a 4-stage smem ring
//               (128-byte swizzle) and counts their bytes on a per-stage mbarrier;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16) into one of two
//               TMEM accumulators and releases each smem stage with tcgen05.commit;
//   warps 2..   epilogue (4 warps, or 8 for the SwiGLU backward): tcgen05.ld the finished
//               accumulator (one TMEM lane = one row per thread; warp w reads lane quarter w % 4,
//               and with 8 warps the two warps of a quarter take alternate 32-column chunks),
//               apply the fused epilogue and store to global memory, then release the
//               accumulator, so the epilogue of tile i overlaps the MMAs of tile i+1.
// Routed rows are laid out per expert padded to multiples of 128, so a row tile belongs to one
// expert and a weight-gradient K slice never crosses into the next expert's rows.
// Tile lists: "grouped-M" products (forward and data gradients) enumerate
// (m-tile, n-tile) with n fastest, so CTAs working at the same time share the A tile in L2;
// weight gradients enumerate (expert, m-tile, n-tile), experts in decreasing token count.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kStages = 4;
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KB

enum Epi : int { EPI_SWIGLU = 0, EPI_GU_ONLY, EPI_WEIGHTED, EPI_SWIGLU_BWD, EPI_PLAIN, EPI_WGRAD };

// Epilogue warps: the SwiGLU backward reads [g|u] and writes three outputs per element and needs
// two warps per TMEM lane quarter to keep up with the MMAs; the other epilogues use one.
template <int EPI>
constexpr int epi_warps() { return EPI == EPI_SWIGLU_BWD ? 8 : 4; }
template <int EPI>
constexpr int gemm_threads() { return 64 + 32 * epi_warps<EPI>(); }

struct GemmArgs {
    const int* mtile;          // [E+1] prefix of 128-row tiles per expert
    const int* order;          // [E] experts by decreasing count
    const int* row_slot;       // padded row -> slot (-1 on padding)
    const float* topk_w;       // [T*k]
    const __nv_bfloat16* gu;   // [rows, 2I] saved pre-activations (SwiGLU backward)
    void* out0;
    void* out1;
    float* dtw;                // [rows, 2 * n_tiles] partial <dA, h> per n-tile and column half
    int* status;
    int E, I;
    int n_tiles, m_tiles, k_blocks;
    int b_rows_e, b_up;
    int ld0;                   // row pitch of out0 in elements
    long long out_e_stride;    // weight gradients: elements per expert
    int out_f32, save_gu;
};

struct Tile {
    int e, m0, n0, nt, kb, row0;
};

__device__ __forceinline__ int find_expert(const int* s_mtile, int E, int gm) {
    int lo = 0, hi = E - 1;  // largest e with s_mtile[e] <= gm
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_mtile[mid] <= gm) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <int BN, bool WGRAD, bool SPLIT>
__device__ __forceinline__ Tile decode_tile(int L, const GemmArgs& a, const int* s_mtile) {
    Tile t;
    if (!WGRAD) {
        const int gm = L / a.n_tiles;
        t.nt = L - gm * a.n_tiles;
        t.m0 = gm * kBM;
        t.e = find_expert(s_mtile, a.E, gm);
        t.n0 = t.nt * (SPLIT ? BN / 2 : BN);
        t.kb = a.k_blocks;
        t.row0 = 0;
    } else {
        const int per = a.m_tiles * a.n_tiles;
        const int ei = L / per;
        const int rem = L - ei * per;
        const int mt = rem / a.n_tiles;
        t.nt = rem - mt * a.n_tiles;
        t.e = a.order[ei];
        t.m0 = mt * kBM;
        t.n0 = t.nt * BN;
        t.row0 = s_mtile[t.e] * kBM;
        t.kb = (s_mtile[t.e + 1] - s_mtile[t.e]) * (kBM / kBK);
    }
    return t;
}

// bounded wait without the abort short-cut, used only while draining after an abort
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitTimeoutCycles / 8) break;
}

template <int BN, bool A_MN, bool B_MN, bool SPLIT, bool WGRAD, int EPI>
__global__ void __launch_bounds__(gemm_threads<EPI>(), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs a) {
    constexpr int kBTileBytes = BN * kBK * 2;
    constexpr int kStageBytes = kATileBytes + kBTileBytes;
    constexpr uint32_t kIdesc = idesc_bf16(kBM, BN, A_MN, B_MN);
    constexpr uint32_t kTmemCols = 2 * BN;
    constexpr int kEpiWarps = epi_warps<EPI>();
    constexpr int kHalves = kEpiWarps / 4;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kATileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBTileBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* tfull = bars + 2 * kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    int* s_mtile = reinterpret_cast<int*>(tslot + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_mtile[i] = a.mtile[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, kEpiWarps * 32);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tslot;
    const int num_tiles = WGRAD ? a.E * a.m_tiles * a.n_tiles : s_mtile[a.E] * a.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int L = blockIdx.x; L < num_tiles && ok; L += gridDim.x) {
                const Tile t = decode_tile<BN, WGRAD, SPLIT>(L, a, s_mtile);
                for (int kb = 0; kb < t.kb; ++kb) {
                    if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag, a.status)) { ok = false; break; }
                    uint8_t* dA = sA + stage * kATileBytes;
                    uint8_t* dB = sB + stage * kBTileBytes;
                    mbar_arrive_expect_tx(full + stage, kStageBytes);
                    const int k0 = kb * kBK;
                    if (!A_MN) {
                        tma_load_2d(dA, &tmA, full + stage, k0, t.m0);
                    } else {
                        tma_load_2d(dA, &tmA, full + stage, t.m0, t.row0 + k0);
                        tma_load_2d(dA + 8192, &tmA, full + stage, t.m0 + 64, t.row0 + k0);
                    }
                    if (!B_MN) {
                        if (SPLIT) {
                            tma_load_2d(dB, &tmB, full + stage, k0, t.e * a.b_rows_e + t.n0);
                            tma_load_2d(dB + (BN / 2) * 128, &tmB, full + stage, k0, t.e * a.b_rows_e + a.b_up + t.n0);
                        } else {
                            tma_load_2d(dB, &tmB, full + stage, k0, t.e * a.b_rows_e + t.n0);
                        }
                    } else {
                        const int krow = WGRAD ? t.row0 + k0 : t.e * a.b_rows_e + k0;
#pragma unroll
                        for (int c = 0; c < BN / 64; ++c) tma_load_2d(dB + c * 8192, &tmB, full + stage, t.n0 + 64 * c, krow);
                    }
                    ++issued;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // wait (bounded) for the copies already in flight before the CTA exits
                for (int s = 0; s < kStages; ++s) {
                    if (issued > s) {
                        const long long n = (issued - s + kStages - 1) / kStages;
                        drain_wait(full + s, (uint32_t)((n - 1) & 1));
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            for (int L = blockIdx.x; L < num_tiles && ok; L += gridDim.x) {
                const Tile t = decode_tile<BN, WGRAD, SPLIT>(L, a, s_mtile);
                if (!mbar_wait(tempty + acc, acc_phase ^ 1u, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < t.kb; ++kb) {
                    if (!mbar_wait(full + stage, phase, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = a_base + stage * kATileBytes, sb = b_base + stage * kBTileBytes;
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks) {
                        const uint64_t ad = A_MN ? sdesc_sw128(sa + ks * 2048, 8192, 1024) : sdesc_sw128(sa + ks * 32, 16, 1024);
                        const uint64_t bd = B_MN ? sdesc_sw128(sb + ks * 2048, 8192, 1024) : sdesc_sw128(sb + ks * 32, 16, 1024);
                        mma_bf16(d_tmem, ad, bd, kIdesc, (kb | ks) != 0);
                    }
                    mma_commit(empty + stage);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (t.kb > 0) mma_commit(tfull + acc); else mbar_arrive(tfull + acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                mma_commit(drain);
                drain_wait(drain, 0);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;               // TMEM lanes [32*quarter, 32*quarter + 32)
        const int half = (warp - 2) >> 2;           // which alternate 32-column chunks (8 warps)
        const int r = quarter * 32 + lane;          // row of the tile owned by this thread
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int L = blockIdx.x; L < num_tiles; L += gridDim.x) {
            const Tile t = decode_tile<BN, WGRAD, SPLIT>(L, a, s_mtile);
            if (!mbar_wait(tfull + acc, acc_phase, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + lane_addr + (uint32_t)(acc * BN);
            const long long grow = (long long)t.m0 + r;
            float v[32];
            if constexpr (EPI == EPI_SWIGLU || EPI == EPI_GU_ONLY) {
                // columns [0, BN/2) = gate, [BN/2, BN) = up, for I-columns [n0, n0 + BN/2)
                __nv_bfloat16* hid = reinterpret_cast<__nv_bfloat16*>(a.out0);
                __nv_bfloat16* gu = reinterpret_cast<__nv_bfloat16*>(a.out1);
#pragma unroll 1
                for (int c = half; c < BN / 64; c += kHalves) {
                    float u[32];
                    tmem_ld32(tacc + 32 * c, v);
                    tmem_ld32(tacc + BN / 2 + 32 * c, u);
                    if (EPI == EPI_GU_ONLY || a.save_gu) {
                        store_bf16x32(gu + grow * (2LL * a.I) + t.n0 + 32 * c, v);
                        store_bf16x32(gu + grow * (2LL * a.I) + a.I + t.n0 + 32 * c, u);
                    }
                    if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = v[j] * sigmoidf_fast(v[j]) * u[j];
                        store_bf16x32(hid + grow * (long long)a.I + t.n0 + 32 * c, v);
                    }
                }
            } else if constexpr (EPI == EPI_WEIGHTED) {
                const int slot = a.row_slot[grow];
                const float w = slot >= 0 ? a.topk_w[slot] : 0.f;
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out0);
#pragma unroll 1
                for (int c = half; c < BN / 32; c += kHalves) {
                    tmem_ld32(tacc + 32 * c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= w;
                    store_bf16x32(out + grow * (long long)a.ld0 + t.n0 + 32 * c, v);
                }
            } else if constexpr (EPI == EPI_SWIGLU_BWD) {
                const int slot = a.row_slot[grow];
                const float w = slot >= 0 ? a.topk_w[slot] : 0.f;
                __nv_bfloat16* dG = reinterpret_cast<__nv_bfloat16*>(a.out0);
                __nv_bfloat16* hw = reinterpret_cast<__nv_bfloat16*>(a.out1);
                const __nv_bfloat16* gurow = a.gu + grow * (2LL * a.I);
                float dot = 0.f;
#pragma unroll 1
                for (int c = half; c < BN / 32; c += kHalves) {
                    float g[32], u[32];
                    tmem_ld32(tacc + 32 * c, v);   // dA
                    const int col = t.n0 + 32 * c;
                    load_bf16x32(gurow + col, g);
                    load_bf16x32(gurow + a.I + col, u);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float s = sigmoidf_fast(g[j]);
                        const float sl = g[j] * s;
                        const float h = sl * u[j];
                        dot += v[j] * h;
                        const float dh = w * v[j];
                        const float dg = dh * u[j] * (s + sl * (1.f - s));
                        const float du = dh * sl;
                        g[j] = dg;
                        u[j] = du;
                        v[j] = w * h;
                    }
                    store_bf16x32(dG + grow * (2LL * a.I) + col, g);
                    store_bf16x32(dG + grow * (2LL * a.I) + a.I + col, u);
                    store_bf16x32(hw + grow * (long long)a.I + col, v);
                }
                a.dtw[grow * (2 * a.n_tiles) + 2 * t.nt + half] = dot;
            } else if constexpr (EPI == EPI_PLAIN) {
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out0);
#pragma unroll 1
                for (int c = half; c < BN / 32; c += kHalves) {
                    tmem_ld32(tacc + 32 * c, v);
                    store_bf16x32(out + grow * (long long)a.ld0 + t.n0 + 32 * c, v);
                }
            } else {  // EPI_WGRAD
                const long long off = (long long)t.e * a.out_e_stride + grow * a.ld0 + t.n0;
#pragma unroll 1
                for (int c = half; c < BN / 32; c += kHalves) {
                    if (t.kb > 0) {
                        tmem_ld32(tacc + 32 * c, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.f;
                    }
                    if (a.out_f32)
                        store_f32x32(reinterpret_cast<float*>(a.out0) + off + 32 * c, v);
                    else
                        store_bf16x32(reinterpret_cast<__nv_bfloat16*>(a.out0) + off + 32 * c, v);
                }
            }
            tc_fence_before();
            mbar_arrive(tempty + acc);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------------------------------
// host side: tensor maps and launches
// ------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 tensor map over a row-major [outer, inner] array, box {64, box_rows}, 128B swizzle.
static bool tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool A_MN, bool B_MN, bool SPLIT, bool WGRAD, int EPI>
static cudaError_t run(const Ctx& c, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a) {
    auto kern = grouped_gemm_kernel<BN, A_MN, B_MN, SPLIT, WGRAD, EPI>;
    const size_t smem = 1024 + (size_t)kStages * (kATileBytes + BN * kBK * 2) + 128 + (size_t)(a.E + 1) * 4;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        1024 + kStages * (kATileBytes + BN * kBK * 2) + 128 + (kMaxExperts + 1) * 4);
    });
    if (attr_err != cudaSuccess) return attr_err;
    kern<<<c.num_sms, gemm_threads<EPI>(), smem, c.st>>>(ta, tb, a);
    return cudaGetLastError();
}

int bwd_down_bn(int64_t I) { return (I % 256 == 0) ? 256 : 128; }

cudaError_t launch_gemm(const Ctx& c, GemmKind kind, const void* W, void* out, bool out_f32, bool save_gu) {
    const Layout& L = *c.L;
    char* b = c.base;
    const int64_t H = L.H, I = L.I, E = L.E, R = L.rows;
    GemmArgs a{};
    a.mtile = reinterpret_cast<const int*>(b + L.mtile);
    a.order = reinterpret_cast<const int*>(b + L.order);
    a.row_slot = reinterpret_cast<const int*>(b + L.row_slot);
    a.topk_w = c.topk_w;
    a.gu = reinterpret_cast<const __nv_bfloat16*>(b + L.gu);
    a.status = c.status;
    a.E = (int)E;
    a.I = (int)I;
    a.out_f32 = out_f32 ? 1 : 0;
    a.save_gu = save_gu ? 1 : 0;
    CUtensorMap ta, tb;
    bool ok = true;
    cudaError_t err = cudaSuccess;
    const int trace_id = 5 + (int)kind;
    trace_begin(c.st, trace_id);
    switch (kind) {
        case GemmKind::FwdGateUp:
        case GemmKind::FwdGateUpSaveOnly:
            ok = tmap_bf16(&ta, b + L.xperm, H, R, 128) && tmap_bf16(&tb, W, H, E * 2 * I, 128);
            a.n_tiles = (int)(I / 128); a.k_blocks = (int)(H / kBK); a.b_rows_e = (int)(2 * I); a.b_up = (int)I;
            a.out0 = b + L.hid; a.out1 = b + L.gu;
            if (!ok) break;
            err = kind == GemmKind::FwdGateUp ? run<256, false, false, true, false, EPI_SWIGLU>(c, ta, tb, a)
                                              : run<256, false, false, true, false, EPI_GU_ONLY>(c, ta, tb, a);
            break;
        case GemmKind::FwdDown:
            ok = tmap_bf16(&ta, b + L.hid, I, R, 128) && tmap_bf16(&tb, W, I, E * H, 256);
            a.n_tiles = (int)(H / 256); a.k_blocks = (int)(I / kBK); a.b_rows_e = (int)H;
            a.out0 = b + L.ypart; a.ld0 = (int)H;
            if (!ok) break;
            err = run<256, false, false, false, false, EPI_WEIGHTED>(c, ta, tb, a);
            break;
        case GemmKind::BwdDown: {
            const int bn = bwd_down_bn(I);
            ok = tmap_bf16(&ta, b + L.dyperm, H, R, 128) && tmap_bf16(&tb, W, I, E * H, 64);
            a.n_tiles = (int)(I / bn); a.k_blocks = (int)(H / kBK); a.b_rows_e = (int)H;
            a.out0 = b + L.dg; a.out1 = b + L.hw; a.dtw = reinterpret_cast<float*>(b + L.dtw);
            if (!ok) break;
            err = bn == 256 ? run<256, false, true, false, false, EPI_SWIGLU_BWD>(c, ta, tb, a)
                            : run<128, false, true, false, false, EPI_SWIGLU_BWD>(c, ta, tb, a);
            break;
        }
        case GemmKind::BwdGateUp:
            ok = tmap_bf16(&ta, b + L.dg, 2 * I, R, 128) && tmap_bf16(&tb, W, H, E * 2 * I, 64);
            a.n_tiles = (int)(H / 256); a.k_blocks = (int)(2 * I / kBK); a.b_rows_e = (int)(2 * I);
            a.out0 = b + L.ypart; a.ld0 = (int)H;
            if (!ok) break;
            err = run<256, false, true, false, false, EPI_PLAIN>(c, ta, tb, a);
            break;
        case GemmKind::WgradDown: {
            const int bn = bwd_down_bn(I);
            ok = tmap_bf16(&ta, b + L.dyperm, H, R, 64) && tmap_bf16(&tb, b + L.hw, I, R, 64);
            a.m_tiles = (int)(H / 128); a.n_tiles = (int)(I / bn);
            a.out0 = out; a.ld0 = (int)I; a.out_e_stride = H * I;
            if (!ok) break;
            err = bn == 256 ? run<256, true, true, false, true, EPI_WGRAD>(c, ta, tb, a)
                            : run<128, true, true, false, true, EPI_WGRAD>(c, ta, tb, a);
            break;
        }
        case GemmKind::WgradGateUp:
            ok = tmap_bf16(&ta, b + L.dg, 2 * I, R, 64) && tmap_bf16(&tb, b + L.xperm, H, R, 64);
            a.m_tiles = (int)(2 * I / 128); a.n_tiles = (int)(H / 256);
            a.out0 = out; a.ld0 = (int)H; a.out_e_stride = 2 * I * H;
            if (!ok) break;
            err = run<256, true, true, false, true, EPI_WGRAD>(c, ta, tb, a);
            break;
    }
    trace_end(c.st, trace_id);
    if (!ok) return cudaErrorInvalidValue;
    return err;
}

}  // namespace moe
