// gemm.cu - persistent grouped GEMMs of the MoE layer on the 5th-generation tensor cores.
//
// The pages' fused layer runs the two expert linear layers with SwiGLU between them and combines
// by routing weight (MarkTechPost, "Prime Intellect Releases Prime Mega MoE", section "How does
// the fused kernel work?"); a grouped GEMM packs many differently sized per-expert products into
// one launch indexed by group offsets (kongchang.com, "Prime Intellect推出Prime Mega MoE", section
// "为什么 MoE 训练特别需要融合内核").  The backward adds the activation- and weight-gradient
// products (ic.work analysis, section "从 3.11 倍到 1.32 倍的性能漏斗").  Operands are BF16, or
// MXFP8 (E4M3 with one E8M0 scale per 32 elements along K) on the block-scaled MMA.
//
// One kernel template serves all eight products in both precisions.  Each CTA is persistent (one
// per SM) and walks a static list of 128 x BN output tiles; its warps are specialised:
//   warp 0      TMA producer: loads 128-byte-deep K slices of A and B (64 bf16 or 128 E4M3
//               elements) into a smem ring of 4 or 6 stages (128-byte swizzle), plus for MXFP8
//               the 512-byte scale-factor atoms of the slice, and counts the bytes on an mbarrier;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN; K=16 bf16 or K=32 E4M3,
//               for MXFP8 after tcgen05.cp of the scale atoms into TMEM) into a TMEM accumulator
//               and releases each smem stage with tcgen05.commit;
//   warps 2..   epilogue (4 or 8 warps): tcgen05.ld the finished accumulator (one TMEM lane = one
//               row per thread; warp w reads lane quarter w % 4, and with 8 warps the two warps of
//               a quarter take alternate 32-column chunks), apply the fused epilogue, stage row
//               blocks in shared memory for TMA stores, and release the accumulator.
// Accumulators: BF16 and the 128-wide MXFP8 tiles keep two, so the epilogue of tile i overlaps
// the MMAs of tile i+1; MXFP8 128 x 256 tiles keep one (two would leave no TMEM for the scales),
// which eight epilogue warps drain to registers before they compute.  The BF16 products with
// N = 256, except the forward gate/up and the reducing forward down, run on CTA pairs
// (cta_group::2, M = 256 per pair, each CTA loading its A rows and half of B).  The SwiGLU backward reads the saved g, u of its tile from
// shared memory (MXFP8: TMA-loaded one tile ahead) or from registers prefetched a chunk ahead (BF16).
// Routed rows are laid out per expert padded to multiples of 128, so a row tile belongs to one
// expert and a weight-gradient K slice never crosses into the next expert's rows.
// Tile lists: "grouped-M" products (forward and data gradients) enumerate
// (m-tile, n-tile) with n fastest, so CTAs working at the same time share the A tile in L2;
// weight gradients enumerate (expert, m-tile, n-tile), experts in decreasing token count.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kStages = 4;
constexpr int kRowBytes = 128;                       // bytes of K per smem row (128-byte swizzle)
constexpr int kATileBytes = kBM * kRowBytes;         // 16 KB
constexpr int kSfAtom = 512;                         // 128 MN x 4 K-blocks of E8M0 scales

enum Epi : int { EPI_SWIGLU = 0, EPI_GU_ONLY, EPI_WEIGHTED, EPI_SWIGLU_BWD, EPI_PLAIN, EPI_WGRAD, EPI_WEIGHTED_RED };

// Epilogue warps: the SwiGLU backward reads [g|u] and writes three outputs per element and needs
// two warps per TMEM lane quarter to keep up with the MMAs; the other epilogues use one.
// MXFP8 tiles 128 x 256 keep a single accumulator (two would leave no TMEM for the scales); their
// epilogue first drains the accumulator into registers, which needs two warps per lane quarter.
template <int EPI, bool SINGLE>
constexpr int epi_warps() { return (EPI == EPI_SWIGLU_BWD || SINGLE) ? 8 : 4; }
template <int EPI, bool SINGLE>
constexpr int gemm_threads() { return 64 + 32 * epi_warps<EPI, SINGLE>(); }
// Epilogues of four warps that write bf16 / fp32 row blocks from the accumulator: they stage
// them in shared memory and store them by TMA (the drained MXFP8 128 x 256 tiles keep direct stores)
template <int EPI, bool MX, int BN>
constexpr bool tma_out() {
    return (!(MX && BN == 256) && epi_warps<EPI, MX && BN == 256>() == 4 &&
            (EPI == EPI_WEIGHTED || EPI == EPI_PLAIN || EPI == EPI_SWIGLU || EPI == EPI_GU_ONLY || EPI == EPI_WGRAD ||
             EPI == EPI_WEIGHTED_RED)) ||
           (!MX && EPI == EPI_SWIGLU_BWD) ||
           (MX && BN == 256 &&
            (EPI == EPI_WEIGHTED || EPI == EPI_PLAIN || EPI == EPI_SWIGLU || EPI == EPI_GU_ONLY || EPI == EPI_WGRAD));
}
// bytes of one warp's staging box: 32 rows x 128 bytes, or 32 x 64 (64-byte swizzle) for the
// eight-warp epilogues (the SwiGLU backward, the drained MXFP8 128 x 256 tiles), whose 4 KB
// boxes would not fit beside the ring
template <int EPI, bool SINGLE>
constexpr int out_box_bytes() { return (EPI == EPI_SWIGLU_BWD || SINGLE) ? 2048 : 4096; }

// ---- staged TMA stores: one 32-row x 128-byte box per epilogue warp, row = lane ----------------
// waits until the warp's previous box has been read out by its TMA store
__device__ __forceinline__ void box_acquire(int lane) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
}
// 16-byte chunk `chunk` of the lane's row, 128-byte swizzle (the box is 1024-byte aligned)
__device__ __forceinline__ void box_put(uint32_t sbox, int lane, int chunk, uint4 v) {
    st_shared_v4(sbox + lane * 128 + ((chunk ^ (lane & 7)) << 4), v);
}
// 32 values as bf16 into chunks [4 h, 4 h + 4) (columns [32 h, 32 h + 32) of a 64-column box)
__device__ __forceinline__ void box_put_bf16x32(uint32_t sbox, int lane, int h, const float* v, float scale) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const float* f = v + 8 * cc;
        box_put(sbox, lane, 4 * h + cc,
                make_uint4(pack_bf16x2(scale * f[0], scale * f[1]), pack_bf16x2(scale * f[2], scale * f[3]),
                           pack_bf16x2(scale * f[4], scale * f[5]), pack_bf16x2(scale * f[6], scale * f[7])));
    }
}
// 32 fp32 values: the whole 128-byte row of a 32-column box
__device__ __forceinline__ void box_put_f32x32(uint32_t sbox, int lane, const float* v) {
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
        box_put(sbox, lane, cc,
                make_uint4(__float_as_uint(v[4 * cc]), __float_as_uint(v[4 * cc + 1]), __float_as_uint(v[4 * cc + 2]),
                           __float_as_uint(v[4 * cc + 3])));
}
// 32 values (times scale) as bf16 into a 32-row x 64-byte box (64-byte swizzle; the box is
// 512-byte aligned)
__device__ __forceinline__ void box64_put_bf16x32(uint32_t sbox, int lane, const float* v, float scale = 1.f) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const float* f = v + 8 * cc;
        st_shared_v4(sbox + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4),
                     make_uint4(pack_bf16x2(scale * f[0], scale * f[1]), pack_bf16x2(scale * f[2], scale * f[3]),
                                pack_bf16x2(scale * f[4], scale * f[5]), pack_bf16x2(scale * f[6], scale * f[7])));
    }
}
// 16 fp32 values into the lane's row of a 32-row x 64-byte box (64-byte swizzle)
__device__ __forceinline__ void box64_put_f32x16(uint32_t sbox, int lane, const float* v) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
        st_shared_v4(sbox + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4),
                     make_uint4(__float_as_uint(v[4 * cc]), __float_as_uint(v[4 * cc + 1]), __float_as_uint(v[4 * cc + 2]),
                                __float_as_uint(v[4 * cc + 3])));
}
// 32 bf16 values already packed in pairs (p[0..15]) into a 32-row x 64-byte box (64-byte swizzle)
__device__ __forceinline__ void box64_put_packed(uint32_t sbox, int lane, const uint32_t* p) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
        st_shared_v4(sbox + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4),
                     make_uint4(p[4 * cc], p[4 * cc + 1], p[4 * cc + 2], p[4 * cc + 3]));
}
// hands the staged box to the async proxy and stores it at {c0 (column), c1 (row)}
__device__ __forceinline__ void box_store(const CUtensorMap* m, uint8_t* box, int lane, int c0, int c1) {
    fence_proxy_async_cta();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(m, box, c0, c1);
        bulk_commit();
    }
}
// stages 32 values in the warp's 2 KB box and stores them at {c0, c1}
__device__ __forceinline__ void box64_emit(const CUtensorMap* m, uint8_t* box, int lane, const float* v, float scale,
                                           int c0, int c1) {
    box_acquire(lane);
    box64_put_bf16x32(smem_u32(box), lane, v, scale);
    box_store(m, box, lane, c0, c1);
}

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
    // MXFP8 scale factors (atoms of 512 bytes, see quant.cu): atom (mn_tile, k_tile) of an
    // operand is at sf + (mn_tile * kt + k_tile) * 512
    const uint8_t* sfA;
    const uint8_t* sfB;
    int sfA_kt, sfB_kt;
    // MXFP8 epilogue outputs (E4M3 values + scale atoms) written in place of bf16 ones:
    // forward gate/up: q0 = h blocked along I; SwiGLU backward: q0 = [dg|du] blocked along 2I,
    // q1 = [dg|du] blocked along the rows, q2 = w h blocked along the rows
    uint8_t* q0;
    uint8_t* q0_sf;
    uint8_t* q1;
    uint8_t* q1_sf;
    uint8_t* q2;
    uint8_t* q2_sf;
    int r_atoms;               // padded row capacity / 128 (K atoms of the row-blocked scales)
    uint32_t b_fmt;            // B-format bits OR-ed into the block-scaled instruction descriptor
                               // (kFmtE2M1B: MXFP4 weights, unpacked to 16-byte rows by the TMA)
    float* yacc;               // fused combine: fp32 [T, H] accumulator the epilogue reduces into
    int k;                     // routed slots per token (slot / k = token)
    int w_in_a;                // BF16 forward down: the routing weight is already in A (w h)
    long long wait_limit;      // cycles after which a pipeline wait gives up (MOE_DEV_TIMEOUT)
    int withhold_loads;        // test of the bounded waits: the producer issues no operand loads
};

struct Tile {
    int e, m0, n0, nt, kb, row0;
    bool valid;   // false: the duplicate tile of an expert's odd last m-tile in a CTA pair (no store)
};

__device__ __forceinline__ int find_expert(const int* s_mtile, int E, int gm) {
    int lo = 0, hi = E - 1;  // largest e with s_mtile[e] <= gm
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_mtile[mid] <= gm) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// kElems: K elements per pipeline stage (64 bf16, 128 E4M3); a 128-row group holds
// 128 / kElems stages of a weight-gradient contraction.
// PAIR: the unit L is shared by the two CTAs of a cluster, which take two m-tiles of the same
// expert (rank 0 the even, rank 1 the odd one) and the same n-tile, so they need the same B tile.
// Grouped-M units enumerate the pairs of each expert (s_pair: prefix of ceil(m-tiles / 2)); an
// expert with an odd m-tile count gives rank 1 a duplicate of rank 0's last tile, not stored.
template <int BN, bool WGRAD, bool SPLIT, int kElems, bool PAIR>
__device__ __forceinline__ Tile decode_tile(int L, const GemmArgs& a, const int* s_mtile, const int* s_pair,
                                            int rank) {
    Tile t;
    t.valid = true;
    if (!WGRAD) {
        int gm;
        if (PAIR) {
            const int P = L / a.n_tiles;
            t.nt = L - P * a.n_tiles;
            t.e = find_expert(s_pair, a.E, P);
            const int mt_e = s_mtile[t.e + 1] - s_mtile[t.e];
            const int lm = 2 * (P - s_pair[t.e]) + rank;
            t.valid = lm < mt_e;
            gm = s_mtile[t.e] + min(lm, mt_e - 1);
        } else {
            gm = L / a.n_tiles;
            t.nt = L - gm * a.n_tiles;
            t.e = find_expert(s_mtile, a.E, gm);
        }
        t.m0 = gm * kBM;
        t.n0 = t.nt * (SPLIT ? BN / 2 : BN);
        t.kb = a.k_blocks;
        t.row0 = 0;
    } else {
        const int mtp = PAIR ? a.m_tiles / 2 : a.m_tiles;
        const int per = mtp * a.n_tiles;
        const int ei = L / per;
        const int rem = L - ei * per;
        const int mq = rem / a.n_tiles;
        const int mt = PAIR ? 2 * mq + rank : mq;
        t.nt = rem - mq * a.n_tiles;
        t.e = a.order[ei];
        t.m0 = mt * kBM;
        t.n0 = t.nt * BN;
        t.row0 = s_mtile[t.e] * kBM;
        t.kb = (s_mtile[t.e + 1] - s_mtile[t.e]) * (kBM / kElems);
    }
    return t;
}

// bounded wait without the abort short-cut, used only while draining after an abort
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kDrainCycles) break;
}

// Epilogue of a 128 x 256 MXFP8 tile from registers: d holds columns [128 h, 128 h + 128) of
// the thread's row.  For the gate/up product these are one [64 gate | 64 up] block of the
// interleaved weight, i.e. g and u of I-columns [n0 + 64 h, n0 + 64 h + 64).  The bf16 and fp32
// row outputs go through the warp's 2 KB staging box (32 rows from brow, 64 bytes a row at a time)
// and leave by TMA store; the E4M3 h of the gate/up product is stored from registers.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_drained(const GemmArgs& a, const Tile& t, long long grow, int h, float* d,
                                                 const CUtensorMap* tmC, const CUtensorMap* tmD, uint8_t* box,
                                                 int lane, int brow) {
    if constexpr (EPI == EPI_SWIGLU || EPI == EPI_GU_ONLY) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float* g = d + 32 * c;
            float* u = d + 64 + 32 * c;
            const int col = t.n0 + 64 * h + 32 * c;
            if (EPI == EPI_GU_ONLY || a.save_gu) {
                box64_emit(tmD, box, lane, g, 1.f, col, brow);
                box64_emit(tmD, box, lane, u, 1.f, a.I + col, brow);
            }
            if constexpr (EPI == EPI_SWIGLU) {
                float hv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) hv[j] = g[j] * sigmoidf_fast(g[j]) * u[j];
                quant_row32(hv, a.q0 + grow * (long long)a.I + col, a.q0_sf + sf_index(grow, col / 32, a.I / 128));
            }
        }
    } else if constexpr (EPI == EPI_WEIGHTED || EPI == EPI_PLAIN) {
        float w = 1.f;
        if constexpr (EPI == EPI_WEIGHTED) {
            const int slot = a.row_slot[grow];
            w = slot >= 0 ? a.topk_w[slot] : 0.f;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) box64_emit(tmC, box, lane, d + 32 * c, w, t.n0 + 128 * h + 32 * c, brow);
    } else if constexpr (EPI == EPI_WGRAD) {
        if (t.kb == 0) {   // an expert without rows: a zero gradient
#pragma unroll
            for (int j = 0; j < 128; ++j) d[j] = 0.f;
        }
        // rows of this expert's block of the weight gradient [E * M, N], whole 64-byte row
        // segments through the warp's box: 16 fp32 or 32 bf16 columns a store
        const int orow = t.e * a.m_tiles * kBM + brow;
        const uint32_t sbox = smem_u32(box);
        if (a.out_f32) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                box_acquire(lane);
                box64_put_f32x16(sbox, lane, d + 16 * c);
                box_store(tmC, box, lane, t.n0 + 128 * h + 16 * c, orow);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) box64_emit(tmC, box, lane, d + 32 * c, 1.f, t.n0 + 128 * h + 32 * c, orow);
        }
    }
}

// Stages of the smem ring: a CTA pair driving one MMA (TWO) holds only half of each B tile per
// CTA, which leaves room for six.
// pipeline stages: six for the two-SM BF16 tiles and the 128 x 128 MXFP8 weight-gradient tiles
// (33 KB a stage), four otherwise (the MXFP8 SwiGLU backward, bound by its epilogue, measured
// 578 µs with four against 592-596 µs with six)
template <bool TWO, bool MX, int BN, bool WGRAD>
constexpr int ring_stages() { return (TWO || (MX && BN == 128 && WGRAD)) ? 6 : kStages; }

// TWO: clusters of two CTAs on two m-tiles of one expert and the same n-tile; the leader CTA
// issues cta_group::2 MMAs (M = 256) over both CTAs' shared memory and tensor memory, each CTA
// holding half of every B tile, which it loads itself (no load is multicast).
template <int BN, bool A_MN, bool B_MN, bool SPLIT, bool WGRAD, int EPI, bool MX, bool TWO>
__global__ void __launch_bounds__(gemm_threads<EPI, MX && BN == 256>(), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                        const GemmArgs a) {
    grid_dep_wait();
    static_assert(!TWO || !MX, "two-SM MMAs run in CTA pairs, BF16 only");
    constexpr bool PAIR = TWO;                           // clusters of two CTAs exist only for them
    constexpr int kStages = ring_stages<TWO, MX, BN, WGRAD>();
    constexpr int kElems = MX ? 128 : 64;                // K elements per stage
    constexpr int kMmaK = MX ? 32 : 16;                  // K elements per MMA
    constexpr int kMnChunk = MX ? 128 : 64;              // MN elements per 128-byte row (MN-major)
    constexpr int kBTileBytes = (TWO ? BN / 2 : BN) * kRowBytes;   // TWO: this CTA's half of B
    constexpr int kSfBAtoms = BN / 128;
    constexpr int kSfBytes = MX ? kSfAtom * (1 + kSfBAtoms) : 0;
    constexpr int kStageBytes = kATileBytes + kBTileBytes + kSfBytes;
    constexpr uint32_t kIdesc = idesc_bf16(TWO ? 2 * kBM : kBM, BN, A_MN, B_MN);
    constexpr uint32_t kSfCols = 4 * (1 + kSfBAtoms);    // TMEM columns of one stage's scales
    constexpr bool kSingle = MX && BN == 256;            // one accumulator, drained to registers
    constexpr int kAccStages = kSingle ? 1 : 2;
    constexpr uint32_t kTmemCols = MX ? 512 : 2 * BN;
    constexpr int kEpiWarps = epi_warps<EPI, kSingle>();
    constexpr int kHalves = kEpiWarps / 4;
    // MN-major operands: the next kMnChunk MN values start one chunk (kElems rows of 128 B) on
    constexpr uint32_t kMnLbo = kElems * kRowBytes;
    constexpr uint32_t kMnStep = kMmaK * kRowBytes;      // MN-major: bytes per MMA K step
    constexpr uint32_t kKStep = kMmaK * (MX ? 1 : 2);    // K-major: bytes per MMA K step
    static_assert(!MX || BN == 128 || BN == 256, "MXFP8 tiles are 128 x 128 or 128 x 256");
    static_assert(!kSingle || EPI != EPI_SWIGLU_BWD, "the SwiGLU backward keeps 128-wide MXFP8 tiles");
    // Row outputs of four-warp epilogues: each warp stages 32 rows x 128 bytes (64 bf16 or 32 fp32
    // columns, 128-byte swizzle) in shared memory and writes them with a TMA store (tmC; tmD for the
    // saved [g|u]), so that L2 receives whole lines rather than 16-byte halves of sectors
    constexpr bool kTmaOut = tma_out<EPI, MX, BN>();
    constexpr int kOutBytes = kTmaOut ? kEpiWarps * out_box_bytes<EPI, kSingle>() : 0;
    static_assert(kTmaOut || EPI == EPI_SWIGLU_BWD, "epilogues other than the MXFP8 SwiGLU backward's stage their "
                                                    "rows for TMA stores");
    // MXFP8 SwiGLU backward: the tile's saved g and u reach shared memory by TMA (tmD, boxes of
    // 128 rows x 64 columns) in two halves of 64 columns each, issued one tile ahead by the first
    // epilogue warp, so that the epilogue does not wait on its own global loads
    constexpr bool kGuSmem = MX && EPI == EPI_SWIGLU_BWD;
    constexpr int kGuHalfBytes = 2 * kBM * kRowBytes;   // the g box and the u box of one half
    constexpr int kGuBytes = kGuSmem ? 2 * kGuHalfBytes : 0;
    static_assert(!kGuSmem || (BN == 128 && !PAIR && kEpiWarps == 8), "two passes of 64 columns, one CTA");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kATileBytes;
    uint8_t* sSF = sB + kStages * kBTileBytes;           // MXFP8: per stage A atom then B atoms
    uint8_t* sOut = sSF + kStages * kSfBytes;           // TMA-stored outputs: a 4 KB box per epilogue warp
    uint8_t* sGu = sOut + kOutBytes;                    // MXFP8 SwiGLU backward: saved g, u of a tile
    uint64_t* bars = reinterpret_cast<uint64_t*>(sGu + kGuBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* tfull = bars + 2 * kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* gu_full = drain + 1;    // [2] a half of the saved g, u has landed
    uint64_t* gu_free = drain + 3;    // [2] every epilogue warp has read that half
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    int* s_mtile = reinterpret_cast<int*>(tslot + 4);
    int* s_pair = s_mtile + (a.E + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = PAIR ? (int)cluster_ctarank() : 0;
    const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // cluster = 2 consecutive CTAs
    const int unit_stride = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    constexpr uint16_t kPeers = 0x3;
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_mtile[i] = a.mtile[i];
    __syncthreads();
    if (threadIdx.x == 0) {
        if (PAIR && !WGRAD) {
            s_pair[0] = 0;
            for (int e = 0; e < a.E; ++e) s_pair[e + 1] = s_pair[e] + (s_mtile[e + 1] - s_mtile[e] + 1) / 2;
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, (TWO ? 2 : 1) * kEpiWarps);   // one arrival per epilogue warp (TWO: both CTAs')
        }
        mbar_init(drain, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(gu_full + b, 1);
            mbar_init(gu_free + b, kEpiWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if constexpr (TWO) tmem_alloc_pair(tslot, kTmemCols);
        else tmem_alloc(tslot, kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // the peer's barriers exist before any copy or commit reaches them
    tc_fence_after();
    const uint32_t tmem_base = *tslot;
    const int num_tiles = WGRAD ? a.E * (PAIR ? a.m_tiles / 2 : a.m_tiles) * a.n_tiles
                                : (PAIR ? s_pair[a.E] : s_mtile[a.E]) * a.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            // bytes one stage's copies complete: a packed-E2M1 B tile counts the bytes it reads
            // (half a byte a value) although it lands in shared memory as a byte a value
            const uint32_t stage_tx = kStageBytes - (a.b_fmt ? kBTileBytes / 2 : 0);
            // (with withhold_loads nothing is issued, so the MMA warp's first wait runs out while no
            // copy is in flight)
            for (int L = unit0; L < num_tiles && ok && !a.withhold_loads; L += unit_stride) {
                const Tile t = decode_tile<BN, WGRAD, SPLIT, kElems, PAIR>(L, a, s_mtile, s_pair, rank);
                // first B row of the tile (K-major B); MXFP8 gate/up weights are stored with
                // 128-row blocks of [64 gate | 64 up] rows, so the split tile is one block
                const int b_row0 = t.e * a.b_rows_e + ((SPLIT && MX) ? t.nt * BN : t.n0);
                for (int kb = 0; kb < t.kb; ++kb) {
                    if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag, a.status, a.wait_limit)) { ok = false; break; }
                    uint8_t* dA = sA + stage * kATileBytes;
                    uint8_t* dB = sB + stage * kBTileBytes;
                    const int k0 = kb * kElems;
                    if (TWO) {
                        // both CTAs' copies land on the leader's barrier, which expects both
                        const uint32_t lbar = cluster_addr(full + stage, 0);
                        if (rank == 0) mbar_arrive_expect_tx(full + stage, 2 * kStageBytes);
                        if (!A_MN) {
                            tma_load_2d_pair(dA, &tmA, lbar, k0, t.m0);
                        } else {
#pragma unroll
                            for (int c = 0; c < kBM / kMnChunk; ++c)
                                tma_load_2d_pair(dA + c * kMnLbo, &tmA, lbar, t.m0 + kMnChunk * c, t.row0 + k0);
                        }
                        if (!B_MN) {
                            const int brow = SPLIT ? t.e * a.b_rows_e + rank * a.b_up + t.n0 : b_row0 + rank * (BN / 2);
                            tma_load_2d_pair(dB, &tmB, lbar, k0, brow);
                        } else {
                            const int krow = WGRAD ? t.row0 + k0 : t.e * a.b_rows_e + k0;
                            constexpr int nch = BN / kMnChunk;
#pragma unroll
                            for (int c = 0; c < nch / 2; ++c)
                                tma_load_2d_pair(dB + c * kMnLbo, &tmB, lbar, t.n0 + kMnChunk * (rank * nch / 2 + c), krow);
                        }
                        ++issued;
                        if (++stage == kStages) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    mbar_arrive_expect_tx(full + stage, stage_tx);
                    if (!A_MN) {
                        tma_load_2d(dA, &tmA, full + stage, k0, t.m0);
                    } else {
#pragma unroll
                        for (int c = 0; c < kBM / kMnChunk; ++c)
                            tma_load_2d(dA + c * kMnLbo, &tmA, full + stage, t.m0 + kMnChunk * c, t.row0 + k0);
                    }
                    if (!B_MN) {
                        if (SPLIT && !MX) {
                            tma_load_2d(dB, &tmB, full + stage, k0, t.e * a.b_rows_e + t.n0);
                            tma_load_2d(dB + (BN / 2) * kRowBytes, &tmB, full + stage, k0,
                                        t.e * a.b_rows_e + a.b_up + t.n0);
                        } else {
                            tma_load_2d(dB, &tmB, full + stage, k0, b_row0);
                        }
                    } else {
                        const int krow = WGRAD ? t.row0 + k0 : t.e * a.b_rows_e + k0;
#pragma unroll
                        for (int c = 0; c < BN / kMnChunk; ++c)
                            tma_load_2d(dB + c * kMnLbo, &tmB, full + stage, t.n0 + kMnChunk * c, krow);
                    }
                    if constexpr (MX) {
                        // scale atoms of this K slice: A (m-tile) then B (n-tiles)
                        uint8_t* dS = sSF + stage * kSfBytes;
                        const int ka = (WGRAD ? t.row0 / 128 : 0) + kb;
                        bulk_load(dS, a.sfA + ((long long)(t.m0 / 128) * a.sfA_kt + ka) * kSfAtom, kSfAtom,
                                  full + stage);
#pragma unroll
                        for (int c = 0; c < kSfBAtoms; ++c) {
                            long long mn_tile, kt;
                            if (!B_MN) {
                                mn_tile = b_row0 / 128 + c;
                                kt = kb;
                            } else if (!WGRAD) {
                                mn_tile = t.n0 / 128 + c;
                                kt = (long long)t.e * a.b_rows_e / 128 + kb;
                            } else {
                                mn_tile = t.n0 / 128 + c;
                                kt = t.row0 / 128 + kb;
                            }
                            bulk_load(dS + kSfAtom * (1 + c), a.sfB + (mn_tile * a.sfB_kt + kt) * kSfAtom, kSfAtom,
                                      full + stage);
                        }
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
        if (lane == 0 && TWO && rank == 1) {
            // peer of a two-SM pair: its copies complete on the leader's barriers and the leader
            // issues the MMAs; before exiting, wait for the leader's releases of its last stages
            long long consumed = 0;
            for (int L = unit0; L < num_tiles; L += unit_stride)
                consumed += decode_tile<BN, WGRAD, SPLIT, kElems, PAIR>(L, a, s_mtile, s_pair, rank).kb;
            for (int s = 0; s < kStages; ++s) {
                if (consumed > s) {
                    const long long n = (consumed - s + kStages - 1) / kStages;
                    drain_wait(empty + s, (uint32_t)((n - 1) & 1));
                }
            }
        } else if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB), sf_base = smem_u32(sSF);
            long long consumed = 0;
            for (int L = unit0; L < num_tiles && ok; L += unit_stride) {
                const Tile t = decode_tile<BN, WGRAD, SPLIT, kElems, PAIR>(L, a, s_mtile, s_pair, rank);
                if (!(TWO ? mbar_wait_cluster(tempty + acc, acc_phase ^ 1u, abort_flag, a.status, a.wait_limit)
                          : mbar_wait(tempty + acc, acc_phase ^ 1u, abort_flag, a.status, a.wait_limit))) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < t.kb; ++kb) {
                    if (!mbar_wait(full + stage, phase, abort_flag, a.status, a.wait_limit)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = a_base + stage * kATileBytes, sb = b_base + stage * kBTileBytes;
                    if constexpr (MX) {
                        const uint32_t sf_cols = tmem_base + kAccStages * BN + stage * kSfCols;
                        const uint32_t ss = sf_base + stage * kSfBytes;
#pragma unroll
                        for (int c = 0; c <= kSfBAtoms; ++c)
                            tmem_cp_sf_atom(sf_cols + 4 * c, sdesc_plain(ss + kSfAtom * c, 128));
#pragma unroll
                        for (int ks = 0; ks < kElems / kMmaK; ++ks) {
                            const uint64_t ad = A_MN ? sdesc_sw128(sa + ks * kMnStep, kMnLbo, 1024)
                                                     : sdesc_sw128(sa + ks * kKStep, 16, 1024);
                            const uint64_t bd = B_MN ? sdesc_sw128(sb + ks * kMnStep, kMnLbo, 1024)
                                                     : sdesc_sw128(sb + ks * kKStep, 16, 1024);
                            mma_mxf8(d_tmem, ad, bd, idesc_mxf8(kBM, BN, A_MN, B_MN, ks, ks) | a.b_fmt, sf_cols,
                                     sf_cols + 4, (kb | ks) != 0);
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < kElems / kMmaK; ++ks) {
                            const uint64_t ad = A_MN ? sdesc_sw128(sa + ks * kMnStep, kMnLbo, 1024)
                                                     : sdesc_sw128(sa + ks * kKStep, 16, 1024);
                            const uint64_t bd = B_MN ? sdesc_sw128(sb + ks * kMnStep, kMnLbo, 1024)
                                                     : sdesc_sw128(sb + ks * kKStep, 16, 1024);
                            if constexpr (TWO) mma_bf16_pair(d_tmem, ad, bd, kIdesc, (kb | ks) != 0);
                            else mma_bf16(d_tmem, ad, bd, kIdesc, (kb | ks) != 0);
                        }
                    }
                    if (TWO)
                        mma_commit_pair_mc(empty + stage, kPeers);
                    else
                        mma_commit(empty + stage);
                    ++consumed;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (TWO) {
                    if (t.kb > 0) {
                        mma_commit_pair_mc(tfull + acc, kPeers);
                    } else {
                        mbar_arrive(tfull + acc);
                        mbar_arrive_cluster(tfull + acc, 1);
                    }
                } else if (t.kb > 0) {
                    mma_commit(tfull + acc);
                } else {
                    mbar_arrive(tfull + acc);
                }
                if (kAccStages == 2) {
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                } else {
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                if constexpr (TWO) mma_commit_pair_mc(drain, 0x1);
                else mma_commit(drain);
                drain_wait(drain, 0);
            } else if (PAIR) {
                // both CTAs' releases of the last stages have landed here before the CTA may exit
                for (int s = 0; s < kStages; ++s) {
                    if (consumed > s) {
                        const long long n = (consumed - s + kStages - 1) / kStages;
                        drain_wait(empty + s, (uint32_t)((n - 1) & 1));
                    }
                }
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
        // saved g, u of the MXFP8 SwiGLU backward: half p of tile L (rows m0.., columns n0 + 64 p..)
        // into its shared-memory half, issued by the first epilogue warp's lane 0
        const bool gu_issuer = kGuSmem && warp == 2 && lane == 0;
        uint32_t gu_phase = 0;
        long long gu_issued[2] = {0, 0};
        auto gu_load = [&](int Ln, int p) {
            const int m0 = (Ln / a.n_tiles) * kBM, n0 = (Ln % a.n_tiles) * BN + 64 * p;
            uint8_t* dst = sGu + p * kGuHalfBytes;
            mbar_arrive_expect_tx(gu_full + p, kGuHalfBytes);
            tma_load_2d(dst, &tmD, gu_full + p, n0, m0);
            tma_load_2d(dst + kBM * kRowBytes, &tmD, gu_full + p, a.I + n0, m0);
            ++gu_issued[p];
        };
        if (gu_issuer && unit0 < num_tiles) {
            gu_load(unit0, 0);
            gu_load(unit0, 1);
        }
        for (int L = unit0; L < num_tiles; L += unit_stride) {
            const Tile t = decode_tile<BN, WGRAD, SPLIT, kElems, PAIR>(L, a, s_mtile, s_pair, rank);
            // MXFP8 SwiGLU backward: the row's routing weight is requested before the accumulator wait
            int w_slot = -1;
            if constexpr (kGuSmem) w_slot = a.row_slot[(long long)t.m0 + r];
            // BF16 SwiGLU backward: the thread's first chunk of saved g, u (32 columns each, packed
            // bf16) is requested before the accumulator wait, so that its latency overlaps the wait
            uint4 gnext[4], unext[4];
            if constexpr (EPI == EPI_SWIGLU_BWD && !MX) {
                const __nv_bfloat16* gurow = a.gu + ((long long)t.m0 + quarter * 32 + lane) * (2LL * a.I);
                const int col = t.n0 + 32 * half;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    gnext[q] = __ldg(reinterpret_cast<const uint4*>(gurow + col) + q);
                    unext[q] = __ldg(reinterpret_cast<const uint4*>(gurow + a.I + col) + q);
                }
            }
            if (!mbar_wait(tfull + acc, acc_phase, abort_flag, a.status, a.wait_limit)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + lane_addr + (uint32_t)(acc * BN);
            const long long grow = (long long)t.m0 + r;
            float v[32];
            if constexpr (kSingle) {
                // drain this thread's 128 columns [128 * half, 128 * half + 128), release the
                // accumulator to the next tile's MMAs, then compute and store from registers
                float d[128];
                const uint32_t tcol = tacc + 128 * half;
                tmem_ld32(tcol, d);
                tmem_ld32(tcol + 32, d + 32);
                tmem_ld32(tcol + 64, d + 64);
                tmem_ld32(tcol + 96, d + 96);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty + acc);
                if (t.valid)
                    epilogue_drained<BN, EPI>(a, t, grow, half, d, &tmC, &tmD,
                                                       sOut + (warp - 2) * out_box_bytes<EPI, kSingle>(), lane,
                                                       t.m0 + 32 * quarter);
                acc_phase ^= 1u;
                continue;
            }
            if (!t.valid) {
                // duplicate tile of a CTA pair: nothing to store
            } else if constexpr (kTmaOut && EPI != EPI_SWIGLU_BWD) {
                uint8_t* box = sOut + (warp - 2) * 4096;
                const uint32_t sbox = smem_u32(box);
                const int brow = t.m0 + 32 * quarter;   // first row of the warp's boxes
                if constexpr (EPI == EPI_SWIGLU || EPI == EPI_GU_ONLY) {
                    // columns [0, BN/2) = gate, [BN/2, BN) = up, for I-columns [n0, n0 + BN/2); per
                    // 64 I-columns: the w h box (the row's routing weight applied here, so that the
                    // down product needs none and the backward reuses w h), then (saving) the g and
                    // u boxes, re-read from TMEM
                    float w = 0.f;
                    if (EPI == EPI_SWIGLU) {
                        const int slot = a.row_slot[grow];
                        w = slot >= 0 ? a.topk_w[slot] : 0.f;
                    }
#pragma unroll 1
                    for (int b = 0; b < BN / 128; ++b) {
                        if (EPI == EPI_SWIGLU) {
                            box_acquire(lane);
#pragma unroll 1
                            for (int h = 0; h < 2; ++h) {
                                float u[32];
                                tmem_ld32(tacc + 64 * b + 32 * h, v);
                                tmem_ld32(tacc + BN / 2 + 64 * b + 32 * h, u);
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] = v[j] * sigmoidf_fast(v[j]) * u[j];
                                box_put_bf16x32(sbox, lane, h, v, w);
                            }
                            box_store(&tmC, box, lane, t.n0 + 64 * b, brow);
                        }
                        if (EPI == EPI_GU_ONLY || a.save_gu) {
#pragma unroll 1
                            for (int p = 0; p < 2; ++p) {   // g, then u
                                box_acquire(lane);
#pragma unroll 1
                                for (int h = 0; h < 2; ++h) {
                                    tmem_ld32(tacc + (BN / 2) * p + 64 * b + 32 * h, v);
                                    box_put_bf16x32(sbox, lane, h, v, 1.f);
                                }
                                box_store(&tmD, box, lane, a.I * p + t.n0 + 64 * b, brow);
                            }
                        }
                    }
                } else if constexpr (EPI == EPI_WGRAD) {
                    // rows of this expert's block of the weight gradient [E * M, N]
                    const int orow = t.e * a.m_tiles * kBM + brow;
                    if (a.out_f32) {
#pragma unroll 1
                        for (int b = 0; b < BN / 32; ++b) {
                            box_acquire(lane);
                            if (t.kb > 0) {
                                tmem_ld32(tacc + 32 * b, v);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] = 0.f;
                            }
                            box_put_f32x32(sbox, lane, v);
                            box_store(&tmC, box, lane, t.n0 + 32 * b, orow);
                        }
                    } else {
#pragma unroll 1
                        for (int b = 0; b < BN / 64; ++b) {
                            box_acquire(lane);
#pragma unroll 1
                            for (int h = 0; h < 2; ++h) {
                                if (t.kb > 0) {
                                    tmem_ld32(tacc + 64 * b + 32 * h, v);
                                } else {
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                                }
                                box_put_bf16x32(sbox, lane, h, v, 1.f);
                            }
                            box_store(&tmC, box, lane, t.n0 + 64 * b, orow);
                        }
                    }
                } else if constexpr (EPI == EPI_WEIGHTED_RED) {
                    // w o of the warp's 32 rows, 32 fp32 columns at a time, staged row-major in the box;
                    // then 8 lanes per row add 16 bytes each into the row's token of the accumulator,
                    // so one vector reduction instruction covers four whole 128-byte row segments
                    const int slot = a.row_slot[grow];
                    const float w = a.w_in_a ? 1.f : (slot >= 0 ? a.topk_w[slot] : 0.f);
                    const int tok = slot >= 0 ? slot / a.k : -1;
#pragma unroll 1
                    for (int b = 0; b < BN / 32; ++b) {
                        tmem_ld32(tacc + 32 * b, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] *= w;
                        __syncwarp();                       // the box's previous chunk is read out
                        box_put_f32x32(sbox, lane, v);
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int rr = 4 * i + (lane >> 3), ch = lane & 7;
                            const int trow = __shfl_sync(0xffffffffu, tok, rr);
                            const uint4 q = ld_shared_v4(sbox + rr * 128 + ((ch ^ (rr & 7)) << 4));
                            if (trow >= 0)
                                red_add_f32x4(a.yacc + (long long)trow * a.ld0 + t.n0 + 32 * b + 4 * ch, q);
                        }
                    }
                } else {   // EPI_WEIGHTED, EPI_PLAIN: one bf16 row block
                    float w = 1.f;
                    if (EPI == EPI_WEIGHTED && !a.w_in_a) {
                        const int slot = a.row_slot[grow];
                        w = slot >= 0 ? a.topk_w[slot] : 0.f;
                    }
#pragma unroll 1
                    for (int b = 0; b < BN / 64; ++b) {
                        box_acquire(lane);
#pragma unroll 1
                        for (int h = 0; h < 2; ++h) {
                            tmem_ld32(tacc + 64 * b + 32 * h, v);
                            box_put_bf16x32(sbox, lane, h, v, w);
                        }
                        box_store(&tmC, box, lane, t.n0 + 64 * b, brow);
                    }
                }
            } else if constexpr (EPI == EPI_SWIGLU_BWD && !MX) {
                // dA -> dg, du per 32-column chunk (w h was saved by the forward); the next chunk's
                // saved g, u are in flight while this one is computed and stored, and outputs are
                // packed to bf16 pairs as they are produced
                const int slot = a.row_slot[grow];
                const float w = slot >= 0 ? a.topk_w[slot] : 0.f;
                const __nv_bfloat16* gurow = a.gu + grow * (2LL * a.I);
                uint8_t* box = sOut + (warp - 2) * 2048;
                const uint32_t sbox = smem_u32(box);
                const int brow = t.m0 + 32 * quarter;
                float dot = 0.f;
#pragma unroll 1
                for (int c = half; c < BN / 32; c += kHalves) {
                    const int col = t.n0 + 32 * c;
                    uint4 graw[4], uraw[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        graw[q] = gnext[q];
                        uraw[q] = unext[q];
                    }
                    if (c + kHalves < BN / 32) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            gnext[q] = __ldg(reinterpret_cast<const uint4*>(gurow + col + 32 * kHalves) + q);
                            unext[q] = __ldg(reinterpret_cast<const uint4*>(gurow + a.I + col + 32 * kHalves) + q);
                        }
                    }
                    tmem_ld32(tacc + 32 * c, v);   // dA
                    uint32_t dgp[16], dup[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t gw[4] = {graw[q].x, graw[q].y, graw[q].z, graw[q].w};
                        const uint32_t uw[4] = {uraw[q].x, uraw[q].y, uraw[q].z, uraw[q].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 gf = unpack_bf16x2(gw[i]), uf = unpack_bf16x2(uw[i]);
                            const float gg[2] = {gf.x, gf.y}, uu[2] = {uf.x, uf.y};
                            float o_dg[2], o_du[2];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const float dA = v[8 * q + 2 * i + e2];
                                const float sg = sigmoidf_fast(gg[e2]);
                                const float sl = gg[e2] * sg;
                                const float h = sl * uu[e2];
                                dot += dA * h;
                                const float dh = w * dA;
                                o_dg[e2] = dh * uu[e2] * (sg + sl * (1.f - sg));
                                o_du[e2] = dh * sl;
                            }
                            dgp[4 * q + i] = pack_bf16x2(o_dg[0], o_dg[1]);
                            dup[4 * q + i] = pack_bf16x2(o_du[0], o_du[1]);
                        }
                    }
                    // dg and du through the warp's 2 KB box, one after the other
                    box_acquire(lane);
                    box64_put_packed(sbox, lane, dgp);
                    box_store(&tmC, box, lane, col, brow);
                    box_acquire(lane);
                    box64_put_packed(sbox, lane, dup);
                    box_store(&tmC, box, lane, a.I + col, brow);
                }
                a.dtw[grow * (2 * a.n_tiles) + 2 * t.nt + half] = dot;
            } else if constexpr (EPI == EPI_SWIGLU_BWD) {
                // MXFP8: dg, du along 2I and along the rows, and w h along the rows, as E4M3 copies
                static_assert(MX, "the BF16 SwiGLU backward has its own epilogue above");
                const float w = w_slot >= 0 ? a.topk_w[w_slot] : 0.f;
                float dot = 0.f;
                bool gu_ok = true;
#pragma unroll 1
                for (int p = 0; p < 2; ++p) {
                    // pass p: chunk c = half + 2 p, 32 columns inside shared-memory half p
                    const int c = half + kHalves * p;
                    float g[32], u[32];
                    const int col = t.n0 + 32 * c;
                    // (the warp leaves together when any lane's bounded wait gave up)
                    if (!__all_sync(0xffffffffu, mbar_wait(gu_full + p, gu_phase, abort_flag, a.status, a.wait_limit))) {
                        gu_ok = false;
                        break;
                    }
                    const uint32_t sg = smem_u32(sGu + p * kGuHalfBytes) + r * kRowBytes;
                    uint4 graw[4], uraw[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t off = (uint32_t)(((4 * half + q) ^ (r & 7)) << 4);   // 128-byte swizzle
                        graw[q] = ld_shared_v4(sg + off);
                        uraw[q] = ld_shared_v4(sg + kBM * kRowBytes + off);
                    }
                    // every lane has its g, u in registers: the warp releases its part of the half
                    __syncwarp();
                    if (lane == 0) mbar_arrive(gu_free + p);
                    bool issued = true;
                    if (gu_issuer && L + unit_stride < num_tiles) {
                        issued = mbar_wait(gu_free + p, gu_phase, abort_flag, a.status, a.wait_limit);
                        if (issued) gu_load(L + unit_stride, p);
                    }
                    if (!__all_sync(0xffffffffu, issued)) {
                        gu_ok = false;
                        break;
                    }
                    tmem_ld32(tacc + 32 * c, v);   // dA
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t gw[4] = {graw[q].x, graw[q].y, graw[q].z, graw[q].w};
                        const uint32_t uw[4] = {uraw[q].x, uraw[q].y, uraw[q].z, uraw[q].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 gf = unpack_bf16x2(gw[i]), uf = unpack_bf16x2(uw[i]);
                            g[8 * q + 2 * i] = gf.x;
                            g[8 * q + 2 * i + 1] = gf.y;
                            u[8 * q + 2 * i] = uf.x;
                            u[8 * q + 2 * i + 1] = uf.y;
                        }
                    }
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
                    const long long gi = grow * (2LL * a.I);
                    const int kq = 2 * a.I / 128;
                    const long long kblk = grow >> 5;       // the warp's 32 rows form one block
                    quant_row32(g, a.q0 + gi + col, a.q0_sf + sf_index(grow, col / 32, kq));
                    quant_row32(u, a.q0 + gi + a.I + col, a.q0_sf + sf_index(grow, (a.I + col) / 32, kq));
                    quant_col32_warp(g, a.q1 + gi + col, a.q1_sf, col, kblk, a.r_atoms);
                    quant_col32_warp(u, a.q1 + gi + a.I + col, a.q1_sf, a.I + col, kblk, a.r_atoms);
                    quant_col32_warp(v, a.q2 + grow * (long long)a.I + col, a.q2_sf, col, kblk, a.r_atoms);
                }
                gu_phase ^= 1u;
                if (!gu_ok) break;
                a.dtw[grow * (2 * a.n_tiles) + 2 * t.nt + half] = dot;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (TWO && rank == 1) mbar_arrive_cluster(tempty + acc, 0);   // the leader's MMAs reuse it
                else mbar_arrive(tempty + acc);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (kTmaOut && lane == 0) bulk_wait_all();   // the stores are complete before the CTA exits
        if (gu_issuer) {
            // every g, u copy issued has landed (bounded) before the CTA exits
            for (int p = 0; p < 2; ++p)
                if (gu_issued[p] > 0) drain_wait(gu_full + p, (uint32_t)((gu_issued[p] - 1) & 1));
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // no commit or release from the peer is still in flight
    if (warp == 1) {
        tc_fence_after();
        if constexpr (TWO) tmem_dealloc_pair(tmem_base, kTmemCols);
        else tmem_dealloc(tmem_base, kTmemCols);
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

// 2-D tensor map over a row-major [outer, inner] array of `esize`-byte elements with box
// {128 bytes, box_rows} and 128-byte swizzle.
static bool tmap_2d(CUtensorMap* m, const void* ptr, int esize, uint64_t inner, uint64_t outer, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * esize};
    const cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / esize), box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUtensorMapDataType dt = esize == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map of packed E2M1 values [outer, inner] (inner / 2 bytes a row), box {128 values,
// box_rows}: the TMA unpacks each 8 bytes (16 values) into a 16-byte shared-memory chunk, so a box
// row lands as 128 bytes with the same 128-byte swizzle as an E4M3 row of 128 values.  The global
// rows must start on 32-byte boundaries and inner must be a multiple of 128.
static bool tmap_2d_fp4(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc || inner % 128 != 0 || reinterpret_cast<uintptr_t>(ptr) % 32 != 0) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner / 2};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map with box {64 bytes, box_rows} and 64-byte swizzle (staged SwiGLU-backward outputs)
static bool tmap_2d_sw64(CUtensorMap* m, const void* ptr, int esize, uint64_t inner, uint64_t outer,
                         uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * esize};
    const cuuint32_t box[2] = {(cuuint32_t)(64 / esize), box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Two-SM MMAs (256 x 256 per CTA pair, each SM holding half of every B tile) for the BF16 weight
// gradients, the backward gate/up product, the SwiGLU backward and the forward down product, where
// they measured faster on GB300 (the pair's shared-memory ring covers half again as much operand
// latency); the forward gate/up keeps one CTA per 128 x 256 tile (a grouped-M pair needs two
// m-tiles of one expert, and the duplicated odd tiles cancel the gain there).
template <int BN, bool MX, bool WGRAD, int EPI>
constexpr bool use_two() {
    return !MX && BN == 256 && (WGRAD || EPI == EPI_PLAIN || EPI == EPI_SWIGLU_BWD || EPI == EPI_WEIGHTED);
}

template <int BN, bool A_MN, bool B_MN, bool SPLIT, bool WGRAD, int EPI, bool MX>
static cudaError_t run(const Ctx& c, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                       const CUtensorMap* tc = nullptr, const CUtensorMap* td = nullptr) {
    constexpr bool TWO = use_two<BN, MX, WGRAD, EPI>();
    constexpr bool PAIR = TWO;
    auto kern = grouped_gemm_kernel<BN, A_MN, B_MN, SPLIT, WGRAD, EPI, MX, TWO>;
    constexpr int kThreads = gemm_threads<EPI, MX && BN == 256>();
    const size_t stage = (size_t)kATileBytes + (TWO ? BN / 2 : BN) * kRowBytes + (MX ? kSfAtom * (1 + BN / 128) : 0);
    const size_t out_bytes = tma_out<EPI, MX, BN>()
                                 ? (size_t)epi_warps<EPI, MX && BN == 256>() * out_box_bytes<EPI, MX && BN == 256>()
                                 : 0;
    const size_t gu_bytes = (MX && EPI == EPI_SWIGLU_BWD) ? (size_t)4 * kBM * kRowBytes : 0;
    const size_t fixed = 1024 + ring_stages<TWO, MX, BN, WGRAD>() * stage + out_bytes + gu_bytes + 256;
    if (tma_out<EPI, MX, BN>() && !tc) return cudaErrorInvalidValue;
    const CUtensorMap& tcm = tc ? *tc : ta;   // kernels without a TMA-stored output never read it
    const CUtensorMap& tdm = td ? *td : tcm;
    const size_t smem = fixed + (size_t)2 * (a.E + 1) * 4;
    const size_t smem_max = fixed + (size_t)2 * (kMaxExperts + 1) * 4;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int grid = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
        grid = c.num_sms;
        if (attr_err == cudaSuccess && PAIR) {
            // as many two-CTA clusters as can be resident at once (one CTA per SM)
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(c.num_sms);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem_max;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int clusters = 0;
            attr_err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (attr_err == cudaSuccess) grid = 2 * std::max(1, std::min(clusters, c.num_sms / 2));
        }
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (!PAIR) return launch_pdl(kern, c.num_sms, kThreads, smem, c.st, ta, tb, tcm, tdm, a);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.st;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tcm, tdm, a);
}

int bwd_down_bn(int64_t I) { return (I % 256 == 0) ? 256 : 128; }

static cudaError_t launch_gemm_bf16(const Ctx& c, GemmKind kind, const void* W, void* out, GemmArgs& a) {
    const Layout& L = *c.L;
    char* b = c.base;
    const int64_t H = L.H, I = L.I, E = L.E, R = L.rows;
    const int oes = a.out_f32 ? 4 : 2;   // weight-gradient output element size
    CUtensorMap ta, tb, tc, td;
    switch (kind) {
        case GemmKind::FwdGateUp:
        case GemmKind::FwdGateUpSaveOnly:
            if (!tmap_2d(&ta, b + L.xperm, 2, H, R, 128) || !tmap_2d(&tb, W, 2, H, E * 2 * I, 128) ||
                !tmap_2d(&tc, b + L.hid, 2, I, R, 32) || !tmap_2d(&td, b + L.gu, 2, 2 * I, R, 32))
                return cudaErrorInvalidValue;
            a.n_tiles = (int)(I / 128); a.k_blocks = (int)(H / 64); a.b_rows_e = (int)(2 * I); a.b_up = (int)I;
            a.out0 = b + L.hid; a.out1 = b + L.gu;
            return kind == GemmKind::FwdGateUp
                       ? run<256, false, false, true, false, EPI_SWIGLU, false>(c, ta, tb, a, &tc, &td)
                       : run<256, false, false, true, false, EPI_GU_ONLY, false>(c, ta, tb, a, &tc, &td);
        case GemmKind::FwdDown:
            // K-major B boxes hold the rows one CTA loads: all 256, or its 128-row half on CTA pairs
            if (!tmap_2d(&ta, b + L.hid, 2, I, R, 128) ||
                !tmap_2d(&tb, W, 2, I, E * H, use_two<256, false, false, EPI_WEIGHTED>() ? 128 : 256) ||
                !tmap_2d(&tc, b + L.ypart, 2, H, R, 32))
                return cudaErrorInvalidValue;
            a.n_tiles = (int)(H / 256); a.k_blocks = (int)(I / 64); a.b_rows_e = (int)H;
            a.out0 = b + L.ypart; a.ld0 = (int)H;
            a.w_in_a = 1;   // A = w h from the gate/up epilogue
            return run<256, false, false, false, false, EPI_WEIGHTED, false>(c, ta, tb, a, &tc);
        case GemmKind::FwdDownReduce:
            if (!tmap_2d(&ta, b + L.hid, 2, I, R, 128) || !tmap_2d(&tb, W, 2, I, E * H, 256))
                return cudaErrorInvalidValue;
            a.n_tiles = (int)(H / 256); a.k_blocks = (int)(I / 64); a.b_rows_e = (int)H;
            a.yacc = reinterpret_cast<float*>(b + L.ypart); a.ld0 = (int)H;
            a.w_in_a = 1;
            // the reducing epilogue stages in its box but stores nothing by TMA: no output map
            return run<256, false, false, false, false, EPI_WEIGHTED_RED, false>(c, ta, tb, a, &ta);
        case GemmKind::BwdDown: {
            const int bn = bwd_down_bn(I);
            // w h is not an output here: the forward's gate/up epilogue saved it (hid)
            if (!tmap_2d(&ta, b + L.dyperm, 2, H, R, 128) || !tmap_2d(&tb, W, 2, I, E * H, 64) ||
                !tmap_2d_sw64(&tc, b + L.dg, 2, 2 * I, R, 32))
                return cudaErrorInvalidValue;
            a.n_tiles = (int)(I / bn); a.k_blocks = (int)(H / 64); a.b_rows_e = (int)H;
            a.out0 = b + L.dg; a.dtw = reinterpret_cast<float*>(b + L.dtw);
            return bn == 256 ? run<256, false, true, false, false, EPI_SWIGLU_BWD, false>(c, ta, tb, a, &tc, &tc)
                             : run<128, false, true, false, false, EPI_SWIGLU_BWD, false>(c, ta, tb, a, &tc, &tc);
        }
        case GemmKind::BwdGateUp:
            if (!tmap_2d(&ta, b + L.dg, 2, 2 * I, R, 128) || !tmap_2d(&tb, W, 2, H, E * 2 * I, 64) ||
                !tmap_2d(&tc, b + L.ypart, 2, H, R, 32))
                return cudaErrorInvalidValue;
            a.n_tiles = (int)(H / 256); a.k_blocks = (int)(2 * I / 64); a.b_rows_e = (int)(2 * I);
            a.out0 = b + L.ypart; a.ld0 = (int)H;
            return run<256, false, true, false, false, EPI_PLAIN, false>(c, ta, tb, a, &tc);
        case GemmKind::WgradDown: {
            const int bn = bwd_down_bn(I);
            if (!tmap_2d(&ta, b + L.dyperm, 2, H, R, 64) || !tmap_2d(&tb, b + L.hid, 2, I, R, 64) ||
                !tmap_2d(&tc, out, oes, I, E * H, 32))
                return cudaErrorInvalidValue;
            a.m_tiles = (int)(H / 128); a.n_tiles = (int)(I / bn);
            a.out0 = out; a.ld0 = (int)I; a.out_e_stride = H * I;
            return bn == 256 ? run<256, true, true, false, true, EPI_WGRAD, false>(c, ta, tb, a, &tc)
                             : run<128, true, true, false, true, EPI_WGRAD, false>(c, ta, tb, a, &tc);
        }
        case GemmKind::WgradGateUp:
            if (!tmap_2d(&ta, b + L.dg, 2, 2 * I, R, 64) || !tmap_2d(&tb, b + L.xperm, 2, H, R, 64) ||
                !tmap_2d(&tc, out, oes, H, E * 2 * I, 32))
                return cudaErrorInvalidValue;
            a.m_tiles = (int)(2 * I / 128); a.n_tiles = (int)(H / 256);
            a.out0 = out; a.ld0 = (int)H; a.out_e_stride = 2 * I * H;
            return run<256, true, true, false, true, EPI_WGRAD, false>(c, ta, tb, a, &tc);
    }
    return cudaErrorInvalidValue;
}

// MXFP8: 128 x 256 tiles (one accumulator, drained to registers) for every product but the SwiGLU
// backward, which keeps 128 x 128 tiles with two accumulators (as does a W2 weight gradient with
// I % 256 != 0).  A 128 x 128 block-scaled MMA with its two scale copies issues at about half the
// rate of a 128 x 256 one with its three.  Operands
// are the E4M3 copies made by the quantiser and the epilogues (quant.cu, the fused epilogues
// above); in the FP8 x FP4 forward the weights are the quantiser's packed E2M1 copies.
static cudaError_t launch_gemm_mx(const Ctx& c, GemmKind kind, void* out, GemmArgs& a) {
    const Layout& L = *c.L;
    const MxLayout& M = L.mx;
    char* b = c.base;
    const int64_t H = L.H, I = L.I, E = L.E, R = L.rows;
    auto u8 = [&](size_t off) { return reinterpret_cast<const uint8_t*>(b + off); };
    const int oes = a.out_f32 ? 4 : 2;   // weight-gradient output element size
    CUtensorMap ta, tb, tc, td;
    switch (kind) {
        case GemmKind::FwdGateUp:
        case GemmKind::FwdGateUpSaveOnly:
            // 256 weight rows = two [64 gate | 64 up] blocks = 128 I-columns per tile
            if (!tmap_2d(&ta, b + M.x_r, 1, H, R, 128) ||
                !(L.fp4w ? tmap_2d_fp4(&tb, b + M.w13_r, H, E * 2 * I, 256)
                         : tmap_2d(&tb, b + M.w13_r, 1, H, E * 2 * I, 256)) ||
                !tmap_2d_sw64(&td, b + L.gu, 2, 2 * I, R, 32))
                return cudaErrorInvalidValue;
            a.b_fmt = L.fp4w ? kFmtE2M1B : 0u;
            a.n_tiles = (int)(I / 128); a.k_blocks = (int)(H / 128); a.b_rows_e = (int)(2 * I);
            a.sfA = u8(M.x_r_sf); a.sfA_kt = (int)(H / 128);
            a.sfB = u8(M.w13_r_sf); a.sfB_kt = (int)(H / 128);
            a.out0 = b + L.hid; a.out1 = b + L.gu;
            a.q0 = reinterpret_cast<uint8_t*>(b + M.h_r); a.q0_sf = reinterpret_cast<uint8_t*>(b + M.h_r_sf);
            return kind == GemmKind::FwdGateUp
                       ? run<256, false, false, true, false, EPI_SWIGLU, true>(c, ta, tb, a, &td, &td)
                       : run<256, false, false, true, false, EPI_GU_ONLY, true>(c, ta, tb, a, &td, &td);
        case GemmKind::FwdDown:
            if (!tmap_2d(&ta, b + M.h_r, 1, I, R, 128) ||
                !(L.fp4w ? tmap_2d_fp4(&tb, b + M.w2_r, I, E * H, 256) : tmap_2d(&tb, b + M.w2_r, 1, I, E * H, 256)) ||
                !tmap_2d_sw64(&tc, b + L.ypart, 2, H, R, 32))
                return cudaErrorInvalidValue;
            a.b_fmt = L.fp4w ? kFmtE2M1B : 0u;
            a.n_tiles = (int)(H / 256); a.k_blocks = (int)(I / 128); a.b_rows_e = (int)H;
            a.sfA = u8(M.h_r_sf); a.sfA_kt = (int)(I / 128);
            a.sfB = u8(M.w2_r_sf); a.sfB_kt = (int)(I / 128);
            a.out0 = b + L.ypart; a.ld0 = (int)H;
            return run<256, false, false, false, false, EPI_WEIGHTED, true>(c, ta, tb, a, &tc);
        case GemmKind::BwdDown:
            // td: the saved [g|u] rows, read by TMA in 128-row x 64-column boxes
            if (!tmap_2d(&ta, b + M.dy_r, 1, H, R, 128) || !tmap_2d(&tb, b + M.w2_c, 1, I, E * H, 128) ||
                !tmap_2d(&td, b + L.gu, 2, 2 * I, R, 128))
                return cudaErrorInvalidValue;
            a.n_tiles = (int)(I / 128); a.k_blocks = (int)(H / 128); a.b_rows_e = (int)H;
            a.sfA = u8(M.dy_r_sf); a.sfA_kt = (int)(H / 128);
            a.sfB = u8(M.w2_c_sf); a.sfB_kt = (int)(E * H / 128);
            a.out0 = b + L.dg; a.dtw = reinterpret_cast<float*>(b + L.dtw);
            a.q0 = reinterpret_cast<uint8_t*>(b + M.dg_r); a.q0_sf = reinterpret_cast<uint8_t*>(b + M.dg_r_sf);
            a.q1 = reinterpret_cast<uint8_t*>(b + M.dg_c); a.q1_sf = reinterpret_cast<uint8_t*>(b + M.dg_c_sf);
            a.q2 = reinterpret_cast<uint8_t*>(b + M.hw_c); a.q2_sf = reinterpret_cast<uint8_t*>(b + M.hw_c_sf);
            a.r_atoms = (int)(R / 128);
            return run<128, false, true, false, false, EPI_SWIGLU_BWD, true>(c, ta, tb, a, nullptr, &td);
        case GemmKind::BwdGateUp:
            if (!tmap_2d(&ta, b + M.dg_r, 1, 2 * I, R, 128) || !tmap_2d(&tb, b + M.w13_c, 1, H, E * 2 * I, 128) ||
                !tmap_2d_sw64(&tc, b + L.ypart, 2, H, R, 32))
                return cudaErrorInvalidValue;
            a.n_tiles = (int)(H / 256); a.k_blocks = (int)(2 * I / 128); a.b_rows_e = (int)(2 * I);
            a.sfA = u8(M.dg_r_sf); a.sfA_kt = (int)(2 * I / 128);
            a.sfB = u8(M.w13_c_sf); a.sfB_kt = (int)(E * 2 * I / 128);
            a.out0 = b + L.ypart; a.ld0 = (int)H;
            return run<256, false, true, false, false, EPI_PLAIN, true>(c, ta, tb, a, &tc);
        case GemmKind::WgradDown:
            // drained 128 x 256 tiles whose fp32 rows leave through 64-byte-swizzled TMA boxes
            if (!tmap_2d(&ta, b + M.dy_c, 1, H, R, 128) || !tmap_2d(&tb, b + M.hw_c, 1, I, R, 128))
                return cudaErrorInvalidValue;
            a.m_tiles = (int)(H / 128);
            a.sfA = u8(M.dy_c_sf); a.sfA_kt = (int)(R / 128);
            a.sfB = u8(M.hw_c_sf); a.sfB_kt = (int)(R / 128);
            a.out0 = out; a.ld0 = (int)I; a.out_e_stride = H * I;
            if (I % 256 == 0) {
                if (!tmap_2d_sw64(&tc, out, oes, I, E * H, 32)) return cudaErrorInvalidValue;
                a.n_tiles = (int)(I / 256);
                return run<256, true, true, false, true, EPI_WGRAD, true>(c, ta, tb, a, &tc);
            }
            if (!tmap_2d(&tc, out, oes, I, E * H, 32)) return cudaErrorInvalidValue;
            a.n_tiles = (int)(I / 128);
            return run<128, true, true, false, true, EPI_WGRAD, true>(c, ta, tb, a, &tc);
        case GemmKind::WgradGateUp:
            if (!tmap_2d(&ta, b + M.dg_c, 1, 2 * I, R, 128) || !tmap_2d(&tb, b + M.x_c, 1, H, R, 128) ||
                !tmap_2d_sw64(&tc, out, oes, H, E * 2 * I, 32))
                return cudaErrorInvalidValue;
            a.m_tiles = (int)(2 * I / 128); a.n_tiles = (int)(H / 256);   // H % 256 == 0
            a.sfA = u8(M.dg_c_sf); a.sfA_kt = (int)(R / 128);
            a.sfB = u8(M.x_c_sf); a.sfB_kt = (int)(R / 128);
            a.out0 = out; a.ld0 = (int)H; a.out_e_stride = 2 * I * H;
            return run<256, true, true, false, true, EPI_WGRAD, true>(c, ta, tb, a, &tc);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(const Ctx& c, GemmKind kind, const void* W, void* out, bool out_f32, bool save_gu) {
    const Layout& L = *c.L;
    char* b = c.base;
    GemmArgs a{};
    a.mtile = reinterpret_cast<const int*>(b + L.mtile);
    a.order = reinterpret_cast<const int*>(b + L.order);
    a.row_slot = reinterpret_cast<const int*>(b + L.row_slot);
    a.topk_w = c.topk_w;
    a.gu = reinterpret_cast<const __nv_bfloat16*>(b + L.gu);
    a.status = c.status;
    a.E = (int)L.E;
    a.I = (int)L.I;
    a.k = (int)L.k;
    a.out_f32 = out_f32 ? 1 : 0;
    a.save_gu = save_gu ? 1 : 0;
    a.wait_limit = c.wait_limit > 0 ? c.wait_limit : kWaitTimeoutCycles;
    a.withhold_loads = (c.test_flags & MOE_TEST_WITHHOLD_LOADS) ? 1 : 0;
    const bool fwd = kind == GemmKind::FwdGateUp || kind == GemmKind::FwdGateUpSaveOnly || kind == GemmKind::FwdDown ||
                     kind == GemmKind::FwdDownReduce;
    const bool mx = fwd ? L.mx_fwd : L.mx_bwd;   // fp8_bwd: BF16 forward products, MXFP8 backward ones
    const int trace_id = (mx ? kTraceGemmMx : kTraceGemm) + (int)kind;
    trace_begin(c.st, trace_id);
    const cudaError_t err = mx ? launch_gemm_mx(c, kind, out, a) : launch_gemm_bf16(c, kind, W, out, a);
    trace_end(c.st, trace_id);
    return err;
}

}  // namespace moe
