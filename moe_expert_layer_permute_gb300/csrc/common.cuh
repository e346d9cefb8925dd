// common.cuh - sm_103a device primitives used by the MoE layer kernels: mbarriers with bounded
// waits, TMA tile loads, tcgen05 (TMEM allocation, MMA, commit, loads) and the shared-memory /
// instruction descriptors of the 5th-generation tensor cores.  All written as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_layer.h"

namespace moe {

// ------------------------------------------------------------------------------------------
// status word (first 4 bytes of the scratch buffer)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, MOE_DEV_OK, code);
}

// A wait that outlives this many SM cycles (about 2 s at 2 GHz) is treated as a hang: the
// kernel records MOE_DEV_TIMEOUT and leaves its loops.  Legitimate waits are microseconds.  This is
// the default; a caller may set another limit per scratch buffer (moe_set_wait_limit).
constexpr long long kWaitTimeoutCycles = 4000000000ll;
// While a kernel that gave up drains its in-flight copies and MMAs before exiting, each wait is
// bounded by this many cycles whatever the configured limit (in-flight work ends in microseconds).
constexpr long long kDrainCycles = kWaitTimeoutCycles / 8;

// Programmatic dependent launch.  Every kernel of this library is launched with programmatic stream
// serialization and starts with grid_dep_wait(): it returns once the kernel launched before it on
// the stream has completed and its memory is visible (at once for a launch without a programmatic
// dependency), so by induction all earlier work on the stream is done before any kernel reads or
// writes global memory.  The next launch is then scheduled as this kernel's blocks exit rather than
// after the whole grid has drained, which hides the launch gap at each kernel boundary (1-2 % of the
// layer on GB300).  No kernel triggers its dependents early: blocks launched ahead of time and
// waiting cost more than they saved (the layer measured 0.6-5 % slower).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete.  Gives up (returns false) when
// *abort becomes non-zero or the wait exceeds `limit` cycles; in the latter case it raises *abort
// itself and records MOE_DEV_TIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                          long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            set_status(status, MOE_DEV_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion counted on an mbarrier)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Plain bulk copy global -> shared (both addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// TMA tile store shared -> global of the box at {c0, c1}, tracked as a bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, const void* src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// waits until at most N of this thread's most recent bulk groups still read their shared source
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// waits until every bulk group this thread committed has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// orders this thread's generic-proxy writes to its CTA's shared memory before later async-proxy
// accesses to them (e.g. a TMA store reading what the thread staged)
__device__ __forceinline__ void fence_proxy_async_cta() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}
// dst[0..3] += the four fp32 values in v, one vector atomic reduction (no return value)
__device__ __forceinline__ void red_add_f32x4(float* dst, uint4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(__uint_as_float(v.x)),
                 "f"(__uint_as_float(v.y)), "f"(__uint_as_float(v.z)), "f"(__uint_as_float(v.w))
                 : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---- clusters of two CTAs (two-SM MMAs): rank, cluster barrier ---------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of both CTAs; orders every shared-memory access before it in either CTA before
// every access after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation (kind::f16).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= (A * 2^sfA) * (B * 2^sfB)^T with E4M3 A/B and one E8M0 scale per 32 K-elements
// (kind::mxf8f6f4, block_scale, scale_vec::1X); scales are read from tensor memory.
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy 32 rows x 128 bits from shared memory to tensor memory, replicated into all four 32-lane
// quarters (4 columns): one 512-byte scale-factor atom.
__device__ __forceinline__ void tmem_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// ---- CTA pairs driving one MMA (cta_group::2): the leader CTA (rank 0) issues each M = 256 MMA,
// which reads A rows [0, 128) and the first half of B's N from the leader's shared memory and the
// rest from the peer's at the same offsets, and writes rows [0, 128) of D to the leader's TMEM
// and rows [128, 256) to the peer's.  Allocation is collective: one warp in each CTA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the mbarrier at `bar`'s offset in every CTA of `mask` once the pair's MMAs issued so
// far by this thread are done.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}
// Shared::cluster address of the object at `p`'s offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// TMA tile load into this CTA's shared memory whose transaction bytes complete on an mbarrier of
// either CTA of the pair (bar_cluster: a shared::cluster address, e.g. the leader's barrier).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int c0,
                                                 int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

// Arrive (release, cluster scope) on the mbarrier at `bar`'s offset in cluster CTA `rank`.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
// try_wait with acquire at cluster scope (for phases completed by arrivals from the peer CTA)
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                                  long long limit) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            set_status(status, MOE_DEV_TIMEOUT);
            return false;
        }
    }
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------------------------------
// descriptors
// ------------------------------------------------------------------------------------------
// Shared-memory matrix descriptor (tcgen05 format): start address, leading / stride byte
// offsets (16-byte units), descriptor version 1 at bits 46-47, 128-byte swizzle at bits 61-63.
//   K-major, 128B swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO); LBO unused.
//   MN-major, 128B swizzle: each 128-byte row holds 64 MN-consecutive 16-bit values at one k;
//     8 k-rows form a 1024-byte group (SBO = 1024) and the next 64 MN values start LBO bytes on.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Descriptor of an unswizzled shared-memory block whose 8-row x 16-byte core matrices are
// `sbo` bytes apart (used for the 512-byte scale-factor atoms: rows of 16 bytes, SBO = 128).
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// B-operand format field of the kind::mxf8f6f4 instruction descriptor for E2M1 (bits 10-12 = 5).
constexpr uint32_t kFmtE2M1B = 5u << 10;

// Instruction descriptor of kind::mxf8f6f4 with E4M3 A/B, fp32 D and E8M0 block scales;
// sfa_id / sfb_id select the byte (K-block) of the 32-bit scale column each MMA reads.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, bool a_mn_major, bool b_mn_major, uint32_t sfa_id,
                                                  uint32_t sfb_id) {
    return ((sfb_id & 3u) << 4)                        // B scale-factor id
           | (0u << 7) | (0u << 10)                    // A, B: E4M3 (B: kFmtE2M1B OR-ed in)
           | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | (1u << 23)     // scales are UE8M0
           | ((uint32_t)(M >> 4) << 24) | ((sfa_id & 3u) << 29);
}

// Instruction descriptor of kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4)                                   // D: f32
           | (1u << 7)                                 // A: bf16
           | (1u << 10)                                // B: bf16
           | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------
// small numeric helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}
// 1/x by the hardware's approximate reciprocal (rcp.approx, about 1 ulp; subnormals flushed).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// sigmoid(z) = 1 / (1 + e^-z); 1 + e^-z is at least 1, and e^-z = inf gives 0
__device__ __forceinline__ float sigmoidf_fast(float z) { return rcp_approx(1.0f + __expf(-z)); }

// ------------------------------------------------------------------------------------------
// MXFP8 (OCP Microscaling v1.0): E4M3 values, one E8M0 scale per 32 values
// ------------------------------------------------------------------------------------------
// Byte of MN-row mn / K-block kblock in the scale-atom layout the block-scaled MMA reads after a
// 32x128b.warpx4 copy: atoms of 128 MN-rows x 4 K-blocks (512 B), k_atoms = K / 128 per MN tile.
__host__ __device__ __forceinline__ long long sf_index(long long mn, long long kblock, long long k_atoms) {
    return ((mn >> 7) * k_atoms + (kblock >> 2)) * 512 + 16 * (mn & 31) + 4 * ((mn >> 5) & 3) + (kblock & 3);
}

// MXFP8 block scale from the bits of a non-negative finite amax: the shared exponent
// floor(log2(amax)) - 8 (8 = the largest E4M3 exponent), stored biased by 127 in one byte, and the
// exact factor 2^-exp.  For a normal amax the biased exponent field is floor(log2(amax)) + 127, so
// the byte is the field - 8; fields below 9 (amax < 2^-118, subnormals and zero) all clamp to
// byte 0.  2^-exp then has the biased exponent 254 - byte, always a normal float.
__device__ __forceinline__ void mx_scale_bits(uint32_t amax_bits, uint8_t* sf, float* inv) {
    const int b = max((int)(amax_bits >> 23) - 8, 0);
    *sf = (uint8_t)b;
    *inv = __uint_as_float((uint32_t)(254 - b) << 23);
}

// MXFP4 (E2M1 values) block scale: floor(log2(amax)) - 2 (2 = the largest E2M1 exponent), by the
// same field arithmetic as mx_scale_bits.
__device__ __forceinline__ void mx_scale_bits_e2m1(uint32_t amax_bits, uint8_t* sf, float* inv) {
    const int b = max((int)(amax_bits >> 23) - 2, 0);
    *sf = (uint8_t)b;
    *inv = __uint_as_float((uint32_t)(254 - b) << 23);
}

// Two values to E2M1 (round to nearest even, saturated to +-6), a in the low nibble.
__device__ __forceinline__ uint32_t to_e2m1x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
}

// Two values to E4M3 (round to nearest even, saturated to +-448), packed low byte first.
__device__ __forceinline__ uint16_t to_e4m3x2(float a, float b) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// 32 values scaled by inv[] (per value) to 32 E4M3 bytes at a 32-byte aligned destination.
__device__ __forceinline__ void store_e4m3x32(uint8_t* dst, const float* v, const float* inv) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        w[j] = (uint32_t)to_e4m3x2(v[4 * j] * inv[4 * j], v[4 * j + 1] * inv[4 * j + 1]) |
               ((uint32_t)to_e4m3x2(v[4 * j + 2] * inv[4 * j + 2], v[4 * j + 3] * inv[4 * j + 3]) << 16);
    // one 32-byte store (dst is 32-byte aligned: a row's 32-column block of E4M3 codes)
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Row block: the thread's 32 consecutive values of one row share one scale.
__device__ __forceinline__ void quant_row32(const float* v, uint8_t* dst, uint8_t* sf_dst) {
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
    uint8_t sf;
    float inv;
    mx_scale_bits(__float_as_uint(amax), &sf, &inv);
    float invs[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) invs[j] = inv;
    store_e4m3x32(dst, v, invs);
    *sf_dst = sf;
}

// Column blocks: the 32 lanes of a warp hold 32 consecutive rows (lane = row), each the same 32
// columns; column j's scale is shared by the 32 rows.  The column maxima come from one warp
// max-reduction each on the |value| bit patterns (non-negative floats order like integers); lane
// j keeps column j's maximum, derives its scale and 2^-exp, and the factors are broadcast back.
// Lane j writes the scale byte of column col0 + j; every lane writes its own row's 32 bytes.
__device__ __forceinline__ void quant_col32_warp(const float* v, uint8_t* dst_row, uint8_t* sf_base,
                                                 long long col0, long long kblock, long long k_atoms) {
    const int lane = threadIdx.x & 31;
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[j])));
        if (j == lane) mine = m;
    }
    uint8_t sf;
    float my_inv;
    mx_scale_bits(mine, &sf, &my_inv);
    float inv[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) inv[j] = __shfl_sync(0xffffffffu, my_inv, j);
    store_e4m3x32(dst_row, v, inv);
    sf_base[sf_index(col0 + lane, kblock, k_atoms)] = sf;
}

}  // namespace moe
