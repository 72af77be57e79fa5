// Inline-PTX wrappers for the sm_103a features the kernels use: mbarrier,
// TMA (cp.async.bulk / cp.async.bulk.tensor), tcgen05 (TMEM allocation,
// block-scaled MMA, scale-factor copy, TMEM loads) and the FP8/FP4 converts.
// Written from the public PTX ISA description of each instruction.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace nvfp4 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
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

// Bounded wait for the phase of the given parity to complete.  Gives up
// after `budget` SM cycles or as soon as *abort becomes non-zero; returns
// false in both cases.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                                  long long budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (clock64() - t0 > budget) return false;
    }
}

// Order this thread's generic-proxy writes to shared memory before later async-proxy reads
// of it (TMA, tcgen05.mma / tcgen05.cp operands) that another thread issues after a barrier.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
        : "memory");
}

// Plain bulk copy global -> shared; dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bring a tensor-map box into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}
// Bring `bytes` (multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 eviction-priority policies for the cache_hint operands.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// Copy a 32-row x 16-byte block of shared memory into TMEM columns
// [taddr, taddr+4) of lanes 0-31, replicated into all four 32-lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D(tmem) (+)= A(smem, E2M1) x B(smem, E2M1)^T with UE4M3 scales per 16 K-elements
// (scale_vec::4X), FP32 accumulation.  M=128, N from idesc, K=64 per instruction.
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}
// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format) of a K-major tile whose rows are
// kSpan bytes (128 or 64) long and swizzled with the same span, 8-row groups
// 8*kSpan bytes apart.  The tile base must be aligned to 8*kSpan bytes (1024 is
// used); advancing the start address by 32 bytes steps K by 64 FP4 elements.
template <int kSpan>
__device__ __forceinline__ uint64_t sdesc_k_swizzled(uint32_t saddr) {
    static_assert(kSpan == 128 || kSpan == 64, "supported swizzle spans");
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);        // start address >> 4, bits 0-13
    d |= static_cast<uint64_t>(1) << 16;                          // leading byte offset (unused here)
    d |= static_cast<uint64_t>((8 * kSpan) >> 4) << 32;           // stride byte offset, bits 32-45
    d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
    d |= static_cast<uint64_t>(kSpan == 128 ? 2 : 4) << 61;       // swizzle: 128B = 2, 64B = 4
    return d;
}
// Descriptor of a 32-row x 16-byte scale-factor block (no swizzle; 8-row groups 128 B apart).
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}
// Instruction descriptor of kind::mxf4nvf4: A and B E2M1, K-major, UE4M3 scales.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7)                                  // A format: E2M1
           | (1u << 10)                               // B format: E2M1
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (0u << 23)                               // scale format: UE4M3
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ------------------------------------------------------------------ elected-lane issue
// Variants for code that the whole warp executes in step: every lane runs the asm and
// elect.sync picks one lane to issue the instruction.  Keeping the issuing loop
// warp-uniform lets its operands live in uniform registers; issuing the same stream
// of tcgen05 operations from one lane of a diverged warp is much slower.
#define NVFP4_ELECT "{\n\t.reg .pred ep;\n\t.reg .b32 er;\n\telect.sync er|ep, 0xffffffff;\n\t@ep "

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint64_t* bar, uint32_t bytes) {
    asm volatile(NVFP4_ELECT "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d_elect(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                  uint64_t policy) {
    asm volatile(NVFP4_ELECT
                 "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void tma_load_4d_elect(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                  int z, int w, uint64_t policy) {
    asm volatile(NVFP4_ELECT
                 "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;\n\t}" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w),
                 "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_load_elect(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
    asm volatile(NVFP4_ELECT
                 "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void tc_cp_32x128b_warpx4_elect(uint32_t taddr, uint64_t sdesc) {
    asm volatile(NVFP4_ELECT "tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}
__device__ __forceinline__ void tc_mma_nvf4_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred ep, acc;\n\t.reg .b32 er;\n\telect.sync er|ep, 0xffffffff;\n\t"
        "setp.ne.b32 acc, %4, 0;\n\t"
        "@ep tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], acc;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}
// tcgen05.commit from the elected lane: it tracks the operations that lane issued, so the
// same (deterministic) lane must have issued them through the _elect variants above.
__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
    asm volatile(NVFP4_ELECT "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// One full stage of the block-scaled main loop from the elected lane: for j = 0..3,
// copy the A scales (512-byte tile at sfa + 512 j) to TMEM column sf_col + 4 j, the two
// B scale tiles (sfb0/sfb1 + 512 j) to sf_col + 16 + 8 j and + 4, then
// D += A[k 64j..] x B[k 64j..] with those scales; `acc0` = accumulate for j = 0 (the
// later MMAs of the stage always accumulate).  Descriptor start fields advance by
// 512 B (32 units of 16 B) per scale tile and 32 B (2 units) per K=64 step.
__device__ __forceinline__ void tc_stage4_nvf4_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                     uint64_t sfa, uint64_t sfb0, uint64_t sfb1, uint32_t sf_col,
                                                     uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred ep, p0, p1;\n\t.reg .b32 er, ca, cb0, cb1;\n\t.reg .b64 a, b, s0, s1, s2;\n\t"
        "elect.sync er|ep, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %8, 0;\n\t"
        "setp.eq.b32 p1, %8, %8;\n\t"
        // j = 0
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [%7], %4;\n\t"
        "add.u32 cb0, %7, 16;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb0], %5;\n\t"
        "add.u32 cb1, %7, 20;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb1], %6;\n\t"
        "@ep tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%7], [cb0], p0;\n\t"
        // j = 1
        "add.u32 ca, %7, 4;\n\t add.u32 cb0, %7, 24;\n\t add.u32 cb1, %7, 28;\n\t"
        "add.s64 s0, %4, 32;\n\t add.s64 s1, %5, 32;\n\t add.s64 s2, %6, 32;\n\t"
        "add.s64 a, %1, 2;\n\t add.s64 b, %2, 2;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [ca], s0;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb0], s1;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb1], s2;\n\t"
        "@ep tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a, b, %3, [ca], [cb0], p1;\n\t"
        // j = 2
        "add.u32 ca, %7, 8;\n\t add.u32 cb0, %7, 32;\n\t add.u32 cb1, %7, 36;\n\t"
        "add.s64 s0, %4, 64;\n\t add.s64 s1, %5, 64;\n\t add.s64 s2, %6, 64;\n\t"
        "add.s64 a, %1, 4;\n\t add.s64 b, %2, 4;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [ca], s0;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb0], s1;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb1], s2;\n\t"
        "@ep tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a, b, %3, [ca], [cb0], p1;\n\t"
        // j = 3
        "add.u32 ca, %7, 12;\n\t add.u32 cb0, %7, 40;\n\t add.u32 cb1, %7, 44;\n\t"
        "add.s64 s0, %4, 96;\n\t add.s64 s1, %5, 96;\n\t add.s64 s2, %6, 96;\n\t"
        "add.s64 a, %1, 6;\n\t add.s64 b, %2, 6;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [ca], s0;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb0], s1;\n\t"
        "@ep tcgen05.cp.cta_group::1.32x128b.warpx4 [cb1], s2;\n\t"
        "@ep tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a, b, %3, [ca], [cb0], p1;\n\t"
        "}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "l"(sfa), "l"(sfb0), "l"(sfb1), "r"(sf_col), "r"(acc0)
        : "memory");
}
#undef NVFP4_ELECT

// ------------------------------------------------------------------ converts
// Two FP32 -> packed E2M1 pair, round-to-nearest-even, saturating; `lo` goes to bits 0-3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;
}
// FP32 -> E4M3 code, round-to-nearest-even, saturating to +-448.
__device__ __forceinline__ uint32_t cvt_e4m3(float x) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
    return r & 0xFFu;
}
// Exact value of an unsigned E4M3 code 0..126 (bias 7, 3 mantissa bits).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    const uint32_t e = code >> 3, m = code & 7u;
    if (e == 0) return static_cast<float>(m) * 0.001953125f;          // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));            // (1 + m/8) * 2^(e-7)
}

}  // namespace nvfp4
