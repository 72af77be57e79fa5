// Grouped block-scaled FP4 GEMMs of the expert forward on tcgen05.
//
//   FC1:  acc[r, n] = sum_k (qa*sa)[r,k] (qw*sw)[e*2I+n, k]      (gate n < I, up n >= I)
//         v = (acc*g^x[r])*g^w[n] in FP32, gate/up = bf16(v),
//         h = bf16( f32( silu(gate)*up ) * p[r] ),  amax2[r] = max|h[r,:]|
//   FC2:  y[pair(r), :] = bf16( (acc*g2[r])*g^w2[:] )
//
// What is computed follows "miniTE diagnoses and narrows the cross-engine
// execution gap of NVFP4 RL" (onedev.kr/papers/1404), sections "How it
// differs" (FP32 epilogue with g^x g^w before the BF16 cast; router
// probability on the SwiGLU activation before FC2) and "How to use it"
// (expert boundaries as device offsets; FC2 maxima from the producer of the
// router-weighted activation; separate FC1/FC2 settings), and "Finishing RL
// training faster...", section 4.4 "Expert GEMM: two layouts, same row
// result" (SiLU(gate)*up in FP32, one rounding; each row accumulated in a
// fixed order, independent of its neighbours).
//
// Kernel design (sm_103a):
//  * persistent: one 608-thread CTA per SM walks the (m-tile, n-tile) list;
//    the list length comes from the device-side expert offsets, so nothing
//    is read back to the host;
//  * two TMA producers, because one issuing thread caps what an SM pulls from
//    L2 well below what it can take in: warp 0 loads the A tile (128 rows x
//    256 K, 16 KB, 128B swizzle) and its scale-factor tiles, warp 18 the B
//    tile (256 rows x 256 K in one box: FC2 256 consecutive weight rows, FC1
//    through a 4D map the 128 gate rows and the matching 128 up rows, so one
//    tile holds both halves of SwiGLU) and its scale-factor tiles; 3-stage
//    mbarrier ring, each stage's barrier counting both producers;
//  * producers and MMA issuer run warp-uniform loops and issue through an
//    elect.sync-chosen lane (a single diverged lane issues tcgen05 work at
//    well under half the rate);
//  * warp 1 = MMA issuer: tcgen05.cp moves the stage's scale factors into
//    TMEM, then 4 x tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//    (M=128, N=256, K=64) accumulate in a 256-column FP32 TMEM tile;
//  * warps 2-17 = epilogue, four warps per 32-lane TMEM quarter, each taking
//    64 accumulator columns (FC1: 32 gate columns and the matching 32 up
//    columns; FC2: 64 output columns), so four epilogue warps share each
//    scheduler to hide their latencies.  They copy their accumulator columns
//    to registers and release TMEM at once, so the next tile's MMAs run while
//    they apply the FP32 scales (staged in shared memory per tile), BF16
//    casts and the fused SwiGLU x prob; every lane writes its own row's
//    values with 32-byte stores (FC2 rows to their (token, slot) places).
//    19 warps leave a thread 96 registers (five warps share three of the
//    SM's sub-partitions, each with 16K registers).
//  Every row's arithmetic is the same whatever tile, expert or batch it is
//  in: one tile shape, no split-K, K always walked 0..K-1 in 64-wide steps.
//  All waits are bounded (NVFP4_ERR_DEVICE_TIMEOUT, then a clean exit).
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "nvfp4_quant.cuh"
#include "ptx.cuh"

namespace nvfp4 {

// SiLU of every BF16 value, correctly rounded to FP32, indexed by the BF16 bit pattern.
// The values are computed at build time (silu_table.py, exact to 60 digits before the one
// rounding) and compiled in, so the table is in device memory as soon as the library loads:
// no launch fills it and nothing waits for it.
__device__ const uint32_t g_silu_bits[65536] = {
#include "silu_table.inc"
};

namespace {

constexpr int kStages = 3;
// The grouped GEMM kernel: producer A, MMA, 16 epilogue warps (four per TMEM lane quarter,
// each owning 64 accumulator columns), producer B.  19 warps put five on three of the SM's
// sub-partitions, so a thread gets at most 96 registers (5 x 32 x 96 <= 16384 per partition).
constexpr int kMainEpiWarps = 16;
constexpr int kMainEpiThreads = kMainEpiWarps * 32;
constexpr int kMainThreads = 96 + kMainEpiThreads;
constexpr int kMainProducerBWarp = 2 + kMainEpiWarps;
// The fused FC2 kernel's epilogue warps.
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;                         // bytes of K per row per stage (256 FP4 values)
constexpr int kMmaPerStage = kBKBytes / 32;           // K=64 MMAs per stage
// K-major operand tiles use the swizzle whose span equals the stage's row length
constexpr int kSwizzleBytes = kBKBytes;               // 128 or 64
constexpr int kABytes = kBM * kBKBytes;
constexpr int kBBytes = kBN * kBKBytes;
constexpr int kSfaOff = kABytes + kBBytes;            // kMmaPerStage scale tiles of A
constexpr int kSfbOff = kSfaOff + kMmaPerStage * kSfAtomBytes;   // 2 x kMmaPerStage scale tiles of B
constexpr int kStageBytes = kSfbOff + 2 * kMmaPerStage * kSfAtomBytes;
static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
constexpr int kEpiStageOff = kStages * kStageBytes;
// SiLU of the BF16 values with 2^-24 <= |a| < 2^7 (bit patterns 0x3380..0x42FF and their
// negatives): 7936 entries copied from the global table into shared memory per FC1 CTA.
// Outside that range silu has a closed form (silu_bf16), so no lookup leaves the SM.
constexpr uint32_t kSiluLo = 0x3380u, kSiluSpan = 0x4300u - 0x3380u;
constexpr int kBarrierBytes = 256;
// Shared-memory layout after the stages: the epilogue warps' column scales, the expert offsets
// and, for FC1, the SiLU range.
template <bool kFC1>
struct Smem {
    static constexpr int scale = kEpiStageOff;                                              // 64 floats per warp
    static constexpr int offsets = scale + kMainEpiWarps * 64 * 4;                          // up to 1025 ints
    static constexpr int silu = offsets + 4352;
    static constexpr int bar = silu + (kFC1 ? 2 * kSiluSpan * 4 : 0);
    static constexpr int bytes = bar + kBarrierBytes + 1024;
    static_assert(bytes <= 232448, "shared memory budget");
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;                     // per stage: SFA 4, SFB 8 columns per MMA
constexpr uint32_t kSfColsPerStage = 12 * kMmaPerStage;
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

// silu of the BF16 value with bit pattern `bits` (low 16 bits), as the FC1 epilogue applies it:
// from the shared-memory copy of the table for 2^-24 <= |a| < 2^7; a/2 below (the correctly
// rounded silu there, a*sigma(a) = a/2 + a^2/4 - ... differing from a/2 by under half an ulp;
// also +-0); a for a >= 2^7 and -0 for a <= -2^7 (e^-128 is far below the rounding); the
// global table for infinities and NaN.  Every value equals the table's (checked over all
// 65536 inputs by the tests through nvfp4_silu_table).
__device__ __noinline__ float silu_bf16_outside(uint32_t bits) {
    const uint32_t mag = bits & 0x7FFFu;
    const float a = __uint_as_float(bits << 16);
    if (mag < kSiluLo) return a * 0.5f;
    if (mag < 0x7F80u) return (bits >> 15) ? -0.0f : a;
    return __uint_as_float(__ldg(g_silu_bits + bits));
}
__device__ __forceinline__ float silu_bf16(uint32_t bits, const float* s_silu) {
    const uint32_t idx = (bits & 0x7FFFu) - kSiluLo;
    if (__builtin_expect(idx < kSiluSpan, 1)) return s_silu[idx + ((bits >> 15) ? kSiluSpan : 0u)];
    return silu_bf16_outside(bits);
}

// Copy the table's SiLU range into shared memory (2 * kSiluSpan floats).
__device__ __forceinline__ void load_silu_range(float* s_silu) {
    for (int i = threadIdx.x; i < 2 * static_cast<int>(kSiluSpan); i += blockDim.x) {
        const uint32_t bits = kSiluLo + (i % kSiluSpan) + (i >= static_cast<int>(kSiluSpan) ? 0x8000u : 0u);
        s_silu[i] = __uint_as_float(__ldg(g_silu_bits + bits));
    }
}

// Every BF16 input through silu_bf16, as the FC1 epilogue evaluates it (one block).
__global__ void __launch_bounds__(1024) silu_eval_kernel(float* out) {
    extern __shared__ float s_silu_eval[];
    load_silu_range(s_silu_eval);
    __syncthreads();
    for (int i = threadIdx.x; i < 65536; i += blockDim.x) out[i] = silu_bf16(static_cast<uint32_t>(i), s_silu_eval);
}

// Expert owning routed row `row`: largest e < E with off[e] <= row (off in shared memory).
__device__ __forceinline__ int expert_of_row(const int32_t* off, int E, int row) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= row) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Pairs of FP32 values in one 64-bit register (low = first) and their elementwise
// round-to-nearest products: each lane is exactly __fmul_rn of its two inputs.
__device__ __forceinline__ uint64_t f2(uint32_t lo_bits, uint32_t hi_bits) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// Elementwise maximum of two BF16 pairs (a NaN operand loses, as with fmaxf).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 64 BF16 values (packed[0..31], column pairs) of this lane's row at dst (32-byte aligned)
// as four 32-byte stores.
__device__ __forceinline__ void store_row_64(uint16_t* dst, const uint32_t (&packed)[32]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * k),
                     "r"(packed[8 * k]), "r"(packed[8 * k + 1]), "r"(packed[8 * k + 2]), "r"(packed[8 * k + 3]),
                     "r"(packed[8 * k + 4]), "r"(packed[8 * k + 5]), "r"(packed[8 * k + 6]), "r"(packed[8 * k + 7])
                     : "memory");
    }
}

// 32 BF16 values (packed[0..15], column pairs) of this lane's row at dst (32-byte aligned) as
// two 32-byte stores.
__device__ __forceinline__ void store_row_32(uint16_t* dst, const uint32_t (&packed)[16]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * k),
                     "r"(packed[8 * k]), "r"(packed[8 * k + 1]), "r"(packed[8 * k + 2]), "r"(packed[8 * k + 3]),
                     "r"(packed[8 * k + 4]), "r"(packed[8 * k + 5]), "r"(packed[8 * k + 6]), "r"(packed[8 * k + 7])
                     : "memory");
    }
}

// FC1 epilogue of one lane's row over the warp's 32 gate columns (acc[0]) and the matching 32
// up columns (acc[1]): gate/up = bf16((acc*g^x)*g^w) with the column scales sc[0..31] (gate)
// and sc[32..63] (up), h = bf16(f32(f32(silu(gate)*up)*p)) into packed[0..15]; returns the
// running max of |h| as a BF16 pair.  kDbg: also write the FP32 gate/up values to dbg
// (gate at dbg[j], up at dbg[I + j]).  kSave: also write the BF16 gate/up values to sv (gate
// at sv[j], up at sv[I + j]; one 4-byte store per pair of values: wider stores need registers
// for the pairs, and the epilogue is at its register limit).
template <bool kDbg, bool kSave>
__device__ __forceinline__ uint32_t fc1_rows(const uint32_t (&acc)[2][32], const float* sc, float gr, float p,
                                             const float* s_silu, float* dbg, uint16_t* sv, int I,
                                             uint32_t (&packed)[16]) {
    const uint64_t gr2 = f2(__float_as_uint(gr), __float_as_uint(gr));
    const uint64_t p2 = f2(__float_as_uint(p), __float_as_uint(p));
    uint32_t hmax2 = 0u;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const uint64_t vg2 = f2_mul(f2_mul(f2(acc[0][j], acc[0][j + 1]), gr2), *reinterpret_cast<const uint64_t*>(sc + j));
        const uint64_t vu2 =
            f2_mul(f2_mul(f2(acc[1][j], acc[1][j + 1]), gr2), *reinterpret_cast<const uint64_t*>(sc + 32 + j));
        float vg[2], vu[2];
        f2_unpack(vg2, vg[0], vg[1]);
        f2_unpack(vu2, vu[0], vu[1]);
        if (kDbg) {
            dbg[j] = vg[0];
            dbg[j + 1] = vg[1];
            dbg[I + j] = vu[0];
            dbg[I + j + 1] = vu[1];
        }
        const uint32_t gb = bf16x2_rn(vg[0], vg[1]), ub = bf16x2_rn(vu[0], vu[1]);
        if (kSave) {
            *reinterpret_cast<uint32_t*>(sv + j) = gb;
            *reinterpret_cast<uint32_t*>(sv + I + j) = ub;
        }
        const float sl0 = silu_bf16(gb & 0xFFFFu, s_silu), sl1 = silu_bf16(gb >> 16, s_silu);
        // silu(gate) * up in FP32, then * p, one BF16 rounding
        const uint64_t h2 =
            f2_mul(f2_mul(f2(__float_as_uint(sl0), __float_as_uint(sl1)), f2(ub << 16, ub & 0xFFFF0000u)), p2);
        float h[2];
        f2_unpack(h2, h[0], h[1]);
        packed[j >> 1] = bf16x2_rn(h[0], h[1]);
        hmax2 = bf16x2_max(hmax2, packed[j >> 1] & 0x7FFF7FFFu);
    }
    return hmax2;
}

// FC2 epilogue of one lane's row over 32 columns: y = bf16((acc*g2)*g^w2) with the column
// scales sc[0..31] into packed[0..15].  kDbg: also write the FP32 values to dbg[0..31].
template <bool kDbg>
__device__ __forceinline__ void fc2_cols(const uint32_t (&acc)[32], const float* sc, float gr, float* dbg,
                                         uint32_t (&packed)[16]) {
    const uint64_t gr2 = f2(__float_as_uint(gr), __float_as_uint(gr));
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const uint64_t v2 = f2_mul(f2_mul(f2(acc[j], acc[j + 1]), gr2), *reinterpret_cast<const uint64_t*>(sc + j));
        float v0, v1;
        f2_unpack(v2, v0, v1);
        if (kDbg) {
            dbg[j] = v0;
            dbg[j + 1] = v1;
        }
        packed[j >> 1] = bf16x2_rn(v0, v1);
    }
}

template <bool kFC1>
__global__ void __maxnreg__(96)
    grouped_gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = Smem<kFC1>;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bar);
    uint64_t* empty = full + kStages;
    uint64_t* tmem_full = empty + kStages;
    uint64_t* tmem_empty = tmem_full + 1;
    uint64_t* drain = tmem_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* scale_buf = reinterpret_cast<float*>(smem + L::scale);
    int32_t* s_off = reinterpret_cast<int32_t*>(smem + L::offsets);
    float* s_silu = reinterpret_cast<float*>(smem + L::silu);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 2);           // producer A and producer B
            mbar_init(&empty[s], 1);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, kMainEpiThreads);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // everything above touches only this CTA's shared memory and TMEM, and the SiLU table is
    // constant data of the library's image, so all of it overlaps the previous kernel's tail;
    // what earlier kernels write is read only after the wait
    if (kFC1) load_silu_range(s_silu);
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = __ldg(args.offsets + i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int E = args.E;
    const int num_m_tiles = s_off[E] / kBM;
    const int n_tiles = kFC1 ? args.I / 128 : args.H / kBN;
    const int num_tiles = num_m_tiles * n_tiles;
    const int num_k64 = args.K / 64;
    const int num_ks = (num_k64 + kMmaPerStage - 1) / kMmaPerStage;

    bool failed = false;

    // The producer and MMA warps run their loops with all 32 lanes in step (every value
    // warp-uniform, waits taken by all lanes and agreed with a vote); the TMA and tcgen05
    // instructions are issued by the lane elect.sync picks.
    if (warp == 0 || warp == kMainProducerBWarp) {
        // ------------------------------------------------------------ producers
        const bool is_a = warp == 0;
        const uint64_t pol = is_a ? policy_evict_last() : policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_parity = 0;
        for (int t = blockIdx.x; t < num_tiles && !failed; t += gridDim.x) {
            const int mt = t / n_tiles, nt = t % n_tiles;
            const int e = expert_of_row(s_off, E, mt * kBM);
            // first weight rows of the tile's two 128-row halves (their scale tiles)
            const int row0 = kFC1 ? e * args.Nw + nt * 128 : e * args.Nw + nt * kBN;
            const int row1 = kFC1 ? row0 + args.I : row0 + 128;
            for (int ks = 0; ks < num_ks; ++ks) {
                const bool ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, kWaitBudgetCycles);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    failed = true;
                    break;
                }
                const int nk = min(kMmaPerStage, num_k64 - kMmaPerStage * ks);
                const uint32_t sf_bytes = static_cast<uint32_t>(nk) * kSfAtomBytes;
                uint8_t* st = smem + stage * kStageBytes;
                if (is_a) {
                    mbar_arrive_expect_tx_elect(&full[stage], kABytes + sf_bytes);
                    tma_load_2d_elect(st, &tmA, &full[stage], ks * kBKBytes, mt * kBM, pol);
                    bulk_load_elect(st + kSfaOff,
                                    args.a_sf + (static_cast<int64_t>(mt) * num_k64 + kMmaPerStage * ks) * kSfAtomBytes,
                                    sf_bytes, &full[stage], pol);
                } else {
                    mbar_arrive_expect_tx_elect(&full[stage], kBBytes + 2 * sf_bytes);
                    if (kFC1) tma_load_4d_elect(st + kABytes, &tmB, &full[stage], ks * kBKBytes, nt * 128, 0, e, pol);
                    else tma_load_2d_elect(st + kABytes, &tmB, &full[stage], ks * kBKBytes, row0, pol);
                    bulk_load_elect(st + kSfbOff,
                                    args.b_sf + (static_cast<int64_t>(row0 / 128) * num_k64 + kMmaPerStage * ks) * kSfAtomBytes,
                                    sf_bytes, &full[stage], pol);
                    bulk_load_elect(st + kSfbOff + kMmaPerStage * kSfAtomBytes,
                                    args.b_sf + (static_cast<int64_t>(row1 / 128) * num_k64 + kMmaPerStage * ks) * kSfAtomBytes,
                                    sf_bytes, &full[stage], pol);
                }
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (failed) {
            if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            // let every copy still in flight land before the CTA's shared memory goes away
            // (a stage the other producer never filled runs out its bounded wait)
            for (int s = 0; s < kStages; ++s) {
                if (issued & (1u << s)) {
                    mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, kWaitBudgetCycles);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_nvf4(kBM, kBN);
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool issued_any = false;
        for (int t = blockIdx.x; t < num_tiles && !failed; t += gridDim.x) {
            const bool ok = mbar_wait_bounded(tmem_empty, acc_phase ^ 1u, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                failed = true;
                break;
            }
            acc_phase ^= 1u;
            tc_fence_after();
            for (int ks = 0; ks < num_ks; ++ks) {
                const bool okf = mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitBudgetCycles);
                if (!__all_sync(0xFFFFFFFFu, okf)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const int nk = min(kMmaPerStage, num_k64 - kMmaPerStage * ks);
                const uint32_t st = smem_u32(smem + stage * kStageBytes);
                const uint32_t sf_col = tmem + kSfCol0 + kSfColsPerStage * stage;
                const uint64_t adesc = sdesc_k_swizzled<kSwizzleBytes>(st);
                const uint64_t bdesc = sdesc_k_swizzled<kSwizzleBytes>(st + kABytes);
                if (kMmaPerStage == 4 && nk == 4) {   // a full stage: one issue block
                    tc_stage4_nvf4_elect(tmem, adesc, bdesc, idesc, sdesc_sf(st + kSfaOff), sdesc_sf(st + kSfbOff),
                                         sdesc_sf(st + kSfbOff + kMmaPerStage * kSfAtomBytes), sf_col, ks != 0 ? 1u : 0u);
                } else {
#pragma unroll
                for (int j = 0; j < kMmaPerStage; ++j) {
                    if (j < nk) {
                        tc_cp_32x128b_warpx4_elect(sf_col + 4 * j, sdesc_sf(st + kSfaOff + kSfAtomBytes * j));
                        tc_cp_32x128b_warpx4_elect(sf_col + 4 * kMmaPerStage + 8 * j,
                                                   sdesc_sf(st + kSfbOff + kSfAtomBytes * j));
                        tc_cp_32x128b_warpx4_elect(
                            sf_col + 4 * kMmaPerStage + 8 * j + 4,
                            sdesc_sf(st + kSfbOff + kMmaPerStage * kSfAtomBytes + kSfAtomBytes * j));
                        tc_mma_nvf4_elect(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sf_col + 4 * j,
                                          sf_col + 4 * kMmaPerStage + 8 * j, (ks | j) != 0 ? 1u : 0u);
                    }
                }
                }
                issued_any = true;
                tc_commit_elect(&empty[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (failed) break;
            tc_commit_elect(tmem_full);
        }
        if (failed) {
            if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            if (issued_any) {   // wait for the MMAs already issued before TMEM is released
                tc_commit_elect(drain);
                mbar_wait_bounded(drain, 0, nullptr, kWaitBudgetCycles);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;                             // 0..15
        const int q = warp & 3;                              // TMEM lane quarter of this warp
        const int sub = ew >> 2;                             // which quarter of the tile's columns
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        float* sc = scale_buf + ew * 64;                     // this warp's 64 column scales
        uint32_t acc_phase = 0;
        // this tile's row data and the weight scales of this warp's 64 columns (FC1: 32 gate
        // then the 32 matching up columns) are loaded one tile ahead, so their latency hides
        // behind the previous tile's epilogue
        int n_pair = -1;
        float n_gr = 0.0f, n_p = 0.0f, n_sc[2] = {0.0f, 0.0f};
        auto prefetch = [&](int tt) {
            const int mt_ = tt / n_tiles, nt_ = tt % n_tiles;
            const int e_ = expert_of_row(s_off, E, mt_ * kBM);
            const int64_t row_ = static_cast<int64_t>(mt_) * kBM + q * 32 + lane;
            n_pair = __ldg(args.row_pair + row_);
            n_gr = __ldg(args.a_g + row_);
            n_p = kFC1 ? __ldg(args.row_prob + row_) : 0.0f;
            const float* gw = args.b_g + static_cast<int64_t>(e_) * args.Nw;
            if (kFC1) {
                n_sc[0] = __ldg(gw + nt_ * 128 + 32 * sub + lane);
                n_sc[1] = __ldg(gw + args.I + nt_ * 128 + 32 * sub + lane);
            } else {
                n_sc[0] = __ldg(gw + nt_ * kBN + 64 * sub + lane);
                n_sc[1] = __ldg(gw + nt_ * kBN + 64 * sub + 32 + lane);
            }
        };
        if (static_cast<int>(blockIdx.x) < num_tiles) prefetch(blockIdx.x);
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const int mt = t / n_tiles, nt = t % n_tiles;
            const int64_t row = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
            const int pair = n_pair;
            const bool live = pair >= 0;
            const float gr = live ? n_gr : 0.0f;
            const float p = live ? n_p : 0.0f;
            __syncwarp();
            sc[lane] = n_sc[0];
            sc[lane + 32] = n_sc[1];
            __syncwarp();
            if (t + static_cast<int>(gridDim.x) < num_tiles) prefetch(t + gridDim.x);
            if (!mbar_wait_bounded(tmem_full, acc_phase, abort_flag, kWaitBudgetCycles)) {
                if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            acc_phase ^= 1u;
            tc_fence_after();
            // copy this warp's 64 accumulator columns to registers, then hand TMEM back
            uint32_t acc[2][32];
            if (kFC1) {
                tmem_ld_32x32b_x32(taddr + 32 * sub, acc[0]);          // gate columns
                tmem_ld_32x32b_x32(taddr + 128 + 32 * sub, acc[1]);    // the matching up columns
            } else {
                tmem_ld_32x32b_x32(taddr + 64 * sub, acc[0]);
                tmem_ld_32x32b_x32(taddr + 64 * sub + 32, acc[1]);
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(tmem_empty);

            if (kFC1) {
                const int I = args.I;
                float* dbg = args.debug && live ? args.debug + row * (2 * I) + nt * 128 + 32 * sub : nullptr;
                uint16_t* sv = args.gu_save && live ? args.gu_save + row * (2 * I) + nt * 128 + 32 * sub : nullptr;
                uint32_t packed[16];
                uint32_t hmax2;
                if (dbg) hmax2 = fc1_rows<true, false>(acc, sc, gr, p, s_silu, dbg, nullptr, I, packed);
                else if (sv) hmax2 = fc1_rows<false, true>(acc, sc, gr, p, s_silu, nullptr, sv, I, packed);
                else hmax2 = fc1_rows<false, false>(acc, sc, gr, p, s_silu, nullptr, nullptr, I, packed);
                const float hmax = __uint_as_float((bf16x2_max(hmax2, hmax2 >> 16) & 0xFFFFu) << 16);
                if (live) {
                    atomicMax(args.amax2 + row, __float_as_uint(hmax));
                    store_row_32(args.h + row * I + nt * 128 + 32 * sub, packed);
                }
            } else {
                const int H = args.H;
                float* dbg = args.debug && live ? args.debug + row * H + nt * kBN + 64 * sub : nullptr;
                uint16_t* yrow = live ? args.y + row * H + nt * kBN + 64 * sub : nullptr;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {            // two 32-column halves, 64 bytes of y each
                    uint32_t packed[16];
                    if (dbg) fc2_cols<true>(acc[c2], sc + 32 * c2, gr, dbg + 32 * c2, packed);
                    else fc2_cols<false>(acc[c2], sc + 32 * c2, gr, nullptr, packed);
                    if (live) store_row_32(yrow + 32 * c2, packed);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- FC2 with the requantisation fused
// The FC2 input h is requantised inside the FC2 kernel, so the requantised operand never goes
// through memory ("miniTE diagnoses and narrows the cross-engine execution gap of NVFP4 RL",
// section "Assumptions and limits": online amax-quantisation-GEMM fusion).  FC2's A operand of
// one m-tile (its 128 routed rows, all I columns) is quantised once into shared memory, in the
// K-major 128B-swizzled layout a TMA load would give, with its block scales in the 512-byte
// scale-tile layout and its outer scales g2 = amax2 / 2688 taken from the maxima FC1 reduced;
// it then stays resident while the W2 tiles of the unit's n-tiles stream through a 2-stage
// ring.  The quantiser is the one the requant kernel runs (nvfp4_quant.cuh) and the MMA walks
// K in the same order over the same codes and scales, so y is bitwise what the staged
// requant + FC2 give.
//
// Work unit: (m-tile, group of n-tiles); the number of groups per m-tile is chosen on the
// device from the number of m-tiles so that the units spread over the SMs with a short tail.
// Warp roles (16 warps, four per SM sub-partition at 128 registers each, which fills its
// 16K-register file): warp 0 loads W2 tiles (TMA), warp 1 issues the MMAs, warps 2-9 run the
// epilogue (reading the accumulator in two halves of 64 columns, so that it fits, and storing
// each lane's row with 32-byte stores), warp 10 copies h into shared memory in chunks of
// consecutive rows (cp.async.bulk, two slots) together with each unit's row map and maxima,
// and warps 11-15 quantise from there into the other of two A buffers, one unit ahead of the
// MMAs.  Fits I <= 768 and E <= 512 (two 54 KB A buffers, two 36 KB W2 stages, two 18 KB h
// slots).
namespace fused {
constexpr int kMaxI = 768;
constexpr int kMaxE = 512;
constexpr int kStagesB = 2;
constexpr int kHWarp = 2 + kEpiWarps;                              // 10
constexpr int kQuantWarp0 = kHWarp + 1;                           // 11
constexpr int kQuantWarps = 5;
constexpr int kThreadsF = 32 * (kQuantWarp0 + kQuantWarps);       // 512
constexpr int kABlockBytes = kBM * kBKBytes;                      // one K=256 block of 128 rows: 16 KB
constexpr int kACodesBytes = (kMaxI / 256) * kABlockBytes;        // 48 KB
constexpr int kASfBytes = (kMaxI / 64) * kSfAtomBytes;            // 6 KB
constexpr int kABufBytes = kACodesBytes + kASfBytes;
static_assert(kABufBytes % 1024 == 0, "A buffers keep 1024-byte alignment");
constexpr int kBStageBytes = kBBytes + 2 * kMmaPerStage * kSfAtomBytes;
constexpr int kHSlotBytes = 12 * 2 * kMaxI;                       // 12 rows of h at I = 768
constexpr int kBOff = 2 * kABufBytes;
constexpr int kHOff = kBOff + kStagesB * kBStageBytes;
constexpr int kRowDataOff = kHOff + 2 * kHSlotBytes;              // per A buffer: pair[128], amax2[128]
constexpr int kScaleOffF = kRowDataOff + 2 * 2 * 128 * 4;
constexpr int kG2Off = kScaleOffF + kEpiWarps * 128 * 4;          // per A buffer: g2[128]
constexpr int kOffsetsOffF = kG2Off + 2 * 128 * 4;
constexpr int kBarOffF = kOffsetsOffF + (kMaxE + 64) * 4;
constexpr int kSmemBytesF = kBarOffF + kBarrierBytes + 1024;
static_assert(kSmemBytesF <= 232448, "shared memory budget");
constexpr uint32_t kSfColsPerStageF = 12 * kMmaPerStage;
static_assert(kSfCol0 + kStagesB * kSfColsPerStageF <= kTmemCols, "TMEM budget");

// Work units of one launch: n-tile groups per m-tile, the smallest estimated makespan
// (rounds of units over the grid, each unit costing its n-tiles plus one).
struct Units {
    int groups, per, count;
    __device__ Units(int num_m, int n_tiles, int grid) {
        groups = 1;
        long long best = -1;
        for (int g = 1; g <= n_tiles && n_tiles % g == 0; g *= 2) {
            const long long rounds = (static_cast<long long>(num_m) * g + grid - 1) / grid;
            const long long cost = rounds * (n_tiles / g + 1);
            if (best < 0 || cost < best) {
                best = cost;
                groups = g;
            }
            if (g > n_tiles / 2) break;
        }
        per = n_tiles / groups;
        count = num_m * groups;
    }
};

// Rows of h per staging slot: every quantiser warp's rows of one pass, capped by the slot.
__device__ __forceinline__ int rows_per_chunk(int I) {
    const int G = I / 64;
    const int rpw = G <= 32 ? 32 / G : 1;
    return min(kQuantWarps * rpw, kHSlotBytes / (2 * I));
}

__global__ void __launch_bounds__(kThreadsF, 1)
    fc2_requant_kernel(const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffF);
    uint64_t* empty = full + kStagesB;
    uint64_t* a_full = empty + kStagesB;          // [2]: quantisers -> MMA and epilogue
    uint64_t* a_empty = a_full + 2;               // [2]: MMA (a unit's MMAs done) + epilogue (its g2 read) -> quantisers
    uint64_t* h_full = a_empty + 2;               // [2]: h chunk (and, with a unit's first chunk, its row data) landed
    uint64_t* h_empty = h_full + 2;               // [2]: quantisers done with the slot
    uint64_t* tmem_full = h_empty + 2;
    uint64_t* tmem_empty = tmem_full + 1;
    uint64_t* drain = tmem_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* scale_buf = reinterpret_cast<float*>(smem + kScaleOffF);
    int32_t* s_off = reinterpret_cast<int32_t*>(smem + kOffsetsOffF);
    float* g2_s = reinterpret_cast<float*>(smem + kG2Off);                  // [2][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesB; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&a_full[b], 32 * kQuantWarps);
            mbar_init(&a_empty[b], 1 + kEpiThreads);
            mbar_init(&h_full[b], 1);
            mbar_init(&h_empty[b], 32 * kQuantWarps);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, kEpiThreads);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) prefetch_tensormap(&tmB);
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = __ldg(args.offsets + i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int E = args.E;
    const int num_m = s_off[E] / kBM;
    const int n_tiles = args.H / kBN;
    const Units U(num_m, n_tiles, gridDim.x);
    const int num_k64 = args.I / 64;
    const int num_ks = (num_k64 + kMmaPerStage - 1) / kMmaPerStage;
    const int rpc = rows_per_chunk(args.I);
    const int nchunks = (kBM + rpc - 1) / rpc;
    bool failed = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer of B (W2 tiles)
        const uint64_t pol = policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_parity = 0;
        for (int u = blockIdx.x; u < U.count && !failed; u += gridDim.x) {
            const int mt = u / U.groups, nt0 = (u % U.groups) * U.per;
            const int e = expert_of_row(s_off, E, mt * kBM);
            for (int nt = nt0; nt < nt0 + U.per && !failed; ++nt) {
                const int row0 = e * args.Nw + nt * kBN;
                for (int ks = 0; ks < num_ks; ++ks) {
                    const bool ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, kWaitBudgetCycles);
                    if (!__all_sync(0xFFFFFFFFu, ok)) {
                        failed = true;
                        break;
                    }
                    const int nk = min(kMmaPerStage, num_k64 - kMmaPerStage * ks);
                    const uint32_t sf_bytes = static_cast<uint32_t>(nk) * kSfAtomBytes;
                    uint8_t* st = smem + kBOff + stage * kBStageBytes;
                    mbar_arrive_expect_tx_elect(&full[stage], kBBytes + 2 * sf_bytes);
                    tma_load_2d_elect(st, &tmB, &full[stage], ks * kBKBytes, row0, pol);
                    bulk_load_elect(st + kBBytes,
                                    args.b_sf + (static_cast<int64_t>(row0 / 128) * num_k64 + kMmaPerStage * ks) * kSfAtomBytes,
                                    sf_bytes, &full[stage], pol);
                    bulk_load_elect(st + kBBytes + kMmaPerStage * kSfAtomBytes,
                                    args.b_sf + (static_cast<int64_t>(row0 / 128 + 1) * num_k64 + kMmaPerStage * ks) * kSfAtomBytes,
                                    sf_bytes, &full[stage], pol);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStagesB) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (failed) {
            if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            for (int s = 0; s < kStagesB; ++s) {
                if (issued & (1u << s)) mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, kWaitBudgetCycles);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_nvf4(kBM, kBN);
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool issued_any = false;
        int local = 0;
        for (int u = blockIdx.x; u < U.count && !failed; u += gridDim.x, ++local) {
            const int ab = local & 1;
            const bool oka = mbar_wait_bounded(&a_full[ab], (local >> 1) & 1, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, oka)) {
                failed = true;
                break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + ab * kABufBytes);
            const uint32_t a_sf = a_base + kACodesBytes;
            for (int j = 0; j < U.per && !failed; ++j) {
                const bool ok = mbar_wait_bounded(tmem_empty, acc_phase ^ 1u, abort_flag, kWaitBudgetCycles);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    failed = true;
                    break;
                }
                acc_phase ^= 1u;
                tc_fence_after();
                for (int ks = 0; ks < num_ks; ++ks) {
                    const bool okf = mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitBudgetCycles);
                    if (!__all_sync(0xFFFFFFFFu, okf)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(kMmaPerStage, num_k64 - kMmaPerStage * ks);
                    const uint32_t st = smem_u32(smem + kBOff + stage * kBStageBytes);
                    const uint32_t sf_col = tmem + kSfCol0 + kSfColsPerStageF * stage;
                    const uint64_t adesc = sdesc_k_swizzled<kSwizzleBytes>(a_base + ks * kABlockBytes);
                    const uint64_t bdesc = sdesc_k_swizzled<kSwizzleBytes>(st);
                    const uint32_t sfa = a_sf + kMmaPerStage * ks * kSfAtomBytes;
                    const uint32_t sfb = st + kBBytes;
                    if (kMmaPerStage == 4 && nk == 4) {
                        tc_stage4_nvf4_elect(tmem, adesc, bdesc, idesc, sdesc_sf(sfa), sdesc_sf(sfb),
                                             sdesc_sf(sfb + kMmaPerStage * kSfAtomBytes), sf_col, ks != 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int jj = 0; jj < kMmaPerStage; ++jj) {
                            if (jj < nk) {
                                tc_cp_32x128b_warpx4_elect(sf_col + 4 * jj, sdesc_sf(sfa + kSfAtomBytes * jj));
                                tc_cp_32x128b_warpx4_elect(sf_col + 4 * kMmaPerStage + 8 * jj,
                                                           sdesc_sf(sfb + kSfAtomBytes * jj));
                                tc_cp_32x128b_warpx4_elect(sf_col + 4 * kMmaPerStage + 8 * jj + 4,
                                                           sdesc_sf(sfb + kMmaPerStage * kSfAtomBytes + kSfAtomBytes * jj));
                                tc_mma_nvf4_elect(tmem, adesc + 2 * jj, bdesc + 2 * jj, idesc, sf_col + 4 * jj,
                                                  sf_col + 4 * kMmaPerStage + 8 * jj, (ks | jj) != 0 ? 1u : 0u);
                            }
                        }
                    }
                    issued_any = true;
                    tc_commit_elect(&empty[stage]);
                    if (++stage == kStagesB) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (failed) break;
                tc_commit_elect(tmem_full);
            }
            if (failed) break;
            tc_commit_elect(&a_empty[ab]);        // this unit's A is free once its MMAs are done
        }
        if (failed) {
            if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            if (issued_any) {
                tc_commit_elect(drain);
                mbar_wait_bounded(drain, 0, nullptr, kWaitBudgetCycles);
            }
        }
    } else if (warp == kHWarp) {
        // ------------------------------------------------------------ producer of h chunks
        // Rows [c*rpc, c*rpc + rpc) of each unit's m-tile are consecutive in h: one bulk copy
        // per chunk.  A unit's first chunk also brings its 128 row-map entries and maxima.
        const uint64_t pol = policy_evict_first();   // last use of h
        int gc = 0;                                  // chunks issued so far (slot gc & 1)
        uint32_t issued = 0, issued_parity = 0;
        int local = 0;
        for (int u = blockIdx.x; u < U.count && !failed; u += gridDim.x, ++local) {
            const int mt = u / U.groups;
            const int ab = local & 1;
            const int64_t row0 = static_cast<int64_t>(mt) * kBM;
            for (int c = 0; c < nchunks; ++c, ++gc) {
                const int slot = gc & 1;
                const bool ok = mbar_wait_bounded(&h_empty[slot], ((gc >> 1) & 1) ^ 1u, abort_flag, kWaitBudgetCycles);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    failed = true;
                    break;
                }
                const int r0 = c * rpc, nr = min(rpc, kBM - r0);
                const uint32_t hbytes = static_cast<uint32_t>(nr) * 2 * args.I;
                uint8_t* rd = smem + kRowDataOff + ab * 1024;
                mbar_arrive_expect_tx_elect(&h_full[slot], hbytes + (c == 0 ? 1024u : 0u));
                bulk_load_elect(smem + kHOff + slot * kHSlotBytes, args.h + (row0 + r0) * args.I, hbytes, &h_full[slot],
                                pol);
                if (c == 0) {
                    bulk_load_elect(rd, args.row_pair + row0, 512, &h_full[slot], pol);
                    bulk_load_elect(rd + 512, args.amax2 + row0, 512, &h_full[slot], pol);
                }
                issued |= 1u << slot;
                issued_parity = (issued_parity & ~(1u << slot)) | (static_cast<uint32_t>((gc >> 1) & 1) << slot);
            }
        }
        if (failed) {
            if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            for (int s = 0; s < 2; ++s) {
                if (issued & (1u << s)) mbar_wait_bounded(&h_full[s], (issued_parity >> s) & 1u, nullptr, kWaitBudgetCycles);
            }
        }
    } else if (warp >= kQuantWarp0) {
        // ------------------------------------------------------------ A quantisers
        const int qw = warp - kQuantWarp0;
        const int G = args.I / 64;
        const RowLanes rl(G);
        int gc = 0;
        int local = 0;
        bool stop = false;
        for (int u = blockIdx.x; u < U.count && !stop; u += gridDim.x, ++local) {
            const int ab = local & 1;
            if (local >= 2) {   // the unit that last used this buffer: its MMAs done, its g2 read
                if (!mbar_wait_bounded(&a_empty[ab], ((local - 2) >> 1) & 1, abort_flag, kWaitBudgetCycles)) {
                    if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
            uint8_t* abuf = smem + ab * kABufBytes;
            float* g2b = g2_s + ab * 128;
            const int32_t* rpair = reinterpret_cast<const int32_t*>(smem + kRowDataOff + ab * 1024);
            const uint32_t* ramax = reinterpret_cast<const uint32_t*>(smem + kRowDataOff + ab * 1024 + 512);
            for (int c = 0; c < nchunks; ++c, ++gc) {
                const int slot = gc & 1;
                if (!mbar_wait_bounded(&h_full[slot], (gc >> 1) & 1, abort_flag, kWaitBudgetCycles)) {
                    if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    stop = true;
                    break;
                }
                const int r0 = c * rpc, nr = min(rpc, kBM - r0);
                const int rr = qw * rl.RPW + rl.slot;            // this lane's row within the chunk
                const bool row_ok = rl.active && rr < nr;
                const int r = r0 + rr;
                const int32_t pair = row_ok ? rpair[r] : -1;
                const uint32_t amax_bits = row_ok ? ramax[r] : 0u;
                uint4 v[1][8];
                if (pair >= 0) {
                    const uint4* src = reinterpret_cast<const uint4*>(smem + kHOff + slot * kHSlotBytes +
                                                                      static_cast<int64_t>(rr) * 2 * args.I + rl.li * 128);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[0][i] = src[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[0][i] = make_uint4(0u, 0u, 0u, 0u);
                }
                // the slot's data is in registers; the next bulk copy into the slot (async proxy)
                // must not overtake these generic-proxy reads
                fence_proxy_async_shared();
                mbar_arrive(&h_empty[slot]);
                if (rl.active) {
                    GroupQ q[1];
                    bool finite = true;
                    float gr = quantize_loaded<1>(v, rl, G, __uint_as_float(amax_bits), q, finite);
                    if (row_ok) {
                        if (pair < 0) {
                            q[0].sfw = 0u;
                            gr = 0.0f;
                        } else if (!finite && rl.li == 0) {
                            set_device_error(args.err, NVFP4_ERR_NONFINITE);
                        }
                        const int grp = rl.li;
                        uint8_t* rowp = abuf + (grp >> 2) * kABlockBytes + r * kBKBytes;
                        const int c0 = 2 * (grp & 3);
                        *reinterpret_cast<uint4*>(rowp + ((c0 ^ (r & 7)) << 4)) =
                            make_uint4(q[0].code[0], q[0].code[1], q[0].code[2], q[0].code[3]);
                        *reinterpret_cast<uint4*>(rowp + (((c0 + 1) ^ (r & 7)) << 4)) =
                            make_uint4(q[0].code[4], q[0].code[5], q[0].code[6], q[0].code[7]);
                        *reinterpret_cast<uint32_t*>(abuf + kACodesBytes + grp * kSfAtomBytes + (r & 31) * 16 +
                                                     (r >> 5) * 4) = q[0].sfw;
                        if (rl.li == 0) g2b[r] = gr;
                    }
                }
            }
            if (stop) break;
            fence_proxy_async_shared();
            mbar_arrive(&a_full[ab]);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;                             // 0..7
        const int q = warp & 3;                              // TMEM lane quarter of this warp
        const int half = ew >> 2;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        float* sc = scale_buf + ew * 128;
        const int H = args.H;
        const int row = q * 32 + lane;
        uint32_t acc_phase = 0;
        int local = 0;
        // the W2 column scales of this warp's 128 columns, loaded one tile ahead
        float n_sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        auto prefetch_sc = [&](int uu, int jj) {
            const int mt_ = uu / U.groups;
            const int nt_ = (uu % U.groups) * U.per + jj;
            const int e_ = expert_of_row(s_off, E, mt_ * kBM);
            const float* gw = args.b_g + static_cast<int64_t>(e_) * args.Nw + nt_ * kBN + 128 * half;
#pragma unroll
            for (int i = 0; i < 4; ++i) n_sc[i] = __ldg(gw + lane + 32 * i);
        };
        if (static_cast<int>(blockIdx.x) < U.count) prefetch_sc(blockIdx.x, 0);
        bool stop = false;
        for (int u = blockIdx.x; u < U.count && !stop; u += gridDim.x, ++local) {
            const int ab = local & 1;
            const int mt = u / U.groups, nt0 = (u % U.groups) * U.per;
            // this unit's outer scales g2: written by the quantisers before they arrived on a_full
            if (!mbar_wait_bounded(&a_full[ab], (local >> 1) & 1, abort_flag, kWaitBudgetCycles)) {
                if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            const int pair = __ldg(args.row_pair + static_cast<int64_t>(mt) * kBM + row);
            const bool live = pair >= 0;
            const float gr = live ? g2_s[ab * 128 + row] : 0.0f;
            mbar_arrive(&a_empty[ab]);                       // g2 read: the buffer may be refilled
            const uint64_t gr2 = f2(__float_as_uint(gr), __float_as_uint(gr));
            for (int j = 0; j < U.per; ++j) {
                const int nt = nt0 + j;
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[lane + 32 * i] = n_sc[i];
                __syncwarp();
                if (j + 1 < U.per) prefetch_sc(u, j + 1);
                else if (u + static_cast<int>(gridDim.x) < U.count) prefetch_sc(u + gridDim.x, 0);
                if (!mbar_wait_bounded(tmem_full, acc_phase, abort_flag, kWaitBudgetCycles)) {
                    if (lane == 0) set_device_error(args.err, NVFP4_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    stop = true;
                    break;
                }
                acc_phase ^= 1u;
                tc_fence_after();
                const int64_t grow = static_cast<int64_t>(mt) * kBM + row;
                float* dbg = args.debug ? args.debug + grow * H + nt * kBN + 128 * half : nullptr;
                uint16_t* yrow = live ? args.y + grow * H + nt * kBN + 128 * half : nullptr;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    // 64 of the warp's 128 accumulator columns at a time; TMEM goes back after the
                    // second half is in registers
                    uint32_t acc[2][32];
                    tmem_ld_32x32b_x32(taddr + 128 * half + 64 * c2, acc[0]);
                    tmem_ld_32x32b_x32(taddr + 128 * half + 64 * c2 + 32, acc[1]);
                    tmem_ld_wait();
                    if (c2 == 1) {
                        tc_fence_before();
                        mbar_arrive(tmem_empty);
                    }
                    uint32_t packed[32];
#pragma unroll
                    for (int jj = 0; jj < 64; jj += 2) {
                        const int c = 64 * c2 + jj;
                        const uint64_t v2 = f2_mul(f2_mul(f2(acc[jj >> 5][jj & 31], acc[jj >> 5][(jj & 31) + 1]), gr2),
                                                   *reinterpret_cast<const uint64_t*>(sc + c));
                        float v0, v1;
                        f2_unpack(v2, v0, v1);
                        if (dbg && live) {
                            dbg[c] = v0;
                            dbg[c + 1] = v1;
                        }
                        packed[jj >> 1] = bf16x2_rn(v0, v1);
                    }
                    if (live) store_row_64(yrow + 64 * c2, packed);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}
}  // namespace fused

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<EncodeTiledFn>(p);
        }
    });
    return fn;
}

constexpr CUtensorMapSwizzle kSwizzleMode =
    kSwizzleBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;

// 2D map over an NVFP4 code matrix [rows][row_bytes]: boxes of box_rows rows x kBKBytes,
// swizzled with the same span (the K-major canonical layout the MMA descriptors describe).
bool make_code_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, kSwizzleMode, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4D map over the FC1 weight codes [E][2][I][row_bytes] (gate rows, then up rows, per
// expert): a box is 128 gate rows and the 128 up rows of the same columns, so one copy
// lands them as 256 consecutive 128-byte rows (gate first), as two 2D boxes would.
bool make_gateup_map(CUtensorMap* m, const void* base, int E, int I, int64_t row_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(I), 2,
                                static_cast<cuuint64_t>(E)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(I * row_bytes),
                                   static_cast<cuuint64_t>(2 * I * row_bytes)};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(kBKBytes), 128, 2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, kSwizzleMode, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
std::mutex g_init_mutex;
bool g_attr_ready[kMaxDevices][3];

// Host-side set-up of the kernel attributes, once per device (no launch, no synchronisation).
// which: 0 FC1, 1 FC2, 2 FC2 with the requantisation fused.
cudaError_t prepare_device(int which) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_init_mutex);
    if (!g_attr_ready[dev][which]) {
        e = which == 0 ? cudaFuncSetAttribute(grouped_gemm_nvf4_kernel<true>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<true>::bytes)
            : which == 1 ? cudaFuncSetAttribute(grouped_gemm_nvf4_kernel<false>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<false>::bytes)
                         : cudaFuncSetAttribute(fused::fc2_requant_kernel,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, fused::kSmemBytesF);
        if (e != cudaSuccess) return e;
        g_attr_ready[dev][which] = true;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm(bool fc1, const GemmArgs& a, cudaStream_t st, bool pdl) {
    cudaError_t e = prepare_device(fc1 ? 0 : 1);
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;
    if (!make_code_map(&ma, a.a_codes, a.rows_cap, a.K / 2, kBM)) return cudaErrorInvalidValue;
    if (fc1 ? !make_gateup_map(&mb, a.b_codes, a.E, a.I, a.K / 2)
            : !make_code_map(&mb, a.b_codes, static_cast<int64_t>(a.E) * a.Nw, a.K / 2, kBN))
        return cudaErrorInvalidValue;
    const int grid = device_sm_count();
    if (fc1)
        return launch_pdl(pdl, grouped_gemm_nvf4_kernel<true>, grid, kMainThreads, Smem<true>::bytes, st, ma, mb, a);
    return launch_pdl(pdl, grouped_gemm_nvf4_kernel<false>, grid, kMainThreads, Smem<false>::bytes, st, ma, mb, a);
}

cudaError_t launch_fc2_requant_impl(const GemmArgs& a, cudaStream_t st, bool pdl) {
    if (a.I > fused::kMaxI || a.I % 128 != 0 || a.E > fused::kMaxE) return cudaErrorInvalidValue;
    cudaError_t e = prepare_device(2);
    if (e != cudaSuccess) return e;
    CUtensorMap mb;
    if (!make_code_map(&mb, a.b_codes, static_cast<int64_t>(a.E) * a.Nw, a.K / 2, kBN)) return cudaErrorInvalidValue;
    return launch_pdl(pdl, fused::fc2_requant_kernel, device_sm_count(), fused::kThreadsF, fused::kSmemBytesF, st, mb,
                      a);
}

}  // namespace

cudaError_t launch_fc2_requant(const GemmArgs& a, cudaStream_t st, bool pdl) {
    return launch_fc2_requant_impl(a, st, pdl);
}
int fc2_requant_max_i() { return fused::kMaxI; }
int fc2_requant_max_e() { return fused::kMaxE; }

cudaError_t launch_fc1(const GemmArgs& a, cudaStream_t st, bool pdl) { return launch_gemm(true, a, st, pdl); }
cudaError_t launch_fc2(const GemmArgs& a, cudaStream_t st, bool pdl) { return launch_gemm(false, a, st, pdl); }

cudaError_t copy_silu_table(float* out, cudaStream_t st) {
    const size_t smem = 2 * kSiluSpan * sizeof(float);
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [smem] {
        attr = cudaFuncSetAttribute(silu_eval_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    if (attr != cudaSuccess) return attr;
    silu_eval_kernel<<<1, 1024, smem, st>>>(out);
    return cudaGetLastError();
}

}  // namespace nvfp4
