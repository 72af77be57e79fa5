// Straight-through (STE) backward of the NVFP4 MoE expert layer: BF16 grouped GEMMs on the
// 5th-generation tensor cores over the saved BF16 originals, the SwiGLU x prob derivative in
// FP32, and the slot-order sum of the activation gradient.
//
// "miniTE diagnoses and narrows the cross-engine execution gap of NVFP4 RL"
// (onedev.kr/papers/1404), section "How it differs": the backward is a straight-through
// approximation that runs BF16 GEMMs on the saved original BF16 activations and weights, so
// no quantisation runs backward; its results paragraph scores the gradients by relative L2
// against an FP32 reference.
//
// For the routed rows r of expert e (the forward's expert-contiguous layout; pair(r) =
// token*k + slot, t(r) its token, p(r) its router probability):
//   dY rows    dy[r] = dOut[t(r)]                                        (gather)
//   FC2 dgrad  dh[r] = bf16( dy[r] W2[e] )                  BF16 GEMM, FP32 accumulation
//   SwiGLU     a, u = the forward's BF16 gate/up of r (saved by FC1; the values SwiGLU ran on),
//              s = 1/(1+exp(-a)):  da = bf16(dh*p*u*s*(1+a*(1-s))),  du = bf16(dh*p*a*s),
//              dprob[pair(r)] = sum_i dh_i*(a_i*s_i)*u_i               (FP32)
//   FC1 dgrad  dxs[pair(r)] = bf16( [da, du] W1[e] )        BF16 GEMM
//   combine    dX[t] = bf16( sum over slots 0..k-1 in order of dxs, FP32 )
//   FC2 wgrad  dW2[e] = sum_r dy[r]^T h[r]                  FP32 output
//   FC1 wgrad  dW1[e] = sum_r [da, du][r]^T x[t(r)]         FP32 output
//
// The GEMMs read every operand where it lies, without transposed copies: an operand whose
// reduction index K runs along its rows (the weights W1[e] [2I][H] and W2[e] [H][I] in the
// activation gradients; dy, h, [da, du] and the gathered x in the weight gradients, whose K is
// the expert's routed rows) is loaded as 64-row x 128-byte TMA boxes (128B swizzle) and handed
// to tcgen05.mma.kind::f16 through MN-major shared-memory descriptors; dy and [da, du] in the
// activation gradients are K-major as stored.  One persistent CTA per SM walks a static tile
// list: warp 0 issues the TMA loads into a stage ring (four stages for the activation
// gradients, three for the weight gradients), warp 1 the MMAs (M=128, N=128 or 256) into one
// of two TMEM accumulators, and warps 2-9 read the other accumulator (two warps per TMEM lane
// quarter, each half of the columns) and store it through a small shared-memory tile as whole
// row segments, so a tile's stores overlap the next tile's loads and MMAs.  Each tile walks K
// in one fixed order, so a token's dX and dprob do not depend on the other tokens.
//
// Pad rows: the forward's h holds whatever was there before in an expert's pad rows (FC1 does
// not store them), so the weight gradients stop at each expert's last real row (found once per
// call from the row map): stages past it are not loaded, and the rows past it in the last
// stage are zeroed in shared memory before the MMAs read them.
#include <algorithm>
#include <mutex>

#include "backward.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kBM = 128;                                // output rows per tile
constexpr int kBK = 64;                                 // BF16 elements of K per stage
constexpr int kBRowBytes = 2 * kBK;                     // 128 bytes, one swizzle span
constexpr int kBMaxN = 256;
constexpr int kBABytes = kBM * kBRowBytes;              // 16 KB
constexpr int kBBBytes = kBMaxN * kBRowBytes;           // 32 KB
constexpr int kBStageBytes = kBABytes + kBBBytes;       // 48 KB
constexpr int kBMnBox = kBK * kBRowBytes;               // 8 KB: 64 K-rows x 64 MN elements
constexpr int kBEpiWarps = 8;
constexpr int kBThreads = 64 + 32 * kBEpiWarps;         // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr uint32_t kBTmemCols = 2 * kBMaxN;             // two accumulators
constexpr int kBMaxE = 1024;

// Shared memory of one instantiation: a ring of kStages operand stages, the barriers, the
// expert offsets (and ends of real rows), and the epilogue staging.  Each epilogue warp passes
// its 32 accumulator rows through a tile of 32 rows x kStgWords 32-bit words (FP32 columns, or
// BF16 column pairs), 16-byte slots swizzled by row so that neither the row-wise writes nor the
// column-wise reads conflict, and stores it as whole kStgWords*4-byte row segments.  The
// activation gradients (24-32 K stages per tile) keep four stages; the weight gradients (a few
// K stages per tile, FP32 output) trade one for wider row segments.
template <bool kWgrad>
struct BCfg {
    static constexpr int kStages = kWgrad ? 3 : 4;
    static constexpr int kStgWords = kWgrad ? 32 : 16;
    static constexpr int kStgSlots = kStgWords / 4;              // 16-byte slots per staged row
    static constexpr int kStgShift = kStgSlots == 8 ? 0 : 1;     // rows sharing a bank group differ here
    static constexpr int kStgRowsPerSt = 32 / kStgSlots;         // rows one warp-wide 16-byte store covers
    static constexpr int kStgBytes = 32 * kStgWords * 4;         // per epilogue warp
    static constexpr int kBarOff = kStages * kBStageBytes;
    static constexpr int kOffOff = kBarOff + 256;                // offsets[0..E] then real_end[0..E)
    static constexpr int kStgOff = kOffOff + ((2 * (kBMaxE + 1) * 4 + 127) & ~127);
    static constexpr int kSmemBytes = kStgOff + kBEpiWarps * kStgBytes + 1024;
    static_assert(kStgWords == 16 || kStgWords == 32, "staged row chunk");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

enum : int { kModeRows = 0, kModePairs = 1, kModeWgrad = 2 };

// One launch of the grouped GEMM D = A B (FP32 accumulation), K in 64-wide stages.
//  kModeRows  (dgrad): tile (m, n) -> routed rows m*128.. of expert e (the one owning them);
//             A = routed rows [rows_cap][K] (K-major), B = weight rows e*K + k, columns n0..
//             ([E*K][N], MN-major); out_bf16[row][n], row stride N.
//  kModePairs (dgrad): as kModeRows, but row r goes to out_bf16[row_pair[r]][n] (pad rows are
//             not stored).
//  kModeWgrad: tile (e, m, n) -> K over expert e's routed rows offsets[e] .. real_end[e];
//             A = [rows_cap][M] columns m0.. (MN-major), B = [rows_cap][N] columns n0..
//             (MN-major); out_f32[e][m][n] (an expert without rows gets zeros).
struct BgemmJob {
    int mode;
    int BN;             // 128 or 256
    int n_tiles;        // N / BN
    int m_tiles;        // dgrad: rows_cap / 128; wgrad: M / 128
    int N;              // output columns
    int M;              // wgrad: output rows per expert
    int num_ks;         // dgrad: K / 64
    int K;              // dgrad: weight rows per expert
    int E;
    const int32_t* offsets;
    const int32_t* real_end;   // wgrad: end of each expert's real rows
    const int32_t* row_pair;
    uint16_t* out_bf16;
    float* out_f32;
    int* err;
};

// Instruction descriptor of tcgen05.mma kind::f16: BF16 A and B, FP32 accumulator; a_mn / b_mn
// select MN-major ("transposed") operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                                  // D format: F32
           | (1u << 7)                                // A format: BF16
           | (1u << 10)                               // B format: BF16
           | (a_mn ? 1u << 15 : 0u)                   // A major-ness
           | (b_mn ? 1u << 16 : 0u)                   // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Shared-memory descriptor of an MN-major BF16 operand laid out as consecutive 8 KB TMA boxes
// (each 64 K-rows of 128 bytes = 64 MN elements, 128B swizzle): 8-row groups along K are
// 1024 bytes apart (stride byte offset), 64-element blocks along MN one box (8 KB) apart
// (leading byte offset).  Base 1024-byte aligned; a K step of 16 rows advances it 2048 bytes.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);        // start address >> 4
    d |= static_cast<uint64_t>(kBMnBox >> 4) << 16;              // leading byte offset: next MN block
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride byte offset: next 8 K-rows
    d |= static_cast<uint64_t>(1) << 46;                         // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                         // 128B swizzle
    return d;
}

// D(tmem, FP32) (+)= A(smem, BF16) x B(smem, BF16), M=128, K=16, issued by the lane
// elect.sync picks while the whole warp executes it in step.
__device__ __forceinline__ void mma_bf16_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred ep, acc;\n\t.reg .b32 er;\n\telect.sync er|ep, 0xffffffff;\n\t"
        "setp.ne.b32 acc, %4, 0;\n\t"
        "@ep tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, acc;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two FP32 values -> packed BF16 pair (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Expert owning routed row `row`: largest e < E with off[e] <= row (off in shared memory).
__device__ __forceinline__ int bwd_expert_of_row(const int32_t* off, int E, int row) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= row) lo = mid;
        else hi = mid;
    }
    return lo;
}

// The work of tile t (identical in every thread; s_off / s_end in shared memory).
struct BTile {
    int e, m0, n0;
    int a_x;        // A box coordinates: K-major (x = K bytes, y = m0) or MN-major (x = m0 bytes)
    int b_row;      // first B row of the tile's K range
    int k0;         // wgrad: first routed row
    int num_ks;     // stages with real rows
    int tail;       // real K-rows in the last stage (1..64)
};

__device__ __forceinline__ BTile bgemm_tile(const BgemmJob& job, const int32_t* s_off, const int32_t* s_end, int t) {
    BTile T;
    const int nt = t % job.n_tiles, rest = t / job.n_tiles;
    T.n0 = nt * job.BN;
    if (job.mode == kModeWgrad) {
        const int mt = rest % job.m_tiles;
        T.e = rest / job.m_tiles;
        T.m0 = mt * kBM;
        T.k0 = s_off[T.e];
        const int rows = s_end[T.e] - T.k0;
        T.num_ks = (rows + kBK - 1) / kBK;
        T.tail = rows - (T.num_ks - 1) * kBK;
        T.b_row = T.k0;
        T.a_x = 2 * T.m0;
    } else {
        T.m0 = rest * kBM;
        T.e = bwd_expert_of_row(s_off, job.E, T.m0);
        T.k0 = 0;
        T.num_ks = job.num_ks;
        T.tail = kBK;
        T.b_row = T.e * job.K;
        T.a_x = 0;
    }
    return T;
}

// The slot of 16-byte chunk j of staged row `row`.
template <class C>
__device__ __forceinline__ int stg_slot(int row, int j) {
    return j ^ ((row >> C::kStgShift) & (C::kStgSlots - 1));
}

// kWgrad: FP32 weight gradients (both operands MN-major); else BF16 activation gradients
// (A K-major, B MN-major), kModeRows or kModePairs.
template <bool kWgrad>
__global__ void __launch_bounds__(kBThreads, 1)
    bgemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const BgemmJob job) {
    using C = BCfg<kWgrad>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* empty = full + C::kStages;
    uint64_t* tmem_full = empty + C::kStages;           // [2]
    uint64_t* tmem_empty = tmem_full + 2;             // [2]
    uint64_t* drain = tmem_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int32_t* s_off = reinterpret_cast<int32_t*>(smem + C::kOffOff);
    int32_t* s_end = s_off + kBMaxE + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], kBEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kBTmemCols);
        tmem_relinquish();
    }
    // the set-up above touches only this CTA's shared memory and TMEM (and the tensor maps,
    // kernel parameters), so it overlaps the previous kernel's tail; every global read and
    // write follows the wait
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i <= job.E; i += kBThreads) {
        s_off[i] = job.offsets[i];
        if (kWgrad && i < job.E) s_end[i] = job.real_end[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int num_tiles = kWgrad ? job.E * job.m_tiles * job.n_tiles : (s_off[job.E] / kBM) * job.n_tiles;
    const int b_boxes = job.BN / 64;
    const uint32_t b_bytes = static_cast<uint32_t>(job.BN) * kBRowBytes;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (warp-uniform)
        const uint64_t pol = policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_parity = 0;
        bool failed = false;
        for (int t = blockIdx.x; t < num_tiles && !failed; t += gridDim.x) {
            const BTile T = bgemm_tile(job, s_off, s_end, t);
            for (int ks = 0; ks < T.num_ks; ++ks) {
                const bool ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, kWaitBudgetCycles);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    failed = true;
                    break;
                }
                uint8_t* st = smem + stage * kBStageBytes;
                const int k = ks * kBK;
                mbar_arrive_expect_tx_elect(&full[stage], kBABytes + b_bytes);
                if (kWgrad) {
                    tma_load_2d_elect(st, &tmA, &full[stage], T.a_x, T.k0 + k, pol);
                    tma_load_2d_elect(st + kBMnBox, &tmA, &full[stage], T.a_x + 128, T.k0 + k, pol);
                } else {
                    tma_load_2d_elect(st, &tmA, &full[stage], 2 * k, T.m0, pol);
                }
                for (int c = 0; c < b_boxes; ++c)
                    tma_load_2d_elect(st + kBABytes + c * kBMnBox, &tmB, &full[stage], 2 * (T.n0 + 64 * c),
                                      T.b_row + k, pol);
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (failed) {
            if (lane == 0) set_device_error(job.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            for (int s = 0; s < C::kStages; ++s) {
                if (issued & (1u << s)) mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, kWaitBudgetCycles);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (warp-uniform)
        const uint32_t idesc = idesc_bf16(kBM, job.BN, kWgrad, true);
        int stage = 0;
        uint32_t phase = 0, acc_iter = 0;
        bool failed = false, issued_any = false;
        for (int t = blockIdx.x; t < num_tiles && !failed; t += gridDim.x) {
            const BTile T = bgemm_tile(job, s_off, s_end, t);
            if (T.num_ks == 0) continue;
            const uint32_t buf = acc_iter & 1u;
            const bool ok_acc =
                mbar_wait_bounded(&tmem_empty[buf], ((acc_iter >> 1) & 1u) ^ 1u, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok_acc)) {
                failed = true;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + buf * kBMaxN;
            for (int ks = 0; ks < T.num_ks; ++ks) {
                const bool ok = mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitBudgetCycles);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                uint8_t* stp = smem + stage * kBStageBytes;
                if (kWgrad && ks == T.num_ks - 1 && T.tail < kBK) {
                    // rows past the expert's real rows: zero B's K-rows tail..63 in every box
                    const int chunks = (kBK - T.tail) * (kBRowBytes / 16);
                    for (int c = 0; c < b_boxes; ++c) {
                        uint4* z = reinterpret_cast<uint4*>(stp + kBABytes + c * kBMnBox + T.tail * kBRowBytes);
                        for (int i = lane; i < chunks; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                }
                const uint32_t st = smem_u32(stp);
                const uint64_t adesc = kWgrad ? sdesc_mn_sw128(st) : sdesc_k_swizzled<128>(st);
                const uint64_t bdesc = sdesc_mn_sw128(st + kBABytes);
                constexpr uint64_t a_step = kWgrad ? 2048 >> 4 : 32 >> 4;
#pragma unroll
                for (int j = 0; j < 4; ++j)   // K = 16 BF16 per MMA
                    mma_bf16_elect(d_tmem, adesc + a_step * j, bdesc + (2048 >> 4) * j, idesc,
                                   (ks | j) != 0 ? 1u : 0u);
                issued_any = true;
                tc_commit_elect(&empty[stage]);
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (failed) break;
            tc_commit_elect(&tmem_full[buf]);
            ++acc_iter;
        }
        if (failed) {
            if (lane == 0) set_device_error(job.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            if (issued_any) {   // let the issued MMAs finish before TMEM is released
                tc_commit_elect(drain);
                mbar_wait_bounded(drain, 0, nullptr, kWaitBudgetCycles);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp w reads TMEM lane quarter w % 4 (rows q*32..+31 of the tile) and one part of the
        // columns; lane l owns row q*32 + l while reading the accumulator, and the staged
        // stores cover C::kStgRowsPerSt rows x C::kStgWords*4 bytes per instruction.
        constexpr int kColsPerChunk = kWgrad ? C::kStgWords : 2 * C::kStgWords;   // accumulator columns
        const int q = warp & 3;
        const int part = (warp - 2) >> 2;
        const int cols = job.BN / (kBEpiWarps / 4);
        uint32_t* stg = reinterpret_cast<uint32_t*>(smem + C::kStgOff) + (warp - 2) * (C::kStgBytes / 4);
        const int srow = lane / C::kStgSlots;                  // this lane's row within a store's rows
        const int sj = lane % C::kStgSlots;                    // and its 16-byte slot
        uint32_t acc_iter = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const BTile T = bgemm_tile(job, s_off, s_end, t);
            const int c0 = T.n0 + part * cols;
            const int row = T.m0 + q * 32 + lane;
            // start of this lane's row segment (nullptr: not stored)
            uint8_t* dst;
            if (kWgrad) {
                dst = reinterpret_cast<uint8_t*>(job.out_f32 + (static_cast<int64_t>(T.e) * job.M + row) * job.N + c0);
            } else if (job.mode == kModeRows) {
                dst = reinterpret_cast<uint8_t*>(job.out_bf16 + static_cast<int64_t>(row) * job.N + c0);
            } else {
                const int pair = job.row_pair[row];
                dst = pair >= 0 ? reinterpret_cast<uint8_t*>(job.out_bf16 + static_cast<int64_t>(pair) * job.N + c0)
                                : nullptr;
            }
            const int chunks = cols / kColsPerChunk;
            if (kWgrad && T.num_ks == 0) {
                // an expert without routed rows: its weight gradient is zero
                for (int ch = 0; ch < chunks; ++ch) {
#pragma unroll
                    for (int i = 0; i < C::kStgSlots; ++i) {
                        const int rr = i * C::kStgRowsPerSt + srow;
                        uint8_t* d = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(dst), rr));
                        *reinterpret_cast<uint4*>(d + ch * C::kStgWords * 4 + sj * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                continue;
            }
            const uint32_t buf = acc_iter & 1u;
            const bool ok = mbar_wait_bounded(&tmem_full[buf], (acc_iter >> 1) & 1u, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                if (lane == 0) set_device_error(job.err, NVFP4_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem + buf * kBMaxN + part * cols + (static_cast<uint32_t>(q * 32) << 16);
            for (int ch = 0; ch < chunks; ++ch) {
                uint32_t v[kColsPerChunk];
#pragma unroll
                for (int l = 0; l < kColsPerChunk / 16; ++l)
                    tmem_ld_32x32b_x16(taddr + ch * kColsPerChunk + 16 * l, reinterpret_cast<uint32_t(&)[16]>(v[16 * l]));
                tmem_ld_wait();
                uint32_t w[C::kStgWords];
#pragma unroll
                for (int i = 0; i < C::kStgWords; ++i)
                    w[i] = kWgrad ? v[i] : pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
#pragma unroll
                for (int j = 0; j < C::kStgSlots; ++j)
                    *reinterpret_cast<uint4*>(stg + lane * C::kStgWords + 4 * stg_slot<C>(lane, j)) =
                        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < C::kStgSlots; ++i) {
                    const int rr = i * C::kStgRowsPerSt + srow;
                    const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * C::kStgWords + 4 * stg_slot<C>(rr, sj));
                    uint8_t* d = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(dst), rr));
                    if (d != nullptr) *reinterpret_cast<uint4*>(d + ch * C::kStgWords * 4 + sj * 16) = val;
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tmem_empty[buf]);
            ++acc_iter;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kBTmemCols);
    }
}

// dst[r][0..C) = src[row_pair[r] / k][0..C) for the routed rows r < offsets[E], zeros for a
// pad row; one warp per row, 16-byte copies, C % 8 == 0.  With real_end != nullptr the grid
// has ceil(E/8) more blocks, whose warps (one per expert e) write real_end[e], the end of e's
// real rows: its rows are real first, then fewer than 128 pad rows (row_pair -1).
__global__ void __launch_bounds__(256)
    gather_token_rows_kernel(const uint16_t* __restrict__ src, int C, const int32_t* __restrict__ row_pair, int k,
                             const int32_t* __restrict__ offsets, int E, int64_t row_blocks, uint16_t* __restrict__ dst,
                             int32_t* __restrict__ real_end) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    if (static_cast<int64_t>(blockIdx.x) >= row_blocks) {
        const int e = static_cast<int>((blockIdx.x - row_blocks) * 8 + (threadIdx.x >> 5));
        if (e >= E) return;
        const int k1 = offsets[e + 1];
        const int lo = max(offsets[e], k1 - 128);
        int first = k1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int idx = lo + 4 * lane + j;
            if (idx < k1 && row_pair[idx] < 0) first = min(first, idx);
        }
        first = __reduce_min_sync(0xFFFFFFFFu, first);
        if (lane == 0) real_end[e] = first;
        return;
    }
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= offsets[E]) return;
    const int pair = row_pair[r];
    const uint4* s = pair >= 0 ? reinterpret_cast<const uint4*>(src + static_cast<int64_t>(pair / k) * C) : nullptr;
    uint4* d = reinterpret_cast<uint4*>(dst + r * C);
    for (int i = lane; i < C / 8; i += 32) d[i] = s != nullptr ? s[i] : make_uint4(0u, 0u, 0u, 0u);
}

// The SwiGLU x prob derivative, one warp per routed row r < offsets[E]:
//   a, u = gu[r][i], gu[r][I + i] (the forward's BF16 gate and up), s = sigma(a)
//   dgu[r][i] = bf16(dh*p*u*s*(1 + a*(1-s))),  dgu[r][I + i] = bf16(dh*p*(a*s))
//   dprob[row_pair[r]] = sum_i dh_i*(a_i*s_i)*u_i   (FP32; per lane in column order, then a
//                                                    fixed butterfly over the lanes)
// A pad row gets zeros.  I % 8 == 0.
__global__ void __launch_bounds__(256)
    swiglu_bwd_kernel(const uint16_t* __restrict__ dh, const uint16_t* __restrict__ gu,
                      const int32_t* __restrict__ row_pair, const float* __restrict__ row_prob,
                      const int32_t* __restrict__ offsets, int E, int I, uint16_t* __restrict__ dgu,
                      float* __restrict__ dprob) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= offsets[E]) return;
    const int pair = row_pair[r];
    uint4* drow = reinterpret_cast<uint4*>(dgu + r * 2 * I);
    const int nvec = I / 8;
    if (pair < 0) {
        for (int c = lane; c < 2 * nvec; c += 32) drow[c] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const float p = row_prob[r];
    const uint4* dhr = reinterpret_cast<const uint4*>(dh + r * I);
    const uint4* gate = reinterpret_cast<const uint4*>(gu + r * 2 * I);
    const uint4* up = gate + nvec;
    float acc = 0.0f;
    for (int c = lane; c < nvec; c += 32) {
        const uint4 d4 = dhr[c], g4 = gate[c], u4 = up[c];
        const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
        const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
        const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
        float da[8], du[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float dhv = (j & 1) ? bf16_hi(dw[j >> 1]) : bf16_lo(dw[j >> 1]);
            const float a = (j & 1) ? bf16_hi(gw[j >> 1]) : bf16_lo(gw[j >> 1]);
            const float u = (j & 1) ? bf16_hi(uw[j >> 1]) : bf16_lo(uw[j >> 1]);
            const float s = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-a)));
            const float silu = __fmul_rn(a, s);
            const float dsilu = __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(a, __fsub_rn(1.0f, s))));
            const float g = __fmul_rn(dhv, p);
            da[j] = __fmul_rn(__fmul_rn(g, u), dsilu);
            du[j] = __fmul_rn(g, silu);
            acc = __fadd_rn(acc, __fmul_rn(__fmul_rn(dhv, silu), u));
        }
        drow[c] = make_uint4(pack_bf16x2(da[0], da[1]), pack_bf16x2(da[2], da[3]), pack_bf16x2(da[4], da[5]),
                             pack_bf16x2(da[6], da[7]));
        drow[nvec + c] = make_uint4(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]), pack_bf16x2(du[4], du[5]),
                                    pack_bf16x2(du[6], du[7]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
    if (lane == 0) dprob[pair] = acc;
}

// ------------------------------------------------------------------ host side
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

// Byte-typed 2D map over a BF16 matrix [rows][cols]: boxes of box_rows rows x 128 bytes
// (64 consecutive elements of a row), 128B swizzle.  A K-major operand takes 128- or 256-row
// boxes (64 elements of K per row); an MN-major one 64-row boxes (64 K-rows of 64 elements).
bool make_box_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * cols)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBRowBytes), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
std::mutex g_bwd_mutex;
bool g_bwd_attr[kMaxDevices];

cudaError_t ensure_smem_attr() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_bwd_mutex);
    if (!g_bwd_attr[dev]) {
        e = cudaFuncSetAttribute(bgemm_bf16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 BCfg<false>::kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(bgemm_bf16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 BCfg<true>::kSmemBytes);
        if (e != cudaSuccess) return e;
        g_bwd_attr[dev] = true;
    }
    return cudaSuccess;
}

int tile_n(int N) { return N % 256 == 0 ? 256 : 128; }

unsigned persistent_grid(int64_t tiles) {
    return static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(tiles, device_sm_count())));
}

// Grouped dgrad: out = A (routed rows [rows_cap][K], K-major) x B[e] (B [E*K][N], rows e*K..
// are expert e's), K % 64 == 0, N % 128 == 0.
cudaError_t launch_dgrad(const uint16_t* A, const uint16_t* B, int64_t rows_cap, int K, int N, int E,
                         const int32_t* offsets, const int32_t* row_pair, int mode, uint16_t* out, int* err,
                         cudaStream_t st, bool pdl) {
    BgemmJob j{};
    j.mode = mode;
    j.BN = tile_n(N);
    j.n_tiles = N / j.BN;
    j.m_tiles = static_cast<int>(rows_cap / kBM);
    j.N = N;
    j.M = 0;
    j.num_ks = K / kBK;
    j.K = K;
    j.E = E;
    j.offsets = offsets;
    j.real_end = nullptr;
    j.row_pair = row_pair;
    j.out_bf16 = out;
    j.out_f32 = nullptr;
    j.err = err;
    CUtensorMap ma, mb;
    if (!make_box_map(&ma, A, rows_cap, K, kBM) || !make_box_map(&mb, B, static_cast<int64_t>(E) * K, N, kBK))
        return cudaErrorInvalidValue;
    return launch_pdl(pdl, bgemm_bf16_kernel<false>, persistent_grid(static_cast<int64_t>(j.m_tiles) * j.n_tiles),
                      kBThreads, BCfg<false>::kSmemBytes, st, ma, mb, j);
}

// Grouped wgrad: out[e] (FP32 [M][N]) = A[rows of e]^T B[rows of e] with A [rows_cap][M],
// B [rows_cap][N] (K over expert e's real routed rows offsets[e] .. real_end[e]).
cudaError_t launch_wgrad(const uint16_t* A, const uint16_t* B, int64_t rows_cap, int M, int N, int E,
                         const int32_t* offsets, const int32_t* real_end, float* out, int* err, cudaStream_t st,
                         bool pdl) {
    BgemmJob j{};
    j.mode = kModeWgrad;
    j.BN = tile_n(N);
    j.n_tiles = N / j.BN;
    j.m_tiles = M / kBM;
    j.N = N;
    j.M = M;
    j.num_ks = 0;
    j.K = 0;
    j.E = E;
    j.offsets = offsets;
    j.real_end = real_end;
    j.row_pair = nullptr;
    j.out_bf16 = nullptr;
    j.out_f32 = out;
    j.err = err;
    CUtensorMap ma, mb;
    if (!make_box_map(&ma, A, rows_cap, M, kBK) || !make_box_map(&mb, B, rows_cap, N, kBK))
        return cudaErrorInvalidValue;
    return launch_pdl(pdl, bgemm_bf16_kernel<true>, persistent_grid(static_cast<int64_t>(E) * j.m_tiles * j.n_tiles),
                      kBThreads, BCfg<true>::kSmemBytes, st, ma, mb, j);
}

cudaError_t launch_gather(const uint16_t* src, int C, const BackwardArgs& a, uint16_t* dst, int32_t* real_end,
                          cudaStream_t st, bool pdl) {
    const int64_t row_blocks = a.rows_cap / 8;
    const int64_t blocks = row_blocks + (real_end != nullptr ? (a.E + 7) / 8 : 0);
    return launch_pdl(pdl, gather_token_rows_kernel, static_cast<unsigned>(blocks), 256, 0, st, src, C, a.row_pair,
                      a.k, a.offsets, a.E, row_blocks, dst, real_end);
}

}  // namespace

cudaError_t launch_moe_backward_ste(const BackwardArgs& a, cudaStream_t st) {
    if (a.E > kBMaxE) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr();
    if (e != cudaSuccess) return e;
    const int64_t rc = a.rows_cap;
    // The first kernel is launched normally (ordered after whatever the caller queued); each
    // later one as a programmatic dependent of the one before it: its CTAs are scheduled while
    // that kernel finishes and wait (griddepcontrol.wait) before their first global access.
    // dY rows (and each expert's end of real rows), FC2 dgrad, SwiGLU x prob derivative
    e = launch_gather(a.dout, a.H, a, a.dy_rows, a.real_end, st, false);
    if (e != cudaSuccess) return e;
    e = launch_dgrad(a.dy_rows, a.w2, rc, a.H, a.I, a.E, a.offsets, a.row_pair, kModeRows, a.dh, a.err, st, true);
    if (e != cudaSuccess) return e;
    e = launch_pdl(true, swiglu_bwd_kernel, static_cast<unsigned>(rc / 8), 256, 0, st, a.dh, a.gu, a.row_pair,
                   a.row_prob, a.offsets, a.E, a.I, a.dgu, a.dprob);
    if (e != cudaSuccess) return e;
    // FC1 dgrad per (token, slot), then the slot-order sum
    e = launch_dgrad(a.dgu, a.w1, rc, 2 * a.I, a.H, a.E, a.offsets, a.row_pair, kModePairs, a.dx_pairs, a.err, st,
                     true);
    if (e != cudaSuccess) return e;
    e = launch_combine(a.dx_pairs, nullptr, a.T, a.k, a.H, a.dx, st, true);
    if (e != cudaSuccess) return e;
    // FC2 wgrad: dW2[e] = dy^T h over the expert's real rows
    e = launch_wgrad(a.dy_rows, a.h, rc, a.H, a.I, a.E, a.offsets, a.real_end, a.dw2, a.err, st, true);
    if (e != cudaSuccess) return e;
    // FC1 wgrad: dW1[e] = [da, du]^T x over the expert's real rows
    e = launch_gather(a.x, a.H, a, a.x_rows, nullptr, st, true);
    if (e != cudaSuccess) return e;
    return launch_wgrad(a.dgu, a.x_rows, rc, 2 * a.I, a.H, a.E, a.offsets, a.real_end, a.dw1, a.err, st, true);
}

}  // namespace nvfp4
