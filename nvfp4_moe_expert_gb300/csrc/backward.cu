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
//   SwiGLU     a, u = bf16 of the forward's FC1 values of r (the gate/up the SwiGLU ran on),
//              s = 1/(1+exp(-a)):  da = bf16(dh*p*u*s*(1+a*(1-s))),  du = bf16(dh*p*a*s),
//              dprob[pair(r)] = sum_i dh_i*(a_i*s_i)*u_i               (FP32)
//   FC1 dgrad  dxs[pair(r)] = bf16( [da, du] W1[e] )        BF16 GEMM
//   combine    dX[t] = bf16( sum over slots 0..k-1 in order of dxs, FP32 )
//   FC2 wgrad  dW2[e] = sum_r dy[r]^T h[r]                  FP32 output
//   FC1 wgrad  dW1[e] = sum_r [da, du][r]^T x[t(r)]         FP32 output
//
// Every GEMM reads both operands K-major through TMA (128B swizzle, 64 BF16 of K per stage)
// and runs tcgen05.mma.kind::f16 (M=128, N=128 or 256, FP32 accumulator in TMEM): the
// weights come as per-expert transposed copies made once per weight version
// (nvfp4_transpose_bf16); for the weight gradients, whose K runs over one expert's routed
// rows, dy, h, [da, du] and the gathered x are transposed into [feature][routed row] copies
// first.  One CTA per 128 x N output tile: warp 0 issues the TMA loads, warp 1 the MMAs,
// warps 2-5 read the accumulator (one row per thread) and store it.  Each tile walks K in
// one fixed order, so a token's dX and dprob do not depend on the other tokens.
#include <mutex>

#include "backward.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kBStages = 4;
constexpr int kBM = 128;                                // output rows per tile
constexpr int kBK = 64;                                 // BF16 elements of K per stage
constexpr int kBRowBytes = 2 * kBK;                     // 128 bytes, one swizzle span
constexpr int kBMaxN = 256;
constexpr int kBABytes = kBM * kBRowBytes;              // 16 KB
constexpr int kBBBytes = kBMaxN * kBRowBytes;           // 32 KB
constexpr int kBStageBytes = kBABytes + kBBBytes;       // 48 KB
constexpr int kBBarOff = kBStages * kBStageBytes;
constexpr int kBSmemBytes = kBBarOff + 128 + 1024;
constexpr int kBThreads = 192;                          // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kBTmemCols = 256;

enum : int { kModeRows = 0, kModePairs = 1, kModeWgrad = 2 };

// One launch of the grouped GEMM C = A B^T (A [.][K], B [.][K], both BF16 K-major).
//  kModeRows  (dgrad): tile (m, n) -> routed rows m*128.., expert e owning them; A rows there,
//             B rows e*N + n0..; K = num_ks*64 from 0; out_bf16[row][n], row stride N.
//  kModePairs (dgrad): as kModeRows, but row r goes to out_bf16[row_pair[r]][n] (pad rows
//             are not stored).
//  kModeWgrad: tile (e, m, n) -> A rows m*128.. and B rows n0.. of [feature][routed row]
//             copies, K over expert e's routed rows [offsets[e], offsets[e+1]);
//             out_f32[e][m][n] (an expert without rows gets zeros).
struct BgemmJob {
    int mode;
    int BN;             // 128 or 256
    int n_tiles;        // N / BN
    int m_tiles;        // dgrad: rows_cap / 128; wgrad: M / 128
    int N;              // output columns
    int M;              // wgrad: output rows per expert
    int num_ks;         // dgrad: K / 64
    int E;
    const int32_t* offsets;
    const int32_t* row_pair;
    uint16_t* out_bf16;
    float* out_f32;
    int* err;
};

// Instruction descriptor of tcgen05.mma kind::f16: BF16 A and B, both K-major, FP32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16_kmajor(int M, int N) {
    return (1u << 4)                                  // D format: F32
           | (1u << 7)                                // A format: BF16
           | (1u << 10)                               // B format: BF16
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// D(tmem, FP32) (+)= A(smem, BF16) x B(smem, BF16)^T, M=128, K=16, issued by the lane
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

// 32-byte store; p 32-byte aligned.
__device__ __forceinline__ void st_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__global__ void __launch_bounds__(kBThreads, 1)
    bgemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const BgemmJob job) {
    // ---- the tile of this CTA (identical in every thread)
    const int nt = static_cast<int>(blockIdx.x % static_cast<unsigned>(job.n_tiles));
    const int rest = static_cast<int>(blockIdx.x / static_cast<unsigned>(job.n_tiles));
    const int n0 = nt * job.BN;
    int e, m0, a_row, b_row, k0, num_ks;
    if (job.mode == kModeWgrad) {
        const int mt = rest % job.m_tiles;
        e = rest / job.m_tiles;
        m0 = mt * kBM;
        a_row = m0;
        b_row = n0;
        k0 = job.offsets[e];
        num_ks = (job.offsets[e + 1] - k0) / kBK;
    } else {
        m0 = rest * kBM;
        if (m0 >= job.offsets[job.E]) return;          // past the last expert's rows
        int lo = 0, hi = job.E - 1;                     // the last e with offsets[e] <= m0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (job.offsets[mid] <= m0) lo = mid; else hi = mid - 1;
        }
        e = lo;
        a_row = m0;
        b_row = e * job.N + n0;
        k0 = 0;
        num_ks = job.num_ks;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBBarOff);
    uint64_t* empty = full + kBStages;
    uint64_t* tmem_full = empty + kBStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tmem_full, 1);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t b_bytes = static_cast<uint32_t>(job.BN) * kBRowBytes;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (warp-uniform)
        const uint64_t pol = policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_parity = 0;
        bool failed = false;
        for (int ks = 0; ks < num_ks; ++ks) {
            const bool ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                failed = true;
                break;
            }
            uint8_t* st = smem + stage * kBStageBytes;
            const int x = (k0 + ks * kBK) * 2;          // byte coordinate along K
            mbar_arrive_expect_tx_elect(&full[stage], kBABytes + b_bytes);
            tma_load_2d_elect(st, &tmA, &full[stage], x, a_row, pol);
            tma_load_2d_elect(st + kBABytes, &tmB, &full[stage], x, b_row, pol);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == kBStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (failed) {
            if (lane == 0) set_device_error(job.err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            for (int s = 0; s < kBStages; ++s) {
                if (issued & (1u << s)) mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, kWaitBudgetCycles);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (warp-uniform)
        const uint32_t idesc = idesc_bf16_kmajor(kBM, job.BN);
        int stage = 0;
        uint32_t phase = 0;
        bool failed = false, issued_any = false;
        for (int ks = 0; ks < num_ks; ++ks) {
            const bool ok = mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                failed = true;
                break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + stage * kBStageBytes);
            const uint64_t adesc = sdesc_k_swizzled<128>(st);
            const uint64_t bdesc = sdesc_k_swizzled<128>(st + kBABytes);
#pragma unroll
            for (int j = 0; j < 4; ++j)   // K = 16 BF16 (32 bytes) per MMA
                mma_bf16_elect(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (ks | j) != 0 ? 1u : 0u);
            issued_any = true;
            tc_commit_elect(&empty[stage]);
            if (++stage == kBStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (num_ks > 0) {
            if (!failed) {
                tc_commit_elect(tmem_full);
            } else {
                if (lane == 0) set_device_error(job.err, NVFP4_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                if (issued_any) {   // let the issued MMAs finish before TMEM is released
                    tc_commit_elect(tmem_full);
                    mbar_wait_bounded(tmem_full, 0, nullptr, kWaitBudgetCycles);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue: one row per thread
        const int q = warp & 3;                             // TMEM lane quarter
        const int r = q * 32 + lane;                        // row of the tile
        // destination of this row (nullptr: not stored)
        uint16_t* orow16 = nullptr;
        float* orow32 = nullptr;
        if (job.mode == kModeRows) {
            orow16 = job.out_bf16 + static_cast<int64_t>(m0 + r) * job.N + n0;
        } else if (job.mode == kModePairs) {
            const int pair = job.row_pair[m0 + r];
            if (pair >= 0) orow16 = job.out_bf16 + static_cast<int64_t>(pair) * job.N + n0;
        } else {
            orow32 = job.out_f32 + (static_cast<int64_t>(e) * job.M + m0 + r) * job.N + n0;
        }
        if (num_ks == 0) {
            // an expert without routed rows: its weight gradient is zero
            const uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (orow32 != nullptr)
                for (int c = 0; c < job.BN; c += 8) st_v8(orow32 + c, z);
        } else {
            const bool ok = mbar_wait_bounded(tmem_full, 0, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                if (lane == 0) set_device_error(job.err, NVFP4_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            } else {
                tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
                for (int c = 0; c < job.BN; c += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(taddr + c, v);
                    tmem_ld_wait();
                    if (orow16 != nullptr) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                        st_v8(orow16 + c, w);
                    } else if (orow32 != nullptr) {
                        uint32_t w0[8], w1[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            w0[i] = v[i];
                            w1[i] = v[8 + i];
                        }
                        st_v8(orow32 + c, w0);
                        st_v8(orow32 + c + 8, w1);
                    }
                }
            }
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
// pad row.  One warp per row, 16-byte copies; C % 8 == 0.
__global__ void __launch_bounds__(256)
    gather_token_rows_kernel(const uint16_t* __restrict__ src, int C, const int32_t* __restrict__ row_pair, int k,
                             const int32_t* __restrict__ offsets, int E, uint16_t* __restrict__ dst) {
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= offsets[E]) return;
    const int pair = row_pair[r];
    const uint4* s = pair >= 0 ? reinterpret_cast<const uint4*>(src + static_cast<int64_t>(pair / k) * C) : nullptr;
    uint4* d = reinterpret_cast<uint4*>(dst + r * C);
    for (int i = lane; i < C / 8; i += 32) d[i] = s != nullptr ? s[i] : make_uint4(0u, 0u, 0u, 0u);
}

enum : int { kSrcPlain = 0, kSrcToken = 1, kSrcRouted = 2 };

// Transpose of one 64 x 64 tile: out[c][r] = S(r)[c] for r in [r0, r0+64), c in [c0, c0+64),
// where S(r) is, for problem z = blockIdx.z,
//   kSrcPlain:   row r of in + z*in_batch (stride ld_in)
//   kSrcToken:   row row_pair[r] / k of in, or zeros if row_pair[r] < 0   (r < offsets[E])
//   kSrcRouted:  row r of in, or zeros if row_pair[r] < 0                  (r < offsets[E])
// out row c (stride ld_out) of problem z starts at out + z*out_batch.  Row tiles past
// offsets[E] are not written in the routed modes.  ld_in, ld_out, in_batch, out_batch,
// r0 and c0 are multiples of 64 elements (16-byte aligned rows).
template <int kSrc>
__global__ void __launch_bounds__(256)
    transpose_tile_kernel(const uint16_t* __restrict__ in, int64_t ld_in, int64_t in_batch,
                          const int32_t* __restrict__ row_pair, int k, const int32_t* __restrict__ offsets, int E,
                          uint16_t* __restrict__ out, int64_t ld_out, int64_t out_batch) {
    __shared__ __align__(16) uint16_t tile[64][66];   // 33-word rows: the column reads spread over the banks
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * 64;
    const int64_t z = blockIdx.z;
    if (kSrc != kSrcPlain && r0 >= offsets[E]) return;
    const int t = threadIdx.x;
    {
        const int rr = t >> 2, cc = (t & 3) * 16;        // 16 elements of source row r0 + rr
        const int64_t r = r0 + rr;
        const uint16_t* src = nullptr;
        if (kSrc == kSrcPlain) {
            src = in + z * in_batch + r * ld_in;
        } else {
            const int pair = row_pair[r];
            if (pair >= 0) src = in + (kSrc == kSrcToken ? static_cast<int64_t>(pair / k) : r) * ld_in;
        }
        uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
        if (src != nullptr) {
            const uint4* s = reinterpret_cast<const uint4*>(src + c0 + cc);
            v0 = s[0];
            v1 = s[1];
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(&tile[rr][cc]);
        dst[0] = v0.x; dst[1] = v0.y; dst[2] = v0.z; dst[3] = v0.w;
        dst[4] = v1.x; dst[5] = v1.y; dst[6] = v1.z; dst[7] = v1.w;
    }
    __syncthreads();
    {
        const int cc = t >> 2, rr = (t & 3) * 16;        // 16 elements of output row c0 + cc
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = static_cast<uint32_t>(tile[rr + 2 * i][cc]) | (static_cast<uint32_t>(tile[rr + 2 * i + 1][cc]) << 16);
        uint4* d = reinterpret_cast<uint4*>(out + z * out_batch + (c0 + cc) * ld_out + r0 + rr);
        d[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// The SwiGLU x prob derivative, one warp per routed row r < offsets[E]:
//   a, u = bf16(fc1_pre[r][i]), bf16(fc1_pre[r][I + i]) (the forward's gate and up), s = sigma(a)
//   dgu[r][i] = bf16(dh*p*u*s*(1 + a*(1-s))),  dgu[r][I + i] = bf16(dh*p*(a*s))
//   dprob[row_pair[r]] = sum_i dh_i*(a_i*s_i)*u_i   (FP32; per lane in column order, then a
//                                                    fixed butterfly over the lanes)
// A pad row gets zeros.  I % 8 == 0.
__global__ void __launch_bounds__(256)
    swiglu_bwd_kernel(const uint16_t* __restrict__ dh, const float* __restrict__ fc1_pre,
                      const int32_t* __restrict__ row_pair, const float* __restrict__ row_prob,
                      const int32_t* __restrict__ offsets, int E, int I, uint16_t* __restrict__ dgu,
                      float* __restrict__ dprob) {
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
    const float4* gate = reinterpret_cast<const float4*>(fc1_pre + r * 2 * I);
    const float4* up = gate + I / 4;
    float acc = 0.0f;
    for (int c = lane; c < nvec; c += 32) {
        const uint4 d4 = dhr[c];
        const float4 g0 = gate[2 * c], g1 = gate[2 * c + 1], u0 = up[2 * c], u1 = up[2 * c + 1];
        const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float uvr[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float da[8], du[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float dhv = (j & 1) ? bf16_hi(dw[j >> 1]) : bf16_lo(dw[j >> 1]);
            const uint32_t ab = pack_bf16x2(gv[j], uvr[j]);      // the forward's BF16 gate and up
            const float a = bf16_lo(ab), u = bf16_hi(ab);
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

// Byte-typed 2D map over a K-major BF16 matrix [rows][K]: boxes of box_rows rows x 128 bytes
// (64 elements of K), 128B swizzle.
bool make_kmajor_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * K)};
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
        e = cudaFuncSetAttribute(bgemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmemBytes);
        if (e != cudaSuccess) return e;
        g_bwd_attr[dev] = true;
    }
    return cudaSuccess;
}

int tile_n(int N) { return N % 256 == 0 ? 256 : 128; }

// Grouped dgrad: out = A (routed rows [rows_cap][K]) x B[e]^T (B [E*N][K]), K % 64 == 0, N % 128 == 0.
cudaError_t launch_dgrad(const uint16_t* A, const uint16_t* B, int64_t rows_cap, int K, int N, int E,
                         const int32_t* offsets, const int32_t* row_pair, int mode, uint16_t* out, int* err,
                         cudaStream_t st) {
    BgemmJob j{};
    j.mode = mode;
    j.BN = tile_n(N);
    j.n_tiles = N / j.BN;
    j.m_tiles = static_cast<int>(rows_cap / kBM);
    j.N = N;
    j.M = 0;
    j.num_ks = K / kBK;
    j.E = E;
    j.offsets = offsets;
    j.row_pair = row_pair;
    j.out_bf16 = out;
    j.out_f32 = nullptr;
    j.err = err;
    CUtensorMap ma, mb;
    if (!make_kmajor_map(&ma, A, rows_cap, K, kBM) || !make_kmajor_map(&mb, B, static_cast<int64_t>(E) * N, K, j.BN))
        return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(j.m_tiles) * j.n_tiles);
    return launch_pdl(false, bgemm_bf16_kernel, grid, kBThreads, kBSmemBytes, st, ma, mb, j);
}

// Grouped wgrad: out[e] (FP32 [M][N]) = A[:, rows of e] x B[:, rows of e]^T with A [M][rows_cap],
// B [N][rows_cap] (K over the routed rows of expert e).
cudaError_t launch_wgrad(const uint16_t* A, const uint16_t* B, int64_t rows_cap, int M, int N, int E,
                         const int32_t* offsets, float* out, int* err, cudaStream_t st) {
    BgemmJob j{};
    j.mode = kModeWgrad;
    j.BN = tile_n(N);
    j.n_tiles = N / j.BN;
    j.m_tiles = M / kBM;
    j.N = N;
    j.M = M;
    j.num_ks = 0;
    j.E = E;
    j.offsets = offsets;
    j.row_pair = nullptr;
    j.out_bf16 = nullptr;
    j.out_f32 = out;
    j.err = err;
    CUtensorMap ma, mb;
    if (!make_kmajor_map(&ma, A, M, rows_cap, kBM) || !make_kmajor_map(&mb, B, N, rows_cap, j.BN))
        return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(E) * j.m_tiles * j.n_tiles);
    return launch_pdl(false, bgemm_bf16_kernel, grid, kBThreads, kBSmemBytes, st, ma, mb, j);
}

template <int kSrc>
cudaError_t launch_transpose(const uint16_t* in, int64_t ld_in, int64_t in_batch, const int32_t* row_pair, int k,
                             const int32_t* offsets, int E, int64_t rows, int64_t cols, int64_t batch, uint16_t* out,
                             int64_t ld_out, int64_t out_batch, cudaStream_t st) {
    const dim3 grid(static_cast<unsigned>(rows / 64), static_cast<unsigned>(cols / 64), static_cast<unsigned>(batch));
    return launch_pdl(false, transpose_tile_kernel<kSrc>, grid, 256, 0, st, in, ld_in, in_batch, row_pair, k, offsets,
                      E, out, ld_out, out_batch);
}

}  // namespace

cudaError_t launch_transpose_bf16(const uint16_t* in, int64_t batch, int64_t rows, int64_t cols, uint16_t* out,
                                  cudaStream_t st) {
    if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
    return launch_transpose<kSrcPlain>(in, cols, rows * cols, nullptr, 1, nullptr, 0, rows, cols, batch, out, rows,
                                       rows * cols, st);
}

cudaError_t launch_moe_backward_ste(const BackwardArgs& a, cudaStream_t st) {
    cudaError_t e = ensure_smem_attr();
    if (e != cudaSuccess) return e;
    const int64_t rc = a.rows_cap;
    const unsigned warp_rows_grid = static_cast<unsigned>(rc / 8);
    // dY rows, FC2 dgrad, SwiGLU x prob derivative
    e = launch_pdl(false, gather_token_rows_kernel, warp_rows_grid, 256, 0, st, a.dout, a.H, a.row_pair, a.k,
                   a.offsets, a.E, a.dy_rows);
    if (e != cudaSuccess) return e;
    e = launch_dgrad(a.dy_rows, a.w2t, rc, a.H, a.I, a.E, a.offsets, a.row_pair, kModeRows, a.dh, a.err, st);
    if (e != cudaSuccess) return e;
    e = launch_pdl(false, swiglu_bwd_kernel, warp_rows_grid, 256, 0, st, a.dh, a.fc1_pre, a.row_pair, a.row_prob,
                   a.offsets, a.E, a.I, a.dgu, a.dprob);
    if (e != cudaSuccess) return e;
    // FC1 dgrad per (token, slot), then the slot-order sum
    e = launch_dgrad(a.dgu, a.w1t, rc, 2 * a.I, a.H, a.E, a.offsets, a.row_pair, kModePairs, a.dx_pairs, a.err, st);
    if (e != cudaSuccess) return e;
    e = launch_combine(a.dx_pairs, nullptr, a.T, a.k, a.H, a.dx, st, false);
    if (e != cudaSuccess) return e;
    // FC2 wgrad: dW2[e] = dy^T h over the expert's rows
    e = launch_transpose<kSrcToken>(a.dout, a.H, 0, a.row_pair, a.k, a.offsets, a.E, rc, a.H, 1, a.dy_t, rc, 0, st);
    if (e != cudaSuccess) return e;
    e = launch_transpose<kSrcRouted>(a.h, a.I, 0, a.row_pair, a.k, a.offsets, a.E, rc, a.I, 1, a.h_t, rc, 0, st);
    if (e != cudaSuccess) return e;
    e = launch_wgrad(a.dy_t, a.h_t, rc, a.H, a.I, a.E, a.offsets, a.dw2, a.err, st);
    if (e != cudaSuccess) return e;
    // FC1 wgrad: dW1[e] = [da, du]^T x over the expert's rows
    e = launch_transpose<kSrcRouted>(a.dgu, 2 * a.I, 0, a.row_pair, a.k, a.offsets, a.E, rc, 2 * a.I, 1, a.dgu_t, rc,
                                     0, st);
    if (e != cudaSuccess) return e;
    e = launch_transpose<kSrcToken>(a.x, a.H, 0, a.row_pair, a.k, a.offsets, a.E, rc, a.H, 1, a.x_t, rc, 0, st);
    if (e != cudaSuccess) return e;
    return launch_wgrad(a.dgu_t, a.x_t, rc, 2 * a.I, a.H, a.E, a.offsets, a.dw1, a.err, st);
}

}  // namespace nvfp4
