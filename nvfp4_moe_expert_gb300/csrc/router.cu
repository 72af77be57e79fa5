// Router step: logits = X W_r^T with BF16 inputs and an FP32 tensor-core accumulator, the top-k
// experts of every token and their probabilities, in one kernel.
//
// "Finishing RL training faster: bitwise consistency, high performance, agent-driven"
// (spke.com/ko/ai/article/3192): section 4.1 "Dense GEMM" — one FP32-output router GEMM for
// every batch size, so a token's scores never depend on the batch it is in; section 2 — top-k
// turns a 1-ulp difference into a different expert set, so ties and output order are fixed;
// section 4.4 — with that single kernel the recomputed routing matches.
//
// Selection: the k largest logits, a larger logit first and the lower expert id first on equal
// logits (softmax is monotonic, so this is the probability order).  Probabilities: the softmax
// over all experts renormalised over the k chosen, computed as the softmax over the chosen,
// p_j = exp(l_j - l_1) / sum_i exp(l_i - l_1) in FP32, the sum in slot order.
//
// Kernel (sm_103a): a cluster of four CTAs per 128-token tile, one per quarter of H.  In each
// CTA warp 0 loads the tile's X rows and W_r over its K quarter through TMA (128 bytes of K
// per row per stage, 128B swizzle, 4-stage ring) and warp 1 issues tcgen05.mma.kind::f16
// (M=128, N=E, K=16) into an FP32 TMEM accumulator, walking its quarter in one fixed order;
// warps 2-5 copy the partial logits into shared memory.  After a cluster barrier, CTA c sums
// rows 32c..32c+31 over the four partials in quarter order on all eight warps, reading the
// peers' shared memory (distributed shared memory), so a logit is ((q0 + q1) + q2) + q3
// whatever T is; eight threads per token then pick the top k (k rounds of a 64-bit key
// maximum) and write ids and probabilities.  A second cluster barrier keeps every CTA's shared
// memory alive until its peers have read it; every thread reaches both barriers on every
// path.  All pipeline waits are bounded (NVFP4_ERR_DEVICE_TIMEOUT, then a clean exit).
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kRStages = 4;
constexpr int kRSplit = 4;                              // K quarters: the CTAs of one cluster
constexpr int kRBM = 128;                               // tokens per cluster
constexpr int kRRowBytes = 128;                         // bytes of K per row per stage (64 BF16)
constexpr int kRMaxE = 256;
constexpr int kRABytes = kRBM * kRRowBytes;             // 16 KB
constexpr int kRBBytes = kRMaxE * kRRowBytes;           // room for 256 expert rows
constexpr int kRStageBytes = kRABytes + kRBBytes;       // 48 KB
constexpr int kRBarOff = kRStages * kRStageBytes;
constexpr int kRSmemBytes = kRBarOff + 128 + 1024;
constexpr int kRWarps = 8;                              // warp 0 TMA, warp 1 MMA, warps 2-5 partial logits;
constexpr int kRThreads = 32 * kRWarps;                 // then all eight sum and select
constexpr uint32_t kRTmemCols = 256;
// after the MMAs, the partial logits sit in the idle stage buffers: 128 rows of E floats at a
// stride of E + 1 (odd: the row-per-thread stores and the column reads are conflict-free)
static_assert(kRBM * (kRMaxE + 1) * 4 <= kRBarOff, "partial logits fit in the stage buffers");
// then each token's picks (32 values, 32 ids) for this CTA's 32 tokens, then the summed logits
// of those 32 tokens (stride E + 1)
constexpr int kRPickOff = kRBM * (kRMaxE + 1) * 4;
constexpr int kRLogitOff = kRPickOff + 32 * 32 * 8;
static_assert(kRLogitOff + 32 * (kRMaxE + 1) * 4 <= kRBarOff, "picks and logits fit in the stage buffers");

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes before it are visible
// to the cluster's reads after it.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address in CTA `rank`'s shared memory of the variable at local shared address `addr`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// (Not volatile: read only between the two cluster barriers, while no CTA writes the data, so
// the compiler may batch the loads.)
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Instruction descriptor of tcgen05.mma kind::f16 with BF16 A and B (both K-major) and an FP32
// accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4)                                  // D format: F32
           | (1u << 7)                                // A format: BF16
           | (1u << 10)                               // B format: BF16
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// D(tmem, FP32) (+)= A(smem, BF16) x B(smem, BF16)^T, M=128, N from idesc, K=16, issued by the
// lane elect.sync picks (the whole warp executes this in step).  A and B are both BF16:
// kind::f16 takes one type for both operands.
__device__ __forceinline__ void tc_mma_bf16_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred ep, acc;\n\t.reg .b32 er;\n\telect.sync er|ep, 0xffffffff;\n\t"
        "setp.ne.b32 acc, %4, 0;\n\t"
        "@ep tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, acc;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Selection key of logit v of expert e: unsigned order = the selection order (a larger logit
// first, the lower id first on equal logits; -0 and +0 are equal); 0 for a NaN (never picked)
// and for no expert.  The logit's bits, made order-preserving, above the complemented id.
__device__ __forceinline__ unsigned long long select_key(float v, int e) {
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0u;
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0ull;
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | static_cast<uint32_t>(~e);
}
__device__ __forceinline__ float key_logit(unsigned long long key) {
    const uint32_t ord = static_cast<uint32_t>(key >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

// kPer: experts per thread (8 threads per token), E <= 8 * kPer
template <int kPer>
__global__ void __cluster_dims__(kRSplit, 1, 1) __launch_bounds__(kRThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, int64_t T,
                       int H, int E, int k, int32_t* __restrict__ ids, float* __restrict__ probs,
                       float* __restrict__ logits, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRBarOff);
    uint64_t* empty = full + kRStages;
    uint64_t* tmem_full = empty + kRStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* part = reinterpret_cast<float*>(smem);       // [kRBM][E + 1], valid after the MMAs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t split = cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tmem_full, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kRTmemCols);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // this CTA's K-blocks of 64: quarter `split` of H / 64 (empty for H < 256 and split 0..)
    const int num_ks = H / 64;
    const int ks0 = static_cast<int>(split) * num_ks / kRSplit;
    const int ks_per = (static_cast<int>(split) + 1) * num_ks / kRSplit - ks0;
    const int m0 = static_cast<int>(blockIdx.x / kRSplit) * kRBM;
    const uint32_t b_bytes = static_cast<uint32_t>(E) * kRRowBytes;
    const int row_stride = E + 1;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (warp-uniform)
        const uint64_t pol_x = policy_evict_first();
        const uint64_t pol_w = policy_evict_last();
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_parity = 0;
        bool failed = false;
        for (int ks = ks0; ks < ks0 + ks_per; ++ks) {
            const bool ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                failed = true;
                break;
            }
            uint8_t* st = smem + stage * kRStageBytes;
            mbar_arrive_expect_tx_elect(&full[stage], kRABytes + b_bytes);
            tma_load_2d_elect(st, &tmX, &full[stage], ks * kRRowBytes, m0, pol_x);
            tma_load_2d_elect(st + kRABytes, &tmW, &full[stage], ks * kRRowBytes, 0, pol_w);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == kRStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (failed) {
            if (lane == 0) set_device_error(err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            for (int s = 0; s < kRStages; ++s) {
                if (issued & (1u << s)) mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, kWaitBudgetCycles);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (warp-uniform)
        const uint32_t idesc = idesc_bf16(kRBM, E);
        int stage = 0;
        uint32_t phase = 0;
        bool failed = false, issued_any = false;
        for (int ks = ks0; ks < ks0 + ks_per; ++ks) {
            const bool ok = mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitBudgetCycles);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                failed = true;
                break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + stage * kRStageBytes);
            const uint64_t adesc = sdesc_k_swizzled<128>(st);
            const uint64_t bdesc = sdesc_k_swizzled<128>(st + kRABytes);
#pragma unroll
            for (int j = 0; j < 4; ++j)   // K = 16 BF16 (32 bytes) per MMA
                tc_mma_bf16_elect(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (ks != ks0 || j != 0) ? 1u : 0u);
            issued_any = true;
            tc_commit_elect(&empty[stage]);
            if (++stage == kRStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!failed) {
            tc_commit_elect(tmem_full);
        } else {
            if (lane == 0) set_device_error(err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            if (issued_any) {   // let the issued MMAs finish before TMEM is released
                tc_commit_elect(tmem_full);
                mbar_wait_bounded(tmem_full, 0, nullptr, kWaitBudgetCycles);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ partial logits to shared memory
        const int q = warp & 3;                             // TMEM lane quarter
        const int r = q * 32 + lane;                        // row of the tile
        const bool ok = mbar_wait_bounded(tmem_full, 0, abort_flag, kWaitBudgetCycles);
        if (ks_per == 0) {                                  // an empty quarter adds zeros
            for (int c = 0; c < E; ++c) part[r * row_stride + c] = 0.0f;
        } else if (!__all_sync(0xFFFFFFFFu, ok)) {
            if (lane == 0) set_device_error(err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        } else {
            tc_fence_after();
            // every MMA has completed, so no copy or MMA touches the stage buffers any more
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
            float* row = part + r * row_stride;
            for (int c = 0; c < E; c += 16) {                // E % 16 == 0
                uint32_t v[16];
                tmem_ld_32x32b_x16(taddr + c, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) row[c + i] = __uint_as_float(v[i]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_barrier();                                      // every CTA's partial logits are in place

    {
        // ------------------------------------------------------------ sum, top-k, probabilities
        // This CTA's rows 32*split .. +31 of the tile, on all eight warps.  First the sums: warp w
        // adds rows w, w + 8, ... over the four quarters' partials in quarter order, its lanes
        // over consecutive experts (each read of a peer's shared memory is 128 contiguous
        // bytes), into a local copy lg.  Then eight threads per token: thread q holds the
        // selection keys of experts 4q + j + 32i (j < 4; with the row stride E + 1 the 32 lanes
        // of a warp, 4 tokens x 8 threads, read 32 different banks) and sorts them once; each
        // round three shuffles find the largest head of the token's eight sorted lists, and the
        // thread holding it moves on, so every thread knows every pick.
        float* lg = reinterpret_cast<float*>(smem + kRLogitOff);
        {
            uint32_t peer[kRSplit];
#pragma unroll
            for (int s = 0; s < kRSplit; ++s) peer[s] = cluster_map(smem_u32(part), static_cast<uint32_t>(s));
            bool finite = true;
            constexpr int kChunks = kPer / 4;               // 32-expert chunks of a row (E <= 8 kPer)
            for (int ri = warp; ri < 32; ri += kRWarps) {
                const int r = 32 * static_cast<int>(split) + ri;
                const int64_t t = m0 + r;
                float pv[kChunks][kRSplit];                   // all of the row's loads in flight at once
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const int e = 32 * c + lane;
#pragma unroll
                    for (int s = 0; s < kRSplit; ++s)
                        pv[c][s] = e < E ? ld_cluster_f32(peer[s] + static_cast<uint32_t>(r * row_stride + e) * 4u) : 0.0f;
                }
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const int e = 32 * c + lane;
                    if (e < E) {
                        float a = pv[c][0];
#pragma unroll
                        for (int s = 1; s < kRSplit; ++s) a = __fadd_rn(a, pv[c][s]);
                        lg[ri * row_stride + e] = a;
                        if (t < T) {
                            finite = finite && (__float_as_uint(a) & 0x7F800000u) != 0x7F800000u;
                            if (logits != nullptr) logits[t * E + e] = a;
                        }
                    }
                }
            }
            if (!finite) set_device_error(err, NVFP4_ERR_NONFINITE);
        }
        __syncthreads();                                    // every row's sums are in lg
        const int ti = threadIdx.x >> 3, q = threadIdx.x & 7;
        const int r = 32 * static_cast<int>(split) + ti;
        const int64_t t = m0 + r;
        unsigned long long key[kPer];
#pragma unroll
        for (int i = 0; i < kPer / 4; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = 4 * q + j + 32 * i;
                key[4 * i + j] = e < E ? select_key(lg[ti * row_stride + e], e) : 0ull;
            }
        }
        float* pick_v = reinterpret_cast<float*>(smem + kRPickOff) + ti * 32;
        int* pick_id = reinterpret_cast<int*>(smem + kRPickOff + 32 * 32 * 4) + ti * 32;
        // the thread's keys in descending order (bitonic network, compile-time indices)
#pragma unroll
        for (int size = 2; size <= kPer; size <<= 1) {
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int l = i ^ stride;
                    if (l > i) {
                        const bool desc = (i & size) == 0;   // this pair's direction in the merge
                        const unsigned long long a = key[i], b = key[l];
                        const bool swap = desc ? (a < b) : (a > b);
                        key[i] = swap ? b : a;
                        key[l] = swap ? a : b;
                    }
                }
            }
        }
        // k rounds: the largest head of the token's eight lists is the next pick; its owner
        // moves on to its next key
        for (int j = 0; j < k; ++j) {
            unsigned long long best = key[0];
#pragma unroll
            for (int o = 1; o <= 4; o <<= 1) {
                const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
                best = other > best ? other : best;
            }
            if (best != 0ull && key[0] == best) {
#pragma unroll
                for (int m = 0; m + 1 < kPer; ++m) key[m] = key[m + 1];
                key[kPer - 1] = 0ull;
            }
            if (q == 0) {
                pick_v[j] = best != 0ull ? key_logit(best) : -INFINITY;
                pick_id[j] = best != 0ull ? static_cast<int>(~static_cast<uint32_t>(best)) : -1;
            }
        }
        __syncwarp();
        // p_j = exp(l_j - l_1) / sum over the picks in slot order, in FP32 (each of the token's
        // threads sums the same terms in the same order); thread q writes slots q, q + 8, ...
        const float l1 = pick_id[0] < 0 ? 0.0f : pick_v[0];
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, pick_id[j] < 0 ? 0.0f : expf(__fsub_rn(pick_v[j], l1)));
        if (t < T) {
            for (int j = q; j < k; j += 8) {
                const int id = pick_id[j];
                ids[t * k + j] = id < 0 ? 0 : id;
                probs[t * k + j] = id < 0 ? 0.0f : __fdiv_rn(expf(__fsub_rn(pick_v[j], l1)), sum);
            }
        }
    }

    cluster_barrier();                                      // the peers are done reading this CTA's shared memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kRTmemCols);
    }
}

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

// 2D byte map over a BF16 matrix [rows][H]: boxes of box_rows rows x 128 bytes, 128B swizzle.
bool make_bf16_map(CUtensorMap* m, const void* base, int64_t rows, int H, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * H), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * H)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kRRowBytes), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
std::mutex g_router_mutex;
bool g_router_attr[kMaxDevices];

}  // namespace

cudaError_t launch_router_topk(const uint16_t* x, int64_t T, int H, const uint16_t* w, int E, int k, int32_t* ids,
                               float* probs, float* logits, int* err, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_router_mutex);
        if (!g_router_attr[dev]) {
            e = cudaFuncSetAttribute(router_topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(router_topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
            if (e != cudaSuccess) return e;
            g_router_attr[dev] = true;
        }
    }
    CUtensorMap mx, mw;
    if (!make_bf16_map(&mx, x, T, H, kRBM) || !make_bf16_map(&mw, w, E, H, E)) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>((T + kRBM - 1) / kRBM * kRSplit);   // whole clusters
    if (E <= 128)
        return launch_pdl(false, router_topk_kernel<16>, grid, kRThreads, kRSmemBytes, st, mx, mw, T, H, E, k, ids,
                          probs, logits, err);
    return launch_pdl(false, router_topk_kernel<32>, grid, kRThreads, kRSmemBytes, st, mx, mw, T, H, E, k, ids, probs,
                      logits, err);
}

}  // namespace nvfp4
