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
// Kernel (sm_103a): one CTA per 128-token tile.  Warp 0 loads the tile's X rows and all of W_r
// through TMA (128 bytes of K per row per stage, 128B swizzle, 4-stage ring); warp 1 issues
// tcgen05.mma.kind::f16 (M=128, N=E, K=16) into an FP32 TMEM accumulator, walking K from 0 to
// H-1 in one fixed order whatever T is; warps 2-5, one token per thread, copy the token's E
// logits from TMEM into registers (E <= 128) or into the (then idle) stage buffers, select the
// top k in k passes and write ids and probabilities.  All waits are bounded (NVFP4_ERR_DEVICE_TIMEOUT, then a clean exit).
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kRStages = 4;
constexpr int kRBM = 128;                               // tokens per CTA
constexpr int kRRowBytes = 128;                         // bytes of K per row per stage (64 BF16)
constexpr int kRMaxE = 256;
constexpr int kRABytes = kRBM * kRRowBytes;             // 16 KB
constexpr int kRBBytes = kRMaxE * kRRowBytes;           // room for 256 expert rows
constexpr int kRStageBytes = kRABytes + kRBBytes;       // 48 KB
constexpr int kRBarOff = kRStages * kRStageBytes;
constexpr int kRSmemBytes = kRBarOff + 128 + 1024;
constexpr int kRThreads = 192;                          // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kRTmemCols = 256;
// epilogue staging in the stage buffers: 128 rows of E logits (stride E+1 floats: no bank
// conflicts when the threads read one column), then 128 rows of 32 selected ids
constexpr int kRIdsOff = kRBM * (kRMaxE + 1) * 4;
constexpr int kRSelVOff = kRIdsOff + kRBM * 32 * 4;      // then 128 rows of 32 selected logits
static_assert(kRSelVOff + kRBM * 32 * 4 <= kRBarOff, "epilogue staging fits in the stage buffers");
constexpr int kRRegE = 128;                               // up to this many experts: logits in registers

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

// (va, ia) comes before (vb, ib) in the selection order
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(kRThreads, 1)
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
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
    const int num_ks = H / 64;
    const int m0 = static_cast<int>(blockIdx.x) * kRBM;
    const uint32_t b_bytes = static_cast<uint32_t>(E) * kRRowBytes;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (warp-uniform)
        const uint64_t pol_x = policy_evict_first();
        const uint64_t pol_w = policy_evict_last();
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_parity = 0;
        bool failed = false;
        for (int ks = 0; ks < num_ks; ++ks) {
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
        for (int ks = 0; ks < num_ks; ++ks) {
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
                tc_mma_bf16_elect(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (ks | j) != 0 ? 1u : 0u);
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
    } else {
        // ------------------------------------------------------------ epilogue: one token per thread
        const int q = warp & 3;                             // TMEM lane quarter
        const int r = q * 32 + lane;                        // row of the tile
        const int64_t t = m0 + r;
        const bool ok = mbar_wait_bounded(tmem_full, 0, abort_flag, kWaitBudgetCycles);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            if (lane == 0) set_device_error(err, NVFP4_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        } else {
            tc_fence_after();
            // every MMA has completed, so no copy or MMA touches the stage buffers any more
            int32_t* sel = reinterpret_cast<int32_t*>(smem + kRIdsOff) + r * 32;
            float* selv = reinterpret_cast<float*>(smem + kRSelVOff) + r * 32;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
            bool finite = true;
            // one 16-column chunk of the token's logits from TMEM (E % 16 == 0: every column
            // read is a logit), optionally stored to the logits output
            auto load16 = [&](int c, uint32_t (&v)[16]) {
                tmem_ld_32x32b_x16(taddr + c, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) finite = finite && (v[i] & 0x7F800000u) != 0x7F800000u;
                if (logits != nullptr && t < T) {
                    float* dst = logits + t * E + c;    // 64-byte aligned (E % 16 == 0, base 32-aligned)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 8 * u),
                                     "r"(v[8 * u]), "r"(v[8 * u + 1]), "r"(v[8 * u + 2]), "r"(v[8 * u + 3]),
                                     "r"(v[8 * u + 4]), "r"(v[8 * u + 5]), "r"(v[8 * u + 6]), "r"(v[8 * u + 7])
                                     : "memory");
                    }
                }
            };
            // k passes; each takes the first entry (in selection order) after the previous
            // pick, scanning in eight independent chains (columns e = 8m + u) merged at the
            // end: the same pick as one chain over all columns, with 8x shorter dependencies
            auto merge = [&](const float (&bv)[8], const int (&bid)[8], float& best_v, int& best_id) {
                best_v = bv[0];
                best_id = bid[0];
#pragma unroll
                for (int u = 1; u < 8; ++u) {
                    if (bid[u] >= 0 && (best_id < 0 || before(bv[u], bid[u], best_v, best_id))) {
                        best_v = bv[u];
                        best_id = bid[u];
                    }
                }
            };
            if (E <= kRRegE) {
                // logits in registers (E <= 128)
                float lv[kRRegE];
#pragma unroll
                for (int c = 0; c < kRRegE / 16; ++c) {
                    if (16 * c < E) {
                        uint32_t v[16];
                        load16(16 * c, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) lv[16 * c + i] = __uint_as_float(v[i]);
                    }
                }
                if (t < T) {
                    float pv = INFINITY;
                    int pid = -1;
                    for (int j = 0; j < k; ++j) {
                        float bv[8];
                        int bid[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            bv[u] = -INFINITY;
                            bid[u] = -1;
                        }
#pragma unroll
                        for (int e = 0; e < kRRegE; ++e) {
                            if (e < E) {
                                const int u = e & 7;
                                const float v = lv[e];
                                const bool after = v < pv || (v == pv && e > pid);
                                if (after && (bid[u] < 0 || before(v, e, bv[u], bid[u]))) {
                                    bv[u] = v;
                                    bid[u] = e;
                                }
                            }
                        }
                        merge(bv, bid, pv, pid);
                        sel[j] = pid;
                        selv[j] = pv;
                    }
                }
            } else {
                // logits staged in shared memory (rows of stride E+1 floats: no bank conflicts)
                float* row = reinterpret_cast<float*>(smem) + r * (kRMaxE + 1);
                for (int c = 0; c < E; c += 16) {
                    uint32_t v[16];
                    load16(c, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) row[c + i] = __uint_as_float(v[i]);
                }
                if (t < T) {
                    float pv = INFINITY;
                    int pid = -1;
                    for (int j = 0; j < k; ++j) {
                        float bv[8];
                        int bid[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            bv[u] = -INFINITY;
                            bid[u] = -1;
                        }
                        for (int e0 = 0; e0 < E; e0 += 8) {   // E % 16 == 0
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const int e = e0 + u;
                                const float v = row[e];
                                const bool after = v < pv || (v == pv && e > pid);
                                if (after && (bid[u] < 0 || before(v, e, bv[u], bid[u]))) {
                                    bv[u] = v;
                                    bid[u] = e;
                                }
                            }
                        }
                        merge(bv, bid, pv, pid);
                        sel[j] = pid;
                        selv[j] = pv;
                    }
                }
            }
            if (t < T) {
                if (!finite) set_device_error(err, NVFP4_ERR_NONFINITE);
                const float l1 = sel[0] < 0 ? 0.0f : selv[0];
                float sum = 0.0f;
                for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, sel[j] < 0 ? 0.0f : expf(__fsub_rn(selv[j], l1)));
                for (int j = 0; j < k; ++j) {
                    const int id = sel[j];
                    ids[t * k + j] = id < 0 ? 0 : id;
                    probs[t * k + j] = id < 0 ? 0.0f : __fdiv_rn(expf(__fsub_rn(selv[j], l1)), sum);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
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
            e = cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
            if (e != cudaSuccess) return e;
            g_router_attr[dev] = true;
        }
    }
    CUtensorMap mx, mw;
    if (!make_bf16_map(&mx, x, T, H, kRBM) || !make_bf16_map(&mw, w, E, H, E)) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>((T + kRBM - 1) / kRBM);
    return launch_pdl(false, router_topk_kernel, grid, kRThreads, kRSmemBytes, st, mx, mw, T, H, E, k, ids, probs,
                      logits, err);
}

}  // namespace nvfp4
