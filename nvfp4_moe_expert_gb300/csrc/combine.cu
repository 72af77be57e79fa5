// Fixed-order top-k combine: out[t, :] = bf16( ((0 + y[t,0,:]) + y[t,1,:]) + ... + y[t,k-1,:] )
// with FP32 additions in top-k slot order.
//
// "Finishing RL training faster: bitwise consistency, high performance,
// agent-driven" (spke.com/ko/ai/article/3192), section 4.5 "Cross-GPU
// reduction": expert outputs are accumulated in FP32 in top-k slot order on
// the token's owner; "miniTE diagnoses and narrows the cross-engine execution
// gap of NVFP4 RL", section "How it differs": the combine order survives
// padding, quantisation and cast.  The router probability was already
// applied before FC2, so the combine is a plain sum.
//
// The forward's y holds one row per routed row (FC2 writes each tile's rows contiguously);
// rows[t*k + s] names the row of token t's slot s (-1 for a pair the fixed-capacity layout
// dropped, which adds nothing).  The backward's dX pairs are in (token, slot) order (rows =
// nullptr).
//
// HBM-bound: each thread owns 8 consecutive columns of one token (16-byte
// loads of the k slot rows, all issued before the adds, one 16-byte store);
// a grid-stride loop over T*H/8 such vectors keeps every access coalesced.
#include "common.cuh"

namespace nvfp4 {
namespace {

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// kMaxK > 0: k <= kMaxK slots, all loads issued before the adds (more bytes in flight).
template <int kMaxK>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ rows,
                                                      int64_t T, int k, int H, uint16_t* __restrict__ out) {
    const int vec_per_row = H / 8;
    const int64_t nvec = T * vec_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    // the row numbers of the next vector are loaded while this vector's rows are in flight
    int32_t rn[kMaxK];
    auto load_rows = [&](int64_t i) {
        const int64_t t = i / vec_per_row;
#pragma unroll
        for (int s = 0; s < kMaxK; ++s) {
            if (s < k) rn[s] = rows ? __ldg(rows + t * k + s) : static_cast<int32_t>(t * k + s);
        }
    };
    // The first ones even before the wait: the row map comes from the route sort, which is
    // complete once the kernel before this one (FC2, which triggers after its own wait) has
    // started; y is read only after the wait.
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < nvec) load_rows(i);
    pdl_wait();
    pdl_launch_dependents();
    for (; i < nvec; i += stride) {
        const int64_t t = i / vec_per_row;
        const int v = static_cast<int>(i - t * vec_per_row);
        int32_t r[kMaxK];
#pragma unroll
        for (int s = 0; s < kMaxK; ++s) r[s] = rn[s];
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        uint4 w[kMaxK];
#pragma unroll
        for (int s = 0; s < kMaxK; ++s) {
            if (s < k && r[s] >= 0) w[s] = __ldcs(reinterpret_cast<const uint4*>(y + static_cast<int64_t>(r[s]) * H) + v);
        }
        if (i + stride < nvec) load_rows(i + stride);
#pragma unroll
        for (int s = 0; s < kMaxK; ++s) {          // slots in top-k order
            if (s < k && r[s] >= 0) {
                const uint32_t ws[4] = {w[s].x, w[s].y, w[s].z, w[s].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[2 * j] = __fadd_rn(acc[2 * j], __uint_as_float(ws[j] << 16));
                    acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __uint_as_float(ws[j] & 0xFFFF0000u));
                }
            }
        }
        uint4 o;
        o.x = bf16x2_rn(acc[0], acc[1]);
        o.y = bf16x2_rn(acc[2], acc[3]);
        o.z = bf16x2_rn(acc[4], acc[5]);
        o.w = bf16x2_rn(acc[6], acc[7]);
        reinterpret_cast<uint4*>(out + t * H)[v] = o;
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* y, const int32_t* rows, int64_t T, int k, int H, uint16_t* out,
                           cudaStream_t st, bool pdl) {
    const int64_t nvec = T * (H / 8);
    if (nvec == 0) return cudaSuccess;
    int64_t blocks = (nvec + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 g(static_cast<unsigned>(blocks));
    if (k <= 2) return launch_pdl(pdl, combine_kernel<2>, g, 256, 0, st, y, rows, T, k, H, out);
    if (k <= 4) return launch_pdl(pdl, combine_kernel<4>, g, 256, 0, st, y, rows, T, k, H, out);
    if (k <= 8) return launch_pdl(pdl, combine_kernel<8>, g, 256, 0, st, y, rows, T, k, H, out);
    if (k <= 16) return launch_pdl(pdl, combine_kernel<16>, g, 256, 0, st, y, rows, T, k, H, out);
    return launch_pdl(pdl, combine_kernel<32>, g, 256, 0, st, y, rows, T, k, H, out);
}

}  // namespace nvfp4
