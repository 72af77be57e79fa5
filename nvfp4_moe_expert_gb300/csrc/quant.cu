// NVFP4 quantisers: plain row quantisation (weights or any rows), the fused
// route sort + per-token amax + pad + quantise of the FC1 input, and the
// requantisation of the FC2 input.
//
// Two-level NVFP4 as defined on "miniTE diagnoses and narrows the
// cross-engine execution gap of NVFP4 RL", section "How it differs":
// g = max|row| / (6*448) in FP32, an E4M3 scale per 16 elements, E2M1 codes,
// round-to-nearest-even.  Block scale s_b = e4m3(bmax / (g*6)), code =
// e2m1(x / (g*s_b)), both divisions IEEE binary32 in that two-step form.
// The route sort follows section "How to use it": the tokens are sorted by
// expert and the row maximum is taken in the same pass that quantises the
// row, so X is read exactly once.
//
// One warp owns one row.  Lane l holds the 16-byte vectors l, l+32, l+64, ...
// of the row (8 BF16 each); a 16-element block is the vector pair (2b, 2b+1),
// held by lanes 2j and 2j+1.  Stores are 4 bytes of codes per vector per lane
// (128 contiguous bytes per warp instruction) and one 32-bit word of four
// block scales per 64 columns, at the position the GEMM's scale-factor tile
// layout gives it.
#include <cfloat>

#include "common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kRouteChunk = 256;   // tokens per route-sort chunk (8 warps x 32 tokens)

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int VPL>
struct QuantRow {
    uint32_t code[VPL];   // 8 nibbles per vector
    uint32_t sfw[VPL];    // valid on lanes with (lane & 7) == 0: scales of 4 blocks
    float g;
    bool finite;
};

// Quantise the row held as `xv` (lane's vectors; `nvec` vectors in the row).
// If `amax_in` >= 0 it is used as max|row| (it must be that maximum).
template <int VPL>
__device__ __forceinline__ void quantize_warp_row(const uint4 (&xv)[VPL], int nvec, float amax_in,
                                                  QuantRow<VPL>& q) {
    const int lane = threadIdx.x & 31;
    float vmax[VPL];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(bf16_lo(w[j])));
            m = fmaxf(m, fabsf(bf16_hi(w[j])));
        }
        // fmaxf drops NaN: remember non-finite inputs separately
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            bad |= ((w[j] & 0x7F80u) == 0x7F80u) || ((w[j] & 0x7F800000u) == 0x7F800000u);
        }
        if (bad) m = __int_as_float(0x7F800000);
        vmax[i] = m;
        amax = fmaxf(amax, m);
    }
    if (amax_in >= 0.0f) {
        amax = amax_in;
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    }
    q.finite = amax <= FLT_MAX;
    const float g = q.finite ? __fdiv_rn(amax, kOuterDivisor) : 0.0f;
    q.g = g;
    const float d1 = __fmul_rn(g, 6.0f);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const float bmax = fmaxf(vmax[i], __shfl_xor_sync(0xFFFFFFFFu, vmax[i], 1));
        const float r = d1 > 0.0f ? __fdiv_rn(bmax, d1) : 0.0f;
        const uint32_t s_code = (d1 > 0.0f && q.finite) ? cvt_e4m3(r) : 0u;
        const float d2 = __fmul_rn(g, e4m3_value(s_code));
        uint32_t word = 0;
        if (d2 > 0.0f) {
            const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
            uint32_t signs = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
                word |= cvt_e2m1x2(__fdiv_rn(a, d2), __fdiv_rn(b, d2)) << (8 * j);
                signs |= ((w[j] >> 15) & 1u) << (8 * j + 3);
                signs |= ((w[j] >> 31) & 1u) << (8 * j + 7);
            }
            // the sign bit of every code is the sign of x (also when the magnitude rounds to 0)
            word = (word & 0x77777777u) | signs;
        }
        q.code[i] = word;
        // gather the four block scales of this lane's 64-column group
        const int base = lane & ~7;
        const uint32_t s0 = __shfl_sync(0xFFFFFFFFu, s_code, base + 0);
        const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, s_code, base + 2);
        const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, s_code, base + 4);
        const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, s_code, base + 6);
        q.sfw[i] = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
    }
    (void)nvec;
}

template <int VPL>
__device__ __forceinline__ void load_warp_row(const uint16_t* src, int nvec, uint4 (&xv)[VPL]) {
    const int lane = threadIdx.x & 31;
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int v = lane + 32 * i;
        xv[i] = v < nvec ? __ldg(s + v) : make_uint4(0, 0, 0, 0);
    }
}

// Write a quantised row as row `r` of an NVFP4 matrix with `cols` columns.
template <int VPL>
__device__ __forceinline__ void store_warp_row(const QuantRow<VPL>& q, int nvec, int64_t r, int cols,
                                               uint8_t* codes, uint8_t* sf) {
    const int lane = threadIdx.x & 31;
    uint32_t* crow = reinterpret_cast<uint32_t*>(codes + r * static_cast<int64_t>(cols / 2));
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int v = lane + 32 * i;
        if (v < nvec) {
            crow[v] = q.code[i];
            if ((lane & 7) == 0) {
                *reinterpret_cast<uint32_t*>(sf + sf_offset(r, v / 2, cols)) = q.sfw[i];
            }
        }
    }
}

// Zero the scales (and optionally the codes) of row r.
__device__ __forceinline__ void zero_warp_row(int64_t r, int cols, uint8_t* codes, uint8_t* sf, bool zero_codes) {
    const int lane = threadIdx.x & 31;
    const int ngroups = cols / 64;
    for (int q = lane; q < ngroups; q += 32) {
        *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * q, cols)) = 0u;
    }
    if (zero_codes) {
        uint4* crow = reinterpret_cast<uint4*>(codes + r * static_cast<int64_t>(cols / 2));
        for (int v = lane; v < cols / 32; v += 32) crow[v] = make_uint4(0, 0, 0, 0);
    }
}

// ------------------------------------------------------------------ plain rows
template <int VPL>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                            int cols, int64_t ld, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ sf, float* __restrict__ g,
                                                            int* err) {
    const int nvec = cols / 8;
    const int64_t rows_pad = (rows + kTileM - 1) / kTileM * kTileM;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows_pad; r += nwarps) {
        if (r >= rows) {
            zero_warp_row(r, cols, codes, sf, true);
            continue;
        }
        uint4 xv[VPL];
        load_warp_row<VPL>(x + r * ld, nvec, xv);
        QuantRow<VPL> q;
        quantize_warp_row<VPL>(xv, nvec, -1.0f, q);
        if (!q.finite && (threadIdx.x & 31) == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
        store_warp_row<VPL>(q, nvec, r, cols, codes, sf);
        if ((threadIdx.x & 31) == 0) g[r] = q.g;
    }
}

// ------------------------------------------------------------------ route sort
// Per 256-token chunk: per-expert pair counts, and each pair's rank among the
// chunk's pairs of the same expert in (token, slot) order.
__global__ void __launch_bounds__(256) route_hist_rank_kernel(const int32_t* __restrict__ ids, int64_t T, int E,
                                                               int k, int64_t n_chunks,
                                                               int32_t* __restrict__ chunk_count,
                                                               int32_t* __restrict__ pair_rank, int* err) {
    extern __shared__ int32_t wcount[];   // [8][E]
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t chunk = blockIdx.x;
    for (int i = threadIdx.x; i < kWarpsPerBlock * E; i += blockDim.x) wcount[i] = 0;
    __syncthreads();
    const int64_t tok0 = chunk * kRouteChunk + w * 32;
    const int64_t npairs = T * k;
    const unsigned lt_mask = (1u << lane) - 1u;
    int my_e[32];
    int my_rank[32];
#pragma unroll
    for (int it = 0; it < 32; ++it) {
        if (it < k) {
            const int64_t p = tok0 * k + it * 32 + lane;
            int e = -1;
            if (p < npairs && tok0 < T) {
                e = ids[p];
                if (e < 0 || e >= E) {
                    set_device_error(err, NVFP4_ERR_BAD_EXPERT_ID);
                    e = -1;
                }
            }
            const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
            const int before = __popc(m & lt_mask);
            const int base = e >= 0 ? wcount[w * E + e] : 0;
            __syncwarp();
            if (e >= 0 && before == 0) wcount[w * E + e] = base + __popc(m);
            __syncwarp();
            my_e[it] = e;
            my_rank[it] = base + before;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int ww = 0; ww < kWarpsPerBlock; ++ww) {
            const int c = wcount[ww * E + e];
            wcount[ww * E + e] = run;
            run += c;
        }
        chunk_count[static_cast<int64_t>(e) * n_chunks + chunk] = run;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 32; ++it) {
        if (it < k && my_e[it] >= 0) {
            const int64_t p = tok0 * k + it * 32 + lane;
            pair_rank[p] = wcount[w * E + my_e[it]] + my_rank[it];
        }
    }
}

// One block: per-expert totals, padded expert offsets, and each chunk's first row.
__global__ void __launch_bounds__(1024) route_scan_kernel(int E, int64_t n_chunks,
                                                          const int32_t* __restrict__ chunk_count,
                                                          int32_t* __restrict__ chunk_base,
                                                          int32_t* __restrict__ expert_count,
                                                          int32_t* __restrict__ offsets) {
    __shared__ int32_t seg_sum[1024];
    __shared__ int32_t e_off[1025];
    const int tid = threadIdx.x;
    const int S = blockDim.x / E;                  // threads per expert (>= 1)
    const int e = tid / S, seg = tid % S;
    const int64_t L = (n_chunks + S - 1) / S;
    const int64_t c0 = seg * L, c1 = min(n_chunks, c0 + L);
    int32_t sum = 0;
    if (e < E) {
        const int32_t* cc = chunk_count + static_cast<int64_t>(e) * n_chunks;
        for (int64_t c = c0; c < c1; ++c) sum += cc[c];
    }
    seg_sum[tid] = sum;
    __syncthreads();
    if (e < E && seg == 0) {
        int32_t run = 0;
        for (int s = 0; s < S; ++s) {
            const int32_t v = seg_sum[tid + s];
            seg_sum[tid + s] = run;
            run += v;
        }
        expert_count[e] = run;
        e_off[e] = (run + kTileM - 1) / kTileM * kTileM;   // padded size for now
    }
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int i = 0; i < E; ++i) {
            const int32_t v = e_off[i];
            e_off[i] = run;
            run += v;
        }
        e_off[E] = run;
    }
    __syncthreads();
    for (int i = tid; i <= E; i += blockDim.x) offsets[i] = e_off[i];
    if (e < E) {
        int32_t run = e_off[e] + seg_sum[tid];
        const int32_t* cc = chunk_count + static_cast<int64_t>(e) * n_chunks;
        int32_t* cb = chunk_base + static_cast<int64_t>(e) * n_chunks;
        for (int64_t c = c0; c < c1; ++c) {
            cb[c] = run;
            run += cc[c];
        }
    }
}

template <int VPL>
__global__ void __launch_bounds__(256) route_quant_scatter_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int E, int k, const int32_t* __restrict__ ids,
    const float* __restrict__ probs, const int32_t* __restrict__ offsets, RouteBufs b, int* err) {
    const int lane = threadIdx.x & 31;
    const int nvec = H / 8;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = warp; t < T; t += nwarps) {
        uint4 xv[VPL];
        load_warp_row<VPL>(x + t * H, nvec, xv);
        QuantRow<VPL> q;
        quantize_warp_row<VPL>(xv, nvec, -1.0f, q);
        if (!q.finite && lane == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
        const int64_t chunk = t / kRouteChunk;
        for (int j = 0; j < k; ++j) {
            const int64_t p = t * k + j;
            const int e = __ldg(ids + p);
            if (e < 0 || e >= E) continue;   // reported by the histogram kernel
            const int64_t r = b.chunk_base[static_cast<int64_t>(e) * b.n_chunks + chunk] + b.pair_rank[p];
            store_warp_row<VPL>(q, nvec, r, H, b.a_codes, b.a_sf);
            if (lane == 0) {
                b.a_g[r] = q.g;
                b.row_pair[r] = static_cast<int32_t>(p);
                b.row_prob[r] = __ldg(probs + p);
                b.amax2[r] = 0u;
            }
        }
    }
    // pad rows: expert e's rows [offsets[e] + count_e, offsets[e+1])
    const int64_t pad_slots = static_cast<int64_t>(E) * kTileM;
    for (int64_t s = warp; s < pad_slots; s += nwarps) {
        const int e = static_cast<int>(s / kTileM), j = static_cast<int>(s % kTileM);
        const int64_t r = static_cast<int64_t>(offsets[e]) + b.expert_count[e] + j;
        if (r >= offsets[e + 1]) continue;
        zero_warp_row(r, H, b.a_codes, b.a_sf, false);
        if (lane == 0) {
            b.a_g[r] = 0.0f;
            b.row_pair[r] = -1;
            b.row_prob[r] = 0.0f;
            b.amax2[r] = 0u;
        }
    }
}

// ------------------------------------------------------------------ requant
template <int VPL>
__global__ void __launch_bounds__(256) requant_kernel(const uint16_t* __restrict__ h,
                                                      const uint32_t* __restrict__ amax2,
                                                      const int32_t* __restrict__ row_pair,
                                                      const int32_t* __restrict__ offsets, int E, int I,
                                                      uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                      float* __restrict__ g, int* err) {
    const int lane = threadIdx.x & 31;
    const int nvec = I / 8;
    const int64_t rows = offsets[E];
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows; r += nwarps) {
        if (row_pair[r] < 0) {
            zero_warp_row(r, I, codes, sf, false);
            if (lane == 0) g[r] = 0.0f;
            continue;
        }
        uint4 xv[VPL];
        load_warp_row<VPL>(h + r * I, nvec, xv);
        QuantRow<VPL> q;
        quantize_warp_row<VPL>(xv, nvec, __uint_as_float(amax2[r]), q);
        if (!q.finite && lane == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
        store_warp_row<VPL>(q, nvec, r, I, codes, sf);
        if (lane == 0) g[r] = q.g;
    }
}

int grid_for_warps(int64_t warps) {
    const int64_t blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

// Dispatch on the number of 16-byte vectors each lane holds.
#define NVFP4_VPL_DISPATCH(nvec, KERNEL, ...)                                       \
    do {                                                                            \
        const int vpl_ = ((nvec) + 31) / 32;                                        \
        if (vpl_ <= 1) KERNEL<1> __VA_ARGS__;                                       \
        else if (vpl_ <= 2) KERNEL<2> __VA_ARGS__;                                  \
        else if (vpl_ <= 4) KERNEL<4> __VA_ARGS__;                                  \
        else if (vpl_ <= 8) KERNEL<8> __VA_ARGS__;                                  \
        else if (vpl_ <= 16) KERNEL<16> __VA_ARGS__;                                \
        else KERNEL<32> __VA_ARGS__;                                                \
    } while (0)

cudaError_t launch_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                                 uint8_t* sf, float* g, int* err, cudaStream_t st) {
    const int64_t rows_pad = (rows + kTileM - 1) / kTileM * kTileM;
    if (rows_pad == 0) return cudaSuccess;
    const int grid = grid_for_warps(rows_pad);
    const int c = static_cast<int>(cols);
    NVFP4_VPL_DISPATCH(c / 8, quantize_rows_kernel, <<<grid, 256, 0, st>>>(x, rows, c, ld, codes, sf, g, err));
    return cudaGetLastError();
}

cudaError_t launch_route_sort_quant(const uint16_t* x, int64_t T, int H, int E, int k, const int32_t* ids,
                                    const float* probs, int32_t* offsets, const RouteBufs& b, int* err,
                                    cudaStream_t st) {
    if (T == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    const size_t smem = sizeof(int32_t) * kWarpsPerBlock * E;
    route_hist_rank_kernel<<<static_cast<unsigned>(b.n_chunks), 256, smem, st>>>(ids, T, E, k, b.n_chunks,
                                                                                 b.chunk_count, b.pair_rank, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    route_scan_kernel<<<1, 1024, 0, st>>>(E, b.n_chunks, b.chunk_count, b.chunk_base, b.expert_count, offsets);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t warps = T > static_cast<int64_t>(E) * kTileM ? T : static_cast<int64_t>(E) * kTileM;
    const int grid = grid_for_warps(warps);
    NVFP4_VPL_DISPATCH(H / 8, route_quant_scatter_kernel,
                       <<<grid, 256, 0, st>>>(x, T, H, E, k, ids, probs, offsets, b, err));
    return cudaGetLastError();
}

cudaError_t launch_requant(const uint16_t* h, const uint32_t* amax2, const int32_t* row_pair,
                           const int32_t* offsets, int E, int64_t rows_cap, int I, uint8_t* codes, uint8_t* sf,
                           float* g, int* err, cudaStream_t st) {
    const int grid = grid_for_warps(rows_cap);
    NVFP4_VPL_DISPATCH(I / 8, requant_kernel,
                       <<<grid, 256, 0, st>>>(h, amax2, row_pair, offsets, E, I, codes, sf, g, err));
    return cudaGetLastError();
}

}  // namespace nvfp4
