// NVFP4 quantisers: plain row quantisation (weights or any rows), the fused
// route sort + per-token amax + pad + quantise of the FC1 input, and the
// requantisation of the FC2 input.
//
// Two-level NVFP4 as defined on "miniTE diagnoses and narrows the
// cross-engine execution gap of NVFP4 RL", section "How it differs":
// g = max|row| / (6*448) in FP32, an E4M3 scale per 16 elements, E2M1 codes,
// round-to-nearest-even.  Block scale s_b = e4m3(bmax / (g*6)), code =
// e2m1(x / (g*s_b)), both quotients the correctly rounded binary32 quotient.
// The route sort follows section "How to use it": the tokens are sorted by
// expert and the row maximum is taken in the same pass that quantises the
// row, so X is read exactly once.
//
// Work split: a lane owns whole 64-element groups (four 16-element blocks,
// 128 bytes of BF16): it loads them with 16-byte loads, finds the block
// maxima with NaN-propagating bf16x2 max, and writes 32 bytes of codes plus
// one 32-bit word of four block scales per group, at the place the GEMM's
// scale-factor tile layout gives it.  A row of G groups is spread over G
// lanes (G <= 32: 32/G rows per warp) or over the whole warp (G > 32: G/32
// groups per lane); the row maximum is one redux.sync over the row's lanes.
//
// Division: x / d for the 16 elements of a block that share d = g*s_b uses
// Markstein's method (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 1990; also
// Muller et al., Handbook of Floating-Point Arithmetic, ch. on FMA-based
// division): with y = RN(1/d) from __frcp_rn, q0 = RN(x*y),
// r = x - d*q0 (exact with an FMA) and q = RN(q0 + r*y) equals RN(x/d) when
// no intermediate leaves the normal range.  Divisors below 2^-60 take IEEE
// __fdiv_rn instead, which keeps every quotient that can reach a code
// boundary (|x/d| >= 0.25) in the normal range.
#include <cfloat>

#include "common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kRouteChunk = 256;       // tokens per route-sort chunk (8 warps x 32 tokens)
constexpr float kMarksteinMinDivisor = 8.6736174e-19f;   // 2^-60

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// max|x| over 16 BF16 values (two 16-byte vectors), as FP32 bits; NaN propagates.
__device__ __forceinline__ uint32_t block_absmax_bits(const uint4& a, const uint4& b) {
    constexpr uint32_t kAbs = 0x7FFF7FFFu;
    uint32_t m = bf16x2_max_nan(bf16x2_max_nan(a.x & kAbs, a.y & kAbs), bf16x2_max_nan(a.z & kAbs, a.w & kAbs));
    m = bf16x2_max_nan(m, bf16x2_max_nan(bf16x2_max_nan(b.x & kAbs, b.y & kAbs),
                                         bf16x2_max_nan(b.z & kAbs, b.w & kAbs)));
    m = bf16x2_max_nan(m, m >> 16);      // low half = max of both halves
    return m << 16;                      // BF16 bits -> FP32 bits
}

// RN(x / d) by Markstein's correction step, given rc = RN(1/d) (see the file header).
__device__ __forceinline__ float div_markstein(float x, float d, float rc) {
    const float q0 = __fmul_rn(x, rc);
    return __fmaf_rn(__fmaf_rn(-q0, d, x), rc, q0);
}

// Eight E2M1 codes (RNE, saturating) of eight FP32 values; q[2j] goes to the low nibble of byte j.
__device__ __forceinline__ uint32_t e2m1x8(const float (&q)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return r;
}

// Eight E2M1 codes of one 16-byte vector of BF16 values, quotient by d (rc = RN(1/d)).
__device__ __forceinline__ uint32_t codes8(const uint4& v, float d, float rc, bool markstein) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float q[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
        q[2 * j] = markstein ? div_markstein(lo, d, rc) : __fdiv_rn(lo, d);
        q[2 * j + 1] = markstein ? div_markstein(hi, d, rc) : __fdiv_rn(hi, d);
    }
    const uint32_t mags = e2m1x8(q) & 0x77777777u;
    // sign bit of every code = sign of x (also when the magnitude rounds to 0):
    // byte 1 of w[j] carries element 2j's sign in bit 7, byte 3 element 2j+1's
    const uint32_t t01 = __byte_perm(w[0], w[1], 0x7531), t23 = __byte_perm(w[2], w[3], 0x7531);
    const uint32_t even = __byte_perm(t01, t23, 0x6420), odd = __byte_perm(t01, t23, 0x7531);
    return mags | ((even >> 4) & 0x08080808u) | (odd & 0x80808080u);
}

// Quantised form of one 64-element group.
struct GroupQ {
    uint32_t code[8];   // 64 nibbles, element 2i in the low nibble of byte i
    uint32_t sfw;       // four E4M3 block scales, block 0 in the low byte
};

// Quantise a group with outer scale g (finite); bm = its four block maxima (FP32 bits);
// d1 = RN(6g) and rc1 = RN(1/d1) (or 0 when d1 is too small for the Markstein step).
__device__ __forceinline__ void quantize_group(const uint4 (&v)[8], const uint32_t (&bm)[4], float g, float d1,
                                               float rc1, GroupQ& q) {
    q.sfw = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const float bmx = __uint_as_float(bm[b]);
        const float r = rc1 != 0.0f ? div_markstein(bmx, d1, rc1) : __fdiv_rn(bmx, d1);
        const uint32_t s_code = d1 > 0.0f ? cvt_e4m3(r) : 0u;
        const float d2 = __fmul_rn(g, e4m3_value(s_code));
        q.sfw |= s_code << (8 * b);
        if (d2 > 0.0f) {
            const bool mk = d2 >= kMarksteinMinDivisor;
            const float rc = mk ? __frcp_rn(d2) : 0.0f;
            q.code[2 * b] = codes8(v[2 * b], d2, rc, mk);
            q.code[2 * b + 1] = codes8(v[2 * b + 1], d2, rc, mk);
        } else {
            q.code[2 * b] = 0u;
            q.code[2 * b + 1] = 0u;
        }
    }
}

__device__ __forceinline__ void load_group(const uint16_t* src, uint4 (&v)[8]) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(s + i);
}

__device__ __forceinline__ void store_group(const GroupQ& q, int64_t r, int grp, int cols, uint8_t* codes,
                                            uint8_t* sf) {
    uint4* c = reinterpret_cast<uint4*>(codes + r * static_cast<int64_t>(cols / 2) + grp * 32);
    c[0] = make_uint4(q.code[0], q.code[1], q.code[2], q.code[3]);
    c[1] = make_uint4(q.code[4], q.code[5], q.code[6], q.code[7]);
    *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * grp, cols)) = q.sfw;
}

// Lane layout of rows of G groups: LPR lanes per row, RPW rows per warp pass,
// GPL groups per lane.
struct RowLanes {
    int LPR, RPW, slot, li;
    unsigned mask;
    bool active;
    __device__ RowLanes(int G) {
        const int lane = threadIdx.x & 31;
        LPR = G <= 32 ? G : 32;
        RPW = 32 / LPR;
        slot = lane / LPR;
        li = lane % LPR;
        active = slot < RPW;
        mask = LPR == 32 ? 0xFFFFFFFFu : (((1u << LPR) - 1u) << (slot * LPR));
    }
};

// Quantise the GPL groups this lane owns of the row at `src`; amax_in >= 0 supplies
// max|row| (it must be that maximum).  Returns g; finite = whether the row is finite.
template <int GPL>
__device__ __forceinline__ float quantize_row_lanes(const uint16_t* src, const RowLanes& rl, int G, float amax_in,
                                                    GroupQ (&q)[GPL], bool& finite) {
    uint4 v[GPL][8];
    uint32_t bm[GPL][4];
    uint32_t amax_bits = 0;
#pragma unroll
    for (int i = 0; i < GPL; ++i) {
        const int grp = rl.li + rl.LPR * i;
        if (grp < G) {
            load_group(src + grp * 64, v[i]);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                bm[i][b] = block_absmax_bits(v[i][2 * b], v[i][2 * b + 1]);
                amax_bits = max(amax_bits, bm[i][b]);
            }
        }
    }
    amax_bits = __reduce_max_sync(rl.mask, amax_bits);
    finite = amax_bits < 0x7F800000u;
    float amax = __uint_as_float(amax_bits);
    if (amax_in >= 0.0f) amax = amax_in;
    const float g = finite ? __fdiv_rn(amax, kOuterDivisor) : 0.0f;
    const float d1 = __fmul_rn(g, 6.0f);
    const float rc1 = d1 >= kMarksteinMinDivisor ? __frcp_rn(d1) : 0.0f;
#pragma unroll
    for (int i = 0; i < GPL; ++i) {
        if (rl.li + rl.LPR * i < G) quantize_group(v[i], bm[i], g, d1, rc1, q[i]);
    }
    return g;
}

// ------------------------------------------------------------------ plain rows
template <int GPL>
__global__ void __launch_bounds__(256, GPL == 1 ? 3 : 1) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                            int cols, int64_t ld, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ sf, float* __restrict__ g,
                                                            int* err) {
    const int G = cols / 64;
    const RowLanes rl(G);
    const int64_t rows_pad = (rows + kTileM - 1) / kTileM * kTileM;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * rl.RPW; base < rows_pad; base += nwarps * rl.RPW) {
        const int64_t r = base + rl.slot;
        if (!rl.active || r >= rows_pad) continue;
        if (r >= rows) {   // padding rows of the last 128-row tile: zero codes and scales
            for (int i = 0; i < GPL; ++i) {
                const int grp = rl.li + rl.LPR * i;
                if (grp < G) {
                    GroupQ z = {};
                    store_group(z, r, grp, cols, codes, sf);
                }
            }
            continue;
        }
        GroupQ q[GPL];
        bool finite;
        const float gr = quantize_row_lanes<GPL>(x + r * ld, rl, G, -1.0f, q, finite);
        if (!finite && rl.li == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
#pragma unroll
        for (int i = 0; i < GPL; ++i) {
            const int grp = rl.li + rl.LPR * i;
            if (grp < G) store_group(q[i], r, grp, cols, codes, sf);
        }
        if (rl.li == 0) g[r] = gr;
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
    const int64_t tok0 = chunk * kRouteChunk + w * 32;
    const int64_t npairs = T * k;
    // all of this warp's ids first, so their loads overlap
    int my_e[32];
#pragma unroll
    for (int it = 0; it < 32; ++it) {
        if (it < k) {
            const int64_t p = tok0 * k + it * 32 + lane;
            int e = -1;
            if (p < npairs && tok0 < T) {
                e = __ldg(ids + p);
                if (e < 0 || e >= E) {
                    set_device_error(err, NVFP4_ERR_BAD_EXPERT_ID);
                    e = -1;
                }
            }
            my_e[it] = e;
        }
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    int my_rank[32];
#pragma unroll
    for (int it = 0; it < 32; ++it) {
        if (it < k) {
            const int e = my_e[it];
            const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
            const int before = __popc(m & lt_mask);
            const int base = e >= 0 ? wcount[w * E + e] : 0;
            __syncwarp();
            if (e >= 0 && before == 0) wcount[w * E + e] = base + __popc(m);
            __syncwarp();
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

// Block-wide exclusive prefix sum of one value per thread (blockDim.x = 1024).
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_tot, int32_t& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
        int32_t t = warp_tot[lane];
        int32_t ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(0xFFFFFFFFu, ti, o);
            if (lane >= o) ti += n;
        }
        warp_tot[lane] = ti - t;
        if (lane == 31) warp_tot[32] = ti;
    }
    __syncthreads();
    total = warp_tot[32];
    return warp_tot[w] + incl - v;
}

// One block of 1024 threads: per-expert totals, padded expert offsets, and each
// chunk's first row.
__global__ void __launch_bounds__(1024) route_scan_kernel(int E, int64_t n_chunks,
                                                          const int32_t* __restrict__ chunk_count,
                                                          int32_t* __restrict__ chunk_base,
                                                          int32_t* __restrict__ expert_count,
                                                          int32_t* __restrict__ offsets) {
    __shared__ int32_t seg_sum[1024];
    __shared__ int32_t e_off[1024];
    __shared__ int32_t warp_tot[33];
    const int tid = threadIdx.x;
    const int S = blockDim.x / E;                  // threads per expert (>= 1)
    const int e = tid / S, seg = tid % S;
    const int64_t L = (n_chunks + S - 1) / S;
    const int64_t c0 = seg * L, c1 = min(n_chunks, c0 + L);
    int32_t sum = 0;
    if (e < E) {
        const int32_t* cc = chunk_count + static_cast<int64_t>(e) * n_chunks;
        for (int64_t c = c0; c < c1; ++c) sum += __ldg(cc + c);
    }
    seg_sum[tid] = sum;
    __syncthreads();
    int32_t padded = 0;
    if (tid < E) {
        int32_t run = 0;
        for (int s = 0; s < S; ++s) run += seg_sum[tid * S + s];
        expert_count[tid] = run;
        padded = (run + kTileM - 1) / kTileM * kTileM;
    }
    int32_t total;
    const int32_t start = block_exclusive_scan(padded, warp_tot, total);
    if (tid < E) {
        e_off[tid] = start;
        offsets[tid] = start;
    }
    if (tid == 0) offsets[E] = total;
    __syncthreads();
    if (e < E) {
        int32_t run = e_off[e];
        for (int s = 0; s < seg; ++s) run += seg_sum[e * S + s];
        const int32_t* cc = chunk_count + static_cast<int64_t>(e) * n_chunks;
        int32_t* cb = chunk_base + static_cast<int64_t>(e) * n_chunks;
        for (int64_t c = c0; c < c1; ++c) {
            cb[c] = run;
            run += __ldg(cc + c);
        }
    }
}

template <int GPL>
__global__ void __launch_bounds__(256, GPL == 1 ? 3 : 1) route_quant_scatter_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int E, int k, const int32_t* __restrict__ ids,
    const float* __restrict__ probs, const int32_t* __restrict__ offsets, RouteBufs b, int* err) {
    const int G = H / 64;
    const RowLanes rl(G);
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * rl.RPW; base < T; base += nwarps * rl.RPW) {
        const int64_t t = base + rl.slot;
        if (!rl.active || t >= T) continue;
        const int64_t chunk = t / kRouteChunk;
        // destination rows of the token's k slots: lane li < k of the row fetches slot li's,
        // before the row itself is loaded, so the two dependent lookups overlap the row load
        int my_dst = -1;
        float my_prob = 0.0f;
        if (rl.LPR >= k && rl.li < k) {
            const int64_t p = t * k + rl.li;
            const int e = __ldg(ids + p);
            if (e >= 0 && e < E) {   // out-of-range ids are reported by the histogram kernel
                my_dst = __ldg(b.chunk_base + static_cast<int64_t>(e) * b.n_chunks + chunk) + __ldg(b.pair_rank + p);
                my_prob = __ldg(probs + p);
            }
        }
        GroupQ q[GPL];
        bool finite;
        const float gr = quantize_row_lanes<GPL>(x + t * H, rl, G, -1.0f, q, finite);
        if (!finite && rl.li == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
        const int src0 = rl.slot * rl.LPR;
        for (int j = 0; j < k; ++j) {
            const int64_t p = t * k + j;
            int64_t r;
            float pj;
            if (rl.LPR >= k) {
                r = __shfl_sync(rl.mask, my_dst, src0 + j);
                pj = __shfl_sync(rl.mask, my_prob, src0 + j);
                if (r < 0) continue;
            } else {                 // rows narrower than k lanes: look the slot up directly
                const int e = __ldg(ids + p);
                if (e < 0 || e >= E) continue;
                r = __ldg(b.chunk_base + static_cast<int64_t>(e) * b.n_chunks + chunk) + __ldg(b.pair_rank + p);
                pj = __ldg(probs + p);
            }
#pragma unroll
            for (int i = 0; i < GPL; ++i) {
                const int grp = rl.li + rl.LPR * i;
                if (grp < G) store_group(q[i], r, grp, H, b.a_codes, b.a_sf);
            }
            if (rl.li == 0) {
                b.a_g[r] = gr;
                b.row_pair[r] = static_cast<int32_t>(p);
                b.row_prob[r] = pj;
                b.amax2[r] = 0u;
            }
        }
    }
    // pad rows: expert e's rows [offsets[e] + count_e, offsets[e+1]); one warp zeroes one row's scales
    const int lane = threadIdx.x & 31;
    const int64_t pad_slots = static_cast<int64_t>(E) * kTileM;
    for (int64_t s = warp; s < pad_slots; s += nwarps) {
        const int e = static_cast<int>(s / kTileM), j = static_cast<int>(s % kTileM);
        const int64_t r = static_cast<int64_t>(offsets[e]) + b.expert_count[e] + j;
        if (r >= offsets[e + 1]) continue;
        for (int grp = lane; grp < G; grp += 32) *reinterpret_cast<uint32_t*>(b.a_sf + sf_offset(r, 4 * grp, H)) = 0u;
        if (lane == 0) {
            b.a_g[r] = 0.0f;
            b.row_pair[r] = -1;
            b.row_prob[r] = 0.0f;
            b.amax2[r] = 0u;
        }
    }
}

// ------------------------------------------------------------------ requant
template <int GPL>
__global__ void __launch_bounds__(256, GPL == 1 ? 3 : 1) requant_kernel(const uint16_t* __restrict__ h,
                                                      const uint32_t* __restrict__ amax2,
                                                      const int32_t* __restrict__ row_pair,
                                                      const int32_t* __restrict__ offsets, int E, int I,
                                                      uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                      float* __restrict__ g, int* err) {
    const int G = I / 64;
    const RowLanes rl(G);
    const int64_t rows = offsets[E];
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * rl.RPW; base < rows; base += nwarps * rl.RPW) {
        const int64_t r = base + rl.slot;
        if (!rl.active || r >= rows) continue;
        if (__ldg(row_pair + r) < 0) {       // pad row: zero scales, g = 0 (codes are never read)
            for (int i = 0; i < GPL; ++i) {
                const int grp = rl.li + rl.LPR * i;
                if (grp < G) *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * grp, I)) = 0u;
            }
            if (rl.li == 0) g[r] = 0.0f;
            continue;
        }
        GroupQ q[GPL];
        bool finite;
        const float gr = quantize_row_lanes<GPL>(h + r * I, rl, G, __uint_as_float(__ldg(amax2 + r)), q, finite);
        if (!finite && rl.li == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
#pragma unroll
        for (int i = 0; i < GPL; ++i) {
            const int grp = rl.li + rl.LPR * i;
            if (grp < G) store_group(q[i], r, grp, I, codes, sf);
        }
        if (rl.li == 0) g[r] = gr;
    }
}

int grid_for_warps(int64_t warps) {
    const int64_t blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

// warps needed to cover `rows` rows of G groups in one pass
int64_t warps_for_rows(int64_t rows, int G) {
    const int rpw = G <= 32 ? 32 / G : 1;
    return (rows + rpw - 1) / rpw;
}

}  // namespace

// Dispatch on the number of 64-element groups each lane owns.
#define NVFP4_GPL_DISPATCH(G, KERNEL, ...)                 \
    do {                                                   \
        const int gpl_ = ((G) + 31) / 32;                  \
        if (gpl_ <= 1) KERNEL<1> __VA_ARGS__;              \
        else if (gpl_ <= 2) KERNEL<2> __VA_ARGS__;         \
        else KERNEL<4> __VA_ARGS__;                        \
    } while (0)

cudaError_t launch_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                                 uint8_t* sf, float* g, int* err, cudaStream_t st) {
    const int64_t rows_pad = (rows + kTileM - 1) / kTileM * kTileM;
    if (rows_pad == 0) return cudaSuccess;
    const int c = static_cast<int>(cols);
    const int grid = grid_for_warps(warps_for_rows(rows_pad, c / 64));
    NVFP4_GPL_DISPATCH(c / 64, quantize_rows_kernel, <<<grid, 256, 0, st>>>(x, rows, c, ld, codes, sf, g, err));
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
    const int64_t tw = warps_for_rows(T, H / 64), pw = static_cast<int64_t>(E) * kTileM;
    const int grid = grid_for_warps(tw > pw ? tw : pw);
    NVFP4_GPL_DISPATCH(H / 64, route_quant_scatter_kernel,
                       <<<grid, 256, 0, st>>>(x, T, H, E, k, ids, probs, offsets, b, err));
    return cudaGetLastError();
}

cudaError_t launch_requant(const uint16_t* h, const uint32_t* amax2, const int32_t* row_pair,
                           const int32_t* offsets, int E, int64_t rows_cap, int I, uint8_t* codes, uint8_t* sf,
                           float* g, int* err, cudaStream_t st) {
    const int grid = grid_for_warps(warps_for_rows(rows_cap, I / 64));
    NVFP4_GPL_DISPATCH(I / 64, requant_kernel,
                       <<<grid, 256, 0, st>>>(h, amax2, row_pair, offsets, E, I, codes, sf, g, err));
    return cudaGetLastError();
}

}  // namespace nvfp4
