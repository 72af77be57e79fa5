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

// Lanes of the warp holding the same expert id as this lane (ids < 2^nbits, or -1 for
// none): one ballot per bit of the id, so the cost does not grow with the number of
// distinct ids in the warp.
__device__ __forceinline__ unsigned match_expert(int e, int nbits) {
    const unsigned valid = __ballot_sync(0xFFFFFFFFu, e >= 0);
    unsigned m = e >= 0 ? valid : ~valid;
    for (int b = 0; b < nbits; ++b) {
        const bool bit = (e >> b) & 1;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}

__host__ __device__ __forceinline__ int expert_id_bits(int E) {
    int b = 0;
    while ((1 << b) < E) ++b;
    return b;
}

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

// Both halves of a BF16 pair as an f32x2 operand (element 2j low, 2j+1 high).
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
    uint64_t x;
    asm("{\n\t.reg .b32 lo, hi;\n\t"
        "shl.b32 lo, %1, 16;\n\t"
        "and.b32 hi, %1, 0xFFFF0000;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(x)
        : "r"(w));
    return x;
}

// RN(x / d) on both lanes of an f32x2 pair by Markstein's step, written in terms of
// nx = -x and nrc = (-rc, -rc), d2 = (d, d):
//   q0 = RN(nx * nrc) = RN(x * rc),  r' = q0*d + nx = -(x - q0*d) exactly,
//   q = RN(r' * nrc + q0) = RN(q0 + (x - q0*d) * rc),
// the same values as the usual form.  For x = +-0 this form also returns the zero with
// x's sign (the usual form turns x = -0 into +0), so the code's sign bit needs no fix-up.
__device__ __forceinline__ void div_markstein_neg_x2(uint64_t nx, uint64_t nrc2, uint64_t d2, float& lo, float& hi) {
    uint64_t q0, r, q;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(nx), "l"(nrc2));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q0), "l"(d2), "l"(nx));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(r), "l"(nrc2), "l"(q0));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(q));
}

__device__ __forceinline__ uint64_t f32x2_splat(float a) {
    uint64_t x;
    asm("mov.b64 %0, {%1, %1};" : "=l"(x) : "f"(a));
    return x;
}

// IEEE quotients for the divisors below the Markstein range; kept out of line so the
// common path stays short (it is taken only for rows whose maximum is below ~2^-48).
__device__ __noinline__ void quotients_fdiv(const uint32_t (&w)[4], float d, float (&q)[8]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        q[2 * j] = __fdiv_rn(__uint_as_float(w[j] << 16), d);
        q[2 * j + 1] = __fdiv_rn(__uint_as_float(w[j] & 0xFFFF0000u), d);
    }
}

__device__ __noinline__ float div_rn_slow(float a, float b) { return __fdiv_rn(a, b); }

// Eight E2M1 codes of one 16-byte vector of BF16 values, quotient by d (rc = RN(1/d)).
__device__ __forceinline__ uint32_t codes8(const uint4& v, float d, float rc, bool markstein) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float q[8];
    if (markstein) {
        const uint64_t nrc2 = f32x2_splat(-rc), d2 = f32x2_splat(d);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            div_markstein_neg_x2(bf16x2_to_f32x2(w[j] ^ 0x80008000u), nrc2, d2, q[2 * j], q[2 * j + 1]);
    } else {
        quotients_fdiv(w, d, q);   // IEEE division keeps the sign of a zero quotient
    }
    // The conversion keeps the quotient's sign, also of a zero (-0.0 and tiny negatives
    // give code 8), and every quotient above carries x's sign: the code's sign is x's.
    return e2m1x8(q);
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
        const float r = rc1 != 0.0f ? div_markstein(bmx, d1, rc1) : div_rn_slow(bmx, d1);
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

// The group's 32 bytes of codes go out in one 32-byte store (a whole sector: fewer,
// fuller L2 write transactions than two 16-byte halves), its scale word in one 4-byte store.
__device__ __forceinline__ void store_group(const GroupQ& q, int64_t r, int grp, int cols, uint8_t* codes,
                                            uint8_t* sf) {
    uint8_t* c = codes + r * static_cast<int64_t>(cols / 2) + grp * 32;
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(c), "r"(q.code[0]), "r"(q.code[1]),
                 "r"(q.code[2]), "r"(q.code[3]), "r"(q.code[4]), "r"(q.code[5]), "r"(q.code[6]), "r"(q.code[7])
                 : "memory");
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
__device__ __forceinline__ void load_row_lanes(const uint16_t* src, const RowLanes& rl, int G, uint4 (&v)[GPL][8]) {
#pragma unroll
    for (int i = 0; i < GPL; ++i) {
        const int grp = rl.li + rl.LPR * i;
        if (grp < G) load_group(src + grp * 64, v[i]);
    }
}

// Quantise the row held in v (loaded by load_row_lanes).
template <int GPL>
__device__ __forceinline__ float quantize_loaded(const uint4 (&v)[GPL][8], const RowLanes& rl, int G, float amax_in,
                                                 GroupQ (&q)[GPL], bool& finite) {
    uint32_t bm[GPL][4];
    uint32_t amax_bits = 0;
#pragma unroll
    for (int i = 0; i < GPL; ++i) {
        const int grp = rl.li + rl.LPR * i;
        if (grp < G) {
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

template <int GPL>
__device__ __forceinline__ float quantize_row_lanes(const uint16_t* src, const RowLanes& rl, int G, float amax_in,
                                                    GroupQ (&q)[GPL], bool& finite) {
    uint4 v[GPL][8];
    load_row_lanes<GPL>(src, rl, G, v);
    return quantize_loaded<GPL>(v, rl, G, amax_in, q, finite);
}

// ------------------------------------------------------------------ plain rows
template <int GPL>
__global__ void __launch_bounds__(256, GPL == 1 ? 3 : 1) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                            int cols, int64_t ld, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ sf, float* __restrict__ g,
                                                            int* err) {
    pdl_wait();
    pdl_launch_dependents();
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
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t chunk = blockIdx.x;
    for (int i = threadIdx.x; i < kWarpsPerBlock * E; i += blockDim.x) wcount[i] = 0;
    const int64_t tok0 = chunk * kRouteChunk + w * 32;
    const int64_t npairs = T * k;
    // all of this warp's ids are loaded before any is used, so the loads overlap
    int my_e[32];
#pragma unroll
    for (int it = 0; it < 32; ++it) {
        const int64_t p = tok0 * k + it * 32 + lane;
        my_e[it] = (it < k && p < npairs) ? __ldg(ids + p) : -1;
    }
#pragma unroll
    for (int it = 0; it < 32; ++it) {
        const bool real = it < k && tok0 * k + it * 32 + lane < npairs;
        if (real && (my_e[it] < 0 || my_e[it] >= E)) {
            set_device_error(err, NVFP4_ERR_BAD_EXPERT_ID);
            my_e[it] = -1;
        }
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    const int nbits = expert_id_bits(E);
    int my_rank[32];
#pragma unroll
    for (int it = 0; it < 32; ++it) {
        if (it < k) {
            const int e = my_e[it];
            const unsigned m = match_expert(e, nbits);
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
                                                          int32_t* __restrict__ offsets, int capacity, int* err) {
    __shared__ int32_t seg_sum[1024];
    __shared__ int32_t e_off[1024];
    __shared__ int32_t warp_tot[33];
    pdl_wait();
    pdl_launch_dependents();
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
    int32_t padded = 0, count = 0;
    if (tid < E) {
        for (int s = 0; s < S; ++s) count += seg_sum[tid * S + s];
        expert_count[tid] = count;
        padded = (count + kTileM - 1) / kTileM * kTileM;
    }
    int32_t total;
    int32_t start = block_exclusive_scan(padded, warp_tot, total);
    if (capacity > 0) {                       // fixed-capacity layout: expert e owns rows [e*C, (e+1)*C)
        start = tid * capacity;
        total = E * capacity;
        if (tid < E && count > capacity) set_device_error(err, NVFP4_ERR_CAPACITY);
    }
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

// One block of 1024 threads sorts all T*k pairs when they are few (one launch
// instead of two; beyond a few thousand pairs one SM's issue rate makes the
// chunked kernels faster): per-warp
// expert counts over contiguous pair ranges, the padded expert offsets, then
// every pair's destination row.  The result is the same stable counting sort
// as the chunked kernels above (rows of an expert in (token, slot) order).
constexpr int kBlockSortWarps = 32;
constexpr int kBlockSortMaxE = 256;
constexpr int64_t kBlockSortMaxPairs = 8192;

__global__ void __launch_bounds__(1024) route_block_sort_kernel(const int32_t* __restrict__ ids, int64_t T, int E,
                                                                int k, int32_t* __restrict__ pair_row,
                                                                int32_t* __restrict__ expert_count,
                                                                int32_t* __restrict__ offsets, int capacity, int* err) {
    extern __shared__ int32_t wc[];   // [32 warps][E]: counts, then running rows
    __shared__ int32_t warp_tot[33];
    __shared__ int32_t s_start[kBlockSortMaxE];
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (int i = tid; i < kBlockSortWarps * E; i += blockDim.x) wc[i] = 0;
    __syncthreads();
    const int64_t P = T * k;
    const int64_t per = (P + kBlockSortWarps * 32 - 1) / (kBlockSortWarps * 32) * 32;
    const int64_t p0 = w * per, p1 = min(P, p0 + per);
    int32_t* mine = wc + w * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int nbits = expert_id_bits(E);
    // counts of this warp's pairs; eight batches of ids are loaded before they are used
    for (int64_t b0 = p0; b0 < p1; b0 += 8 * 32) {
        int e8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t p = b0 + u * 32 + lane;
            e8[u] = p < p1 ? __ldg(ids + p) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool real = b0 + u * 32 + lane < p1;
            if (real && (e8[u] < 0 || e8[u] >= E)) {
                set_device_error(err, NVFP4_ERR_BAD_EXPERT_ID);
                e8[u] = -1;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const unsigned m = match_expert(e8[u], nbits);
            if (e8[u] >= 0 && (m & lt_mask) == 0) mine[e8[u]] += __popc(m);
            __syncwarp();
        }
    }
    __syncthreads();
    int32_t cnt = 0;
    if (tid < E) {
        for (int ww = 0; ww < kBlockSortWarps; ++ww) cnt += wc[ww * E + tid];
        expert_count[tid] = cnt;
    }
    int32_t total;
    int32_t start = block_exclusive_scan(tid < E ? (cnt + kTileM - 1) / kTileM * kTileM : 0, warp_tot, total);
    if (capacity > 0) {                       // fixed-capacity layout: expert e owns rows [e*C, (e+1)*C)
        start = tid * capacity;
        total = E * capacity;
        if (tid < E && cnt > capacity) set_device_error(err, NVFP4_ERR_CAPACITY);
    }
    if (tid < E) {
        s_start[tid] = start;
        offsets[tid] = start;
        int32_t run = start;   // first row of each warp's pairs of expert tid
        for (int ww = 0; ww < kBlockSortWarps; ++ww) {
            const int32_t c = wc[ww * E + tid];
            wc[ww * E + tid] = run;
            run += c;
        }
    }
    if (tid == 0) offsets[E] = total;
    __syncthreads();
    for (int64_t b0 = p0; b0 < p1; b0 += 8 * 32) {
        int e8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t p = b0 + u * 32 + lane;
            e8[u] = p < p1 ? __ldg(ids + p) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (e8[u] < 0 || e8[u] >= E) e8[u] = -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e8[u];
            const unsigned m = match_expert(e, nbits);
            const int32_t base = e >= 0 ? mine[e] : 0;
            __syncwarp();
            if (e >= 0 && (m & lt_mask) == 0) mine[e] = base + __popc(m);
            __syncwarp();
            const int64_t p = b0 + u * 32 + lane;
            int32_t row = e >= 0 ? base + __popc(m & lt_mask) : -1;              // -1: bad id, skipped
            if (capacity > 0 && row >= 0 && row - s_start[e] >= capacity) row = -1;   // over capacity: dropped
            if (p < p1) pair_row[p] = row;
        }
    }
}

// Destination rows of pair p (token t, chunk t / kRouteChunk): either stored directly
// by route_block_sort_kernel, or chunk base + rank from the chunked kernels.
// With a fixed capacity C (> 0), a pair whose row falls past its expert's C rows is dropped
// (-1; reported by the counting kernels).
__device__ __forceinline__ int32_t pair_dest(const RouteBufs& b, const int32_t* ids, int E, int64_t p, int64_t chunk,
                                             int capacity) {
    if (b.direct_rows) return __ldg(b.pair_rank + p);
    const int e = __ldg(ids + p);
    const int32_t rank = __ldg(b.pair_rank + p);
    if (e < 0 || e >= E) return -1;   // reported by the counting kernels
    const int32_t row = __ldg(b.chunk_base + static_cast<int64_t>(e) * b.n_chunks + chunk) + rank;
    return (capacity > 0 && row - e * capacity >= capacity) ? -1 : row;
}

// Blocks [0, pad_blocks) give one warp per expert for its pad rows
// [offsets[e] + count_e, offsets[e+1]): zero scales, g = 0, row_pair = -1.
// The remaining blocks quantise tokens (X read once) and write the k copies.
template <int GPL>
__global__ void __launch_bounds__(256, GPL == 1 ? 3 : 1) route_quant_scatter_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int E, int k, const int32_t* __restrict__ ids,
    const float* __restrict__ probs, const int32_t* __restrict__ offsets, RouteBufs b, int pad_blocks, int capacity,
    int* err) {
    pdl_wait();
    pdl_launch_dependents();
    const int G = H / 64;
    const int lane = threadIdx.x & 31;
    if (static_cast<int>(blockIdx.x) < pad_blocks) {
        const int e = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
        if (e >= E) return;
        const int64_t r0 = static_cast<int64_t>(__ldg(offsets + e)) + __ldg(b.expert_count + e);
        const int64_t r1 = __ldg(offsets + e + 1);
        for (int64_t r = r0 + lane; r < r1; r += 32) {
            b.a_g[r] = 0.0f;
            b.row_pair[r] = -1;
            b.row_prob[r] = 0.0f;
            b.amax2[r] = 0u;
        }
        for (int64_t r = r0; r < r1; ++r) {
            for (int grp = lane; grp < G; grp += 32)
                *reinterpret_cast<uint32_t*>(b.a_sf + sf_offset(r, 4 * grp, H)) = 0u;
        }
        return;
    }
    const RowLanes rl(G);
    const int64_t warp = (static_cast<int64_t>(blockIdx.x - pad_blocks) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x - pad_blocks) * blockDim.x) >> 5;
    for (int64_t base = warp * rl.RPW; base < T; base += nwarps * rl.RPW) {
        const int64_t t = base + rl.slot;
        if (!rl.active || t >= T) continue;
        const int64_t chunk = t / kRouteChunk;
        // lane li < k of the row looks up slot li's destination and probability; these
        // loads and the row's are all in flight together
        uint4 v[GPL][8];
        load_row_lanes<GPL>(x + t * H, rl, G, v);
        const bool slot_lane = rl.LPR >= k && rl.li < k;
        int32_t my_dst = -1;
        float my_prob = 0.0f;
        if (slot_lane) {
            const int64_t p = t * k + rl.li;
            my_prob = __ldg(probs + p);
            my_dst = pair_dest(b, ids, E, p, chunk, capacity);
        }
        GroupQ q[GPL];
        bool finite;
        const float gr = quantize_loaded<GPL>(v, rl, G, -1.0f, q, finite);
        if (!finite && rl.li == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
        if (slot_lane && my_dst >= 0) {   // the routed row's per-row data, one slot per lane
            b.a_g[my_dst] = gr;
            b.row_pair[my_dst] = static_cast<int32_t>(t * k + rl.li);
            b.row_prob[my_dst] = my_prob;
            b.amax2[my_dst] = 0u;
        }
        const int src0 = rl.slot * rl.LPR;
        for (int j = 0; j < k; ++j) {
            const int64_t p = t * k + j;
            int64_t r;
            if (rl.LPR >= k) {
                r = __shfl_sync(rl.mask, my_dst, src0 + j);
            } else {                 // rows narrower than k lanes: look the slot up directly
                r = pair_dest(b, ids, E, p, chunk, capacity);
                if (r >= 0 && rl.li == 0) {
                    b.a_g[r] = gr;
                    b.row_pair[r] = static_cast<int32_t>(p);
                    b.row_prob[r] = __ldg(probs + p);
                    b.amax2[r] = 0u;
                }
            }
            if (r < 0) continue;
#pragma unroll
            for (int i = 0; i < GPL; ++i) {
                const int grp = rl.li + rl.LPR * i;
                if (grp < G) store_group(q[i], r, grp, H, b.a_codes, b.a_sf);
            }
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
    pdl_wait();
    pdl_launch_dependents();
    const int G = I / 64;
    const RowLanes rl(G);
    const int64_t rows = offsets[E];
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * rl.RPW; base < rows; base += nwarps * rl.RPW) {
        const int64_t r = base + rl.slot;
        if (!rl.active || r >= rows) continue;
        // the row's flags and values are loaded together (a pad row's h is never used)
        const int32_t pair = __ldg(row_pair + r);
        const uint32_t amax_bits = __ldg(amax2 + r);
        uint4 v[GPL][8];
        load_row_lanes<GPL>(h + r * I, rl, G, v);
        if (pair < 0) {       // pad row: zero scales, g = 0 (codes are never read)
            for (int i = 0; i < GPL; ++i) {
                const int grp = rl.li + rl.LPR * i;
                if (grp < G) *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * grp, I)) = 0u;
            }
            if (rl.li == 0) g[r] = 0.0f;
            continue;
        }
        GroupQ q[GPL];
        bool finite;
        const float gr = quantize_loaded<GPL>(v, rl, G, __uint_as_float(amax_bits), q, finite);
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
#define NVFP4_GPL_LAUNCH(PDL, G, KERNEL, GRID, ...)                                   \
    (((G) + 31) / 32 <= 1   ? launch_pdl(PDL, KERNEL<1>, GRID, 256, 0, __VA_ARGS__)   \
     : ((G) + 31) / 32 <= 2 ? launch_pdl(PDL, KERNEL<2>, GRID, 256, 0, __VA_ARGS__)   \
                            : launch_pdl(PDL, KERNEL<4>, GRID, 256, 0, __VA_ARGS__))

cudaError_t launch_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                                 uint8_t* sf, float* g, int* err, cudaStream_t st) {
    const int64_t rows_pad = (rows + kTileM - 1) / kTileM * kTileM;
    if (rows_pad == 0) return cudaSuccess;
    const int c = static_cast<int>(cols);
    const int grid = grid_for_warps(warps_for_rows(rows_pad, c / 64));
    return NVFP4_GPL_LAUNCH(false, c / 64, quantize_rows_kernel, grid, st, x, rows, c, ld, codes, sf, g, err);
}

// capacity > 0: the fixed-capacity layout (expert e's rows at [e*C, e*C + count_e), pad rows to
// (e+1)*C; pairs past the capacity are dropped and NVFP4_ERR_CAPACITY is recorded).
cudaError_t launch_route_sort_quant_cap(const uint16_t* x, int64_t T, int H, int E, int k, const int32_t* ids,
                                        const float* probs, int32_t* offsets, const RouteBufs& b_in, int capacity,
                                        int* err, cudaStream_t st) {
    if (T == 0) return capacity > 0 ? cudaSuccess : cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    RouteBufs b = b_in;
    cudaError_t e;
    if (E <= kBlockSortMaxE && T * k <= kBlockSortMaxPairs) {
        b.direct_rows = 1;
        const size_t smem = sizeof(int32_t) * kBlockSortWarps * E;
        e = launch_pdl(false, route_block_sort_kernel, 1, kBlockSortWarps * 32, smem, st, ids, T, E, k, b.pair_rank,
                       b.expert_count, offsets, capacity, err);
        if (e != cudaSuccess) return e;
    } else {
        b.direct_rows = 0;
        const size_t smem = sizeof(int32_t) * kWarpsPerBlock * E;
        e = launch_pdl(false, route_hist_rank_kernel, static_cast<unsigned>(b.n_chunks), 256, smem, st, ids, T, E, k,
                       b.n_chunks, b.chunk_count, b.pair_rank, err);
        if (e != cudaSuccess) return e;
        e = launch_pdl(true, route_scan_kernel, 1, 1024, 0, st, E, b.n_chunks, b.chunk_count, b.chunk_base,
                       b.expert_count, offsets, capacity, err);
        if (e != cudaSuccess) return e;
    }
    const int pad_blocks = (E + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int grid = pad_blocks + grid_for_warps(warps_for_rows(T, H / 64));
    return NVFP4_GPL_LAUNCH(true, H / 64, route_quant_scatter_kernel, grid, st, x, T, H, E, k, ids, probs, offsets, b,
                            pad_blocks, capacity, err);
}

cudaError_t launch_route_sort_quant(const uint16_t* x, int64_t T, int H, int E, int k, const int32_t* ids,
                                    const float* probs, int32_t* offsets, const RouteBufs& b, int* err,
                                    cudaStream_t st) {
    return launch_route_sort_quant_cap(x, T, H, E, k, ids, probs, offsets, b, 0, err, st);
}

cudaError_t launch_requant(const uint16_t* h, const uint32_t* amax2, const int32_t* row_pair,
                           const int32_t* offsets, int E, int64_t rows_cap, int I, uint8_t* codes, uint8_t* sf,
                           float* g, int* err, cudaStream_t st, bool pdl) {
    const int grid = grid_for_warps(warps_for_rows(rows_cap, I / 64));
    return NVFP4_GPL_LAUNCH(pdl, I / 64, requant_kernel, grid, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
}

}  // namespace nvfp4
