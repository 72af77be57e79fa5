// The NVFP4 row quantiser's device code, shared by the quantiser kernels (quant.cu) and
// the FC2 kernel that requantises its A operand in shared memory (gemm.cu).
//
// Two-level NVFP4 as defined on "miniTE diagnoses and narrows the cross-engine execution gap
// of NVFP4 RL", section "How it differs": g = max|row| / (6*448) in FP32, an E4M3 scale per
// 16 elements, E2M1 codes, round-to-nearest-even.  Block scale s_b = e4m3(bmax / (g*6)),
// code = e2m1(x / (g*s_b)), both quotients the correctly rounded binary32 quotient.
//
// Work split: a lane owns whole 64-element groups (four 16-element blocks, 128 bytes of
// BF16): it loads them with 16-byte loads, finds the block maxima with NaN-propagating
// bf16x2 max, and produces 32 bytes of codes plus one 32-bit word of four block scales per
// group.  A row of G groups is spread over G lanes (G <= 32: 32/G rows per warp) or over the
// whole warp (G > 32: G/32 groups per lane); the row maximum is one redux.sync over the
// row's lanes.
//
// Division: x / d for the 16 elements of a block that share d = g*s_b uses Markstein's
// method (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 1990; also Muller et al., Handbook of Floating-Point
// Arithmetic, ch. on FMA-based division): with y = RN(1/d) from __frcp_rn, q0 = RN(x*y),
// r = x - d*q0 (exact with an FMA) and q = RN(q0 + r*y) equals RN(x/d) when no intermediate
// leaves the normal range.  Divisors below 2^-60 take IEEE __fdiv_rn instead, which keeps
// every quotient that can reach a code boundary (|x/d| >= 0.25) in the normal range.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

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

// Codes by IEEE division for the divisors below the Markstein range; kept out of line so
// the common path stays short (it is taken only for rows whose maximum is below ~2^-48).
// Its arguments and result are scalars, so the call keeps everything in registers.
__device__ __noinline__ uint32_t codes8_fdiv(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, float d) {
    const uint32_t w[4] = {w0, w1, w2, w3};
    float q[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        q[2 * j] = __fdiv_rn(__uint_as_float(w[j] << 16), d);
        q[2 * j + 1] = __fdiv_rn(__uint_as_float(w[j] & 0xFFFF0000u), d);
    }
    return e2m1x8(q);   // IEEE division keeps the sign of a zero quotient
}

__device__ __noinline__ float div_rn_slow(float a, float b) { return __fdiv_rn(a, b); }

// Eight E2M1 codes of one 16-byte vector of BF16 values, quotient by d (rc = RN(1/d)).
__device__ __forceinline__ uint32_t codes8(const uint4& v, float d, float rc, bool markstein) {
    if (!markstein) return codes8_fdiv(v.x, v.y, v.z, v.w, d);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float q[8];
    const uint64_t nrc2 = f32x2_splat(-rc), d2 = f32x2_splat(d);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        div_markstein_neg_x2(bf16x2_to_f32x2(w[j] ^ 0x80008000u), nrc2, d2, q[2 * j], q[2 * j + 1]);
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

}  // namespace
}  // namespace nvfp4
