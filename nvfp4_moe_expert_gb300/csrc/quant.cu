// NVFP4 quantisers: plain row quantisation (weights or any rows), the fused
// route sort + per-token amax + pad + quantise of the FC1 input, and the
// requantisation of the FC2 input.  The row quantiser itself (two-level NVFP4,
// the lane-owns-a-64-element-group work split and the correctly rounded
// quotients) is in nvfp4_quant.cuh.
//
// The route sort follows "miniTE diagnoses and narrows the cross-engine
// execution gap of NVFP4 RL", section "How to use it": the tokens are sorted
// by expert and the row maximum is taken in the same pass that quantises the
// row, so X is read exactly once.
#include <cfloat>

#include "common.cuh"
#include "nvfp4_quant.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kRouteChunk = 256;       // tokens per route-sort chunk (8 warps x 32 tokens)

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

// The group's 32 bytes of codes go out in one 32-byte store (a whole sector: fewer,
// fuller L2 write transactions than two 16-byte halves), its scale word in one 4-byte store.
__device__ __forceinline__ void store_codes(const GroupQ& q, int64_t r, int grp, int cols, uint8_t* codes) {
    uint8_t* c = codes + r * static_cast<int64_t>(cols / 2) + grp * 32;
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(c), "r"(q.code[0]), "r"(q.code[1]),
                 "r"(q.code[2]), "r"(q.code[3]), "r"(q.code[4]), "r"(q.code[5]), "r"(q.code[6]), "r"(q.code[7])
                 : "memory");
}
// Scales in the 512-byte scale tiles (weights: the GEMM copies their tiles as they are).
__device__ __forceinline__ void store_group(const GroupQ& q, int64_t r, int grp, int cols, uint8_t* codes,
                                            uint8_t* sf) {
    store_codes(q, r, grp, cols, codes);
    *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * grp, cols)) = q.sfw;
}
// Scales row-major (routed activations: a row's scale words are contiguous, so a warp's k
// copies of a token write whole lines; the GEMM rearranges them into tiles per stage).
__device__ __forceinline__ void store_group_rows(const GroupQ& q, int64_t r, int grp, int cols, uint8_t* codes,
                                                 uint8_t* sf) {
    store_codes(q, r, grp, cols, codes);
    *reinterpret_cast<uint32_t*>(sf + sf_row_offset(r, 4 * grp, cols)) = q.sfw;
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
__global__ void __launch_bounds__(256, GPL == 1 ? 3 : (GPL == 2 ? 2 : 1)) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
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
    // The quantise-scatter that follows may start at once: it reads only inputs written
    // before the histogram kernel (which starts after all earlier work has finished) until
    // its own wait, which covers this kernel and, through this kernel's wait, the histogram.
    pdl_launch_dependents();
    pdl_wait();
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
// The same given the pair's expert id e (already loaded): its rank and chunk base are loaded
// together.
__device__ __forceinline__ int32_t pair_dest_e(const RouteBufs& b, int e, int E, int64_t p, int64_t chunk,
                                               int capacity) {
    if (b.direct_rows) return __ldg(b.pair_rank + p);
    if (e < 0 || e >= E) return -1;   // reported by the counting kernels
    const int32_t rank = __ldg(b.pair_rank + p);
    const int32_t row = __ldg(b.chunk_base + static_cast<int64_t>(e) * b.n_chunks + chunk) + rank;
    return (capacity > 0 && row - e * capacity >= capacity) ? -1 : row;
}
__device__ __forceinline__ int32_t pair_dest(const RouteBufs& b, const int32_t* ids, int E, int64_t p, int64_t chunk,
                                             int capacity) {
    return pair_dest_e(b, b.direct_rows ? 0 : __ldg(ids + p), E, p, chunk, capacity);
}

// Blocks [0, pad_blocks) give one warp per expert for its pad rows
// [offsets[e] + count_e, offsets[e+1]): zero scales, g = 0, row_pair = -1.
// The remaining blocks quantise tokens (X read once) and write the k copies.  A token's
// row and routing probabilities are inputs of the route stage, so they are loaded and the
// row quantised before the wait on the sorting kernels; only the destination rows (and
// the stores) come after it.
// Narrow rows (one group per lane) run in 128-thread blocks held to 72 registers, seven
// blocks (28 warps) per SM, so that 4096 tokens at one token per warp fit in one wave.
template <int GPL>
__global__ void __launch_bounds__(GPL == 1 ? 128 : 256, GPL == 1 ? 7 : (GPL == 2 ? 2 : 1)) route_quant_scatter_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int E, int k, const int32_t* __restrict__ ids,
    const float* __restrict__ probs, const int32_t* __restrict__ offsets, RouteBufs b, int pad_blocks, int capacity,
    int* err) {
    pdl_launch_dependents();
    const int G = H / 64;
    const int lane = threadIdx.x & 31;
    if (static_cast<int>(blockIdx.x) < pad_blocks) {
        pdl_wait();
        const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
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
                *reinterpret_cast<uint32_t*>(b.a_sf_rows + sf_row_offset(r, 4 * grp, H)) = 0u;
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
        // lane li < k of the row holds slot li's probability and expert id (inputs) and,
        // after the wait, its destination row
        uint4 v[GPL][8];
        load_row_lanes<GPL>(x + t * H, rl, G, v);
        const bool slot_lane = rl.LPR >= k && rl.li < k;
        float my_prob = 0.0f;
        int my_e = -1;
        if (slot_lane) {
            my_prob = __ldg(probs + t * k + rl.li);
            my_e = __ldg(ids + t * k + rl.li);
        }
        GroupQ q[GPL];
        bool finite;
        const float gr = quantize_loaded<GPL>(v, rl, G, -1.0f, q, finite);
        if (!finite && rl.li == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
        pdl_wait();
        int32_t my_dst = -1;
        if (slot_lane) my_dst = pair_dest_e(b, my_e, E, t * k + rl.li, chunk, capacity);
        if (slot_lane) b.pair_row[t * k + rl.li] = my_dst;
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
                if (rl.li == 0) b.pair_row[p] = static_cast<int32_t>(r);
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
                if (grp < G) store_group_rows(q[i], r, grp, H, b.a_codes, b.a_sf_rows);
            }
        }
    }
}

// ------------------------------------------------------------------ scale tiles
// The scatter writes each routed copy's block scales row-major (a copy's scale words are one
// contiguous line instead of 32 words in 32 different 512-byte tiles); this kernel rearranges
// them into the tiles FC1 copies into TMEM.  A block takes one m-tile (128 rows) and `chunk`
// K=64 blocks (16, or 32 when that leaves more than 4096 blocks): each thread loads its row's
// 4 * chunk bytes (16-byte loads, all in flight), and after a barrier the block writes the
// chunk's tiles contiguously, one 16-byte slot per thread and step (slot s of tile j: the
// K-block j words of rows s, s + 32, s + 64, s + 96).  Only rows below expert_offsets[E] are
// touched (FC1 reads no others).
constexpr int kTileMaxChunk = 32;

__global__ void __launch_bounds__(128) route_scale_tiles_kernel(const uint8_t* __restrict__ rows_sf,
                                                                 uint8_t* __restrict__ sf, int H, int chunk,
                                                                 const int32_t* __restrict__ offsets, int E) {
    extern __shared__ uint32_t s_rows[];                    // [kTileM][chunk + 1]: odd pitch, conflict-free column reads
    pdl_wait();
    pdl_launch_dependents();
    const int64_t mt = blockIdx.x;
    if (mt * kTileM >= __ldg(offsets + E)) return;
    const int tid = threadIdx.x;
    const int W = H / 64;                                   // scale words per row
    const int j0 = static_cast<int>(blockIdx.y) * chunk;
    const int n = min(chunk, W - j0);                      // a multiple of 4 (H % 256 == 0)
    const uint4* row =
        reinterpret_cast<const uint4*>(rows_sf + (mt * kTileM + tid) * static_cast<int64_t>(H / 16)) + j0 / 4;
    uint4 v[kTileMaxChunk / 4];
#pragma unroll
    for (int c = 0; c < kTileMaxChunk / 4; ++c)
        if (4 * c < n) v[c] = __ldg(row + c);
#pragma unroll
    for (int c = 0; c < kTileMaxChunk / 4; ++c) {
        if (4 * c < n) {
            uint32_t* dst = s_rows + tid * (chunk + 1) + 4 * c;
            dst[0] = v[c].x;
            dst[1] = v[c].y;
            dst[2] = v[c].z;
            dst[3] = v[c].w;
        }
    }
    __syncthreads();
    uint4* tiles = reinterpret_cast<uint4*>(sf + (mt * W + j0) * kSfAtomBytes);
    for (int i = tid; i < 32 * n; i += kTileM) {
        const int j = i >> 5, slot = i & 31;
        tiles[j * (kSfAtomBytes / 16) + slot] =
            make_uint4(s_rows[slot * (chunk + 1) + j], s_rows[(slot + 32) * (chunk + 1) + j],
                       s_rows[(slot + 64) * (chunk + 1) + j], s_rows[(slot + 96) * (chunk + 1) + j]);
    }
}

// ------------------------------------------------------------------ requant
template <int GPL>
__global__ void __launch_bounds__(256, GPL == 1 ? 3 : (GPL == 2 ? 2 : 1)) requant_kernel(const uint16_t* __restrict__ h,
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

// ------------------------------------------------------------------ requant, coalesced
// The same quantisation with a warp per row and the row's bytes spread over the lanes in
// 16-byte chunks: lane l holds elements 256 j + 8 l .. +7 for chunks j = 0..C-1 (C = I/256
// rounded up; the last chunk may cover only the first lanes).  Every load and every code
// store of a warp covers whole 128-byte lines, which takes an eighth of the L1 wavefronts of
// the lane-owns-a-group layout.  A 16-element block is the lane pair (2m, 2m+1) of a chunk:
// its maximum is one shuffle, both lanes derive the same block scale, and each lane divides
// its own 8 elements; the 4-byte scale word of a 64-element group is gathered to the group's
// first lane.  Arithmetic and results are those of quantize_group.
constexpr int kCoalescedMaxChunks = 8;   // I <= 2048

template <int C>
__global__ void __launch_bounds__(256) requant_coalesced_kernel(const uint16_t* __restrict__ h,
                                                                const uint32_t* __restrict__ amax2,
                                                                const int32_t* __restrict__ row_pair,
                                                                const int32_t* __restrict__ offsets, int E, int I,
                                                                uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                                float* __restrict__ g, int* err) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t rows = offsets[E];
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int last_lanes = (I - 256 * (C - 1)) / 8;          // lanes holding data in the last chunk
    for (int64_t r = warp; r < rows; r += nwarps) {
        const int32_t pair = __ldg(row_pair + r);
        const uint32_t amax_bits = __ldg(amax2 + r);
        uint4 v[C];
        if (pair >= 0) {
#pragma unroll
            for (int j = 0; j < C; ++j)
                v[j] = (j < C - 1 || lane < last_lanes)
                           ? __ldg(reinterpret_cast<const uint4*>(h + r * I + 256 * j + 8 * lane))
                           : make_uint4(0u, 0u, 0u, 0u);
        }
        if (pair < 0) {       // pad row: zero scales, g = 0 (codes are never read)
#pragma unroll
            for (int j = 0; j < C; ++j) {
                const int grp = 4 * j + (lane >> 3);
                if ((lane & 7) == 0 && (j < C - 1 || lane < last_lanes))
                    *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * grp, I)) = 0u;
            }
            if (lane == 0) g[r] = 0.0f;
            continue;
        }
        // block maxima (this lane's 8 elements, then its pair lane's) and the row's finiteness
        uint32_t bm[C];
        uint32_t m_all = 0u;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            constexpr uint32_t kAbs = 0x7FFF7FFFu;
            uint32_t m = bf16x2_max_nan(bf16x2_max_nan(v[j].x & kAbs, v[j].y & kAbs),
                                        bf16x2_max_nan(v[j].z & kAbs, v[j].w & kAbs));
            m = bf16x2_max_nan(m, m >> 16);
            m = bf16x2_max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1)) << 16;
            bm[j] = m;
            m_all = max(m_all, m);
        }
        m_all = __reduce_max_sync(0xFFFFFFFFu, m_all);
        const bool finite = m_all < 0x7F800000u;
        if (!finite && lane == 0) set_device_error(err, NVFP4_ERR_NONFINITE);
        const float amax = __uint_as_float(amax_bits);
        const float gr = finite ? __fdiv_rn(amax, kOuterDivisor) : 0.0f;
        const float d1 = __fmul_rn(gr, 6.0f);
        const float rc1 = d1 >= kMarksteinMinDivisor ? __frcp_rn(d1) : 0.0f;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const bool have = j < C - 1 || lane < last_lanes;
            const float bmx = __uint_as_float(bm[j]);
            const float q1 = rc1 != 0.0f ? div_markstein(bmx, d1, rc1) : div_rn_slow(bmx, d1);
            const uint32_t s_code = d1 > 0.0f ? cvt_e4m3(q1) : 0u;
            const float d2 = __fmul_rn(gr, e4m3_value(s_code));
            uint32_t cw = 0u;
            if (d2 > 0.0f) {
                const bool mk = d2 >= kMarksteinMinDivisor;
                cw = codes8(v[j], d2, mk ? __frcp_rn(d2) : 0.0f, mk);
            }
            if (have) *reinterpret_cast<uint32_t*>(codes + r * (I / 2) + 128 * j + 4 * lane) = cw;
            // the group's four block scales (lanes 8m, 8m+2, 8m+4, 8m+6) into one word on lane 8m
            const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, s_code, 2);
            const uint32_t s4 = __shfl_down_sync(0xFFFFFFFFu, s_code, 4);
            const uint32_t s6 = __shfl_down_sync(0xFFFFFFFFu, s_code, 6);
            if ((lane & 7) == 0 && have) {
                const int grp = 4 * j + (lane >> 3);
                *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * grp, I)) = s_code | (s2 << 8) | (s4 << 16) | (s6 << 24);
            }
        }
        if (lane == 0) g[r] = gr;
    }
}

// ------------------------------------------------------------------ requant, a block per lane
// The same quantisation with every lane owning whole 16-element blocks.  A warp takes R
// consecutive rows at a time, R the smallest count for which the batch's R*B blocks (B = I/16)
// fill whole passes of 32 lanes, in P = R*B/32 passes: in pass p lane l quantises block
// f = 32 p + l of the batch (row f / B, block f % B).  Consecutive rows are contiguous in h, so
// each pass reads 1 KB (one 32-byte load per lane) and writes 256 contiguous bytes of codes.
// Each block's scale, reciprocal and codes are computed once, by its own lane; per row, the
// finiteness is one ballot per pass and the outer scale is computed by lane rho for row rho
// and shuffled.  Arithmetic and results are those of quantize_group.
constexpr int kBlockLanesMaxPasses = 4;

__device__ __forceinline__ void load32_nc(const uint16_t* p, uint4& a, uint4& b) {
    asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
        : "l"(p));
}

// Passes per batch for rows of I columns (0 when the batch would need more than
// kBlockLanesMaxPasses).
int block_lanes_passes(int I) {
    if (I % 16 != 0 || I <= 0) return 0;
    const int B = I / 16;
    int gcd = B, b = 32;
    while (b) {
        const int t = gcd % b;
        gcd = b;
        b = t;
    }
    const int R = 32 / gcd;
    const int P = R * B / 32;
    return P <= kBlockLanesMaxPasses ? P : 0;
}

// ICT: the width I compiled in (0: I_rt at run time); with it the index and scale-tile address
// arithmetic folds to constants (I = 768 and 1536: 8-9% fewer cycles).
template <int P, int ICT = 0>
__global__ void __launch_bounds__(256, P <= 3 ? 4 : 2) requant_blocks_kernel(const uint16_t* __restrict__ h,
                                                             const uint32_t* __restrict__ amax2,
                                                             const int32_t* __restrict__ row_pair,
                                                             const int32_t* __restrict__ offsets, int E, int I_rt,
                                                             uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                             float* __restrict__ g, int* err) {
    const int I = ICT ? ICT : I_rt;
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int B = I / 16;
    const int R = 32 * P / B;
    const int64_t rows = offsets[E];
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    int rho[P], blk[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int f = 32 * p + lane;
        rho[p] = f / B;
        blk[p] = f - rho[p] * B;
    }
    for (int64_t r0 = warp * R; r0 < rows; r0 += nwarps * R) {
        // row data on lane rho for row r0 + rho
        int32_t pair_l = -1;
        uint32_t amax_l = 0u;
        const bool row_lane = lane < R && r0 + lane < rows;
        if (row_lane) {
            pair_l = __ldg(row_pair + r0 + lane);
            amax_l = __ldg(amax2 + r0 + lane);
        }
        // h is loaded for every row below the used count, pad rows included, so that these
        // loads need not wait for the row map; a pad row's (stale) values are never used
        uint4 v[P][2];
        bool in_range[P], live[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            in_range[p] = r0 + rho[p] < rows;
            if (in_range[p]) {
                load32_nc(h + (r0 + rho[p]) * I + 16 * blk[p], v[p][0], v[p][1]);
            } else {
                v[p][0] = make_uint4(0u, 0u, 0u, 0u);
                v[p][1] = v[p][0];
            }
        }
#pragma unroll
        for (int p = 0; p < P; ++p) live[p] = in_range[p] && __shfl_sync(0xFFFFFFFFu, pair_l, rho[p]) >= 0;
        // block maxima; a row is finite when none of its blocks holds an infinity or NaN
        uint32_t bm[P];
        unsigned nonfinite_mask[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            bm[p] = block_absmax_bits(v[p][0], v[p][1]);
            nonfinite_mask[p] = __ballot_sync(0xFFFFFFFFu, bm[p] >= 0x7F800000u);
        }
        float g_l = 0.0f, d1_l = 0.0f, rc1_l = 0.0f;
        if (row_lane) {
            bool finite = true;
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int lo = max(lane * B - 32 * p, 0), hi = min(lane * B + B - 32 * p, 32);
                if (lo < hi) {
                    const unsigned m = (hi - lo == 32 ? 0xFFFFFFFFu : ((1u << (hi - lo)) - 1u)) << lo;
                    if (nonfinite_mask[p] & m) finite = false;
                }
            }
            if (pair_l >= 0) {
                if (!finite) set_device_error(err, NVFP4_ERR_NONFINITE);
                g_l = finite ? __fdiv_rn(__uint_as_float(amax_l), kOuterDivisor) : 0.0f;
                d1_l = __fmul_rn(g_l, 6.0f);
                rc1_l = d1_l >= kMarksteinMinDivisor ? __frcp_rn(d1_l) : 0.0f;
            }
            g[r0 + lane] = g_l;                  // pad rows: g = 0
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const float gr = __shfl_sync(0xFFFFFFFFu, g_l, rho[p]);
            const float d1 = __shfl_sync(0xFFFFFFFFu, d1_l, rho[p]);
            const float rc1 = __shfl_sync(0xFFFFFFFFu, rc1_l, rho[p]);
            if (!in_range[p]) continue;
            const int64_t r = r0 + rho[p];
            uint32_t s_code = 0u;
            if (live[p]) {
                const float bmx = __uint_as_float(bm[p]);
                const float q1 = rc1 != 0.0f ? div_markstein(bmx, d1, rc1) : div_rn_slow(bmx, d1);
                s_code = d1 > 0.0f ? cvt_e4m3(q1) : 0u;
                const float d2 = __fmul_rn(gr, e4m3_value(s_code));
                uint32_t c0 = 0u, c1 = 0u;
                if (d2 > 0.0f) {
                    const bool mk = d2 >= kMarksteinMinDivisor;
                    const float rc = mk ? __frcp_rn(d2) : 0.0f;
                    c0 = codes8(v[p][0], d2, rc, mk);
                    c1 = codes8(v[p][1], d2, rc, mk);
                }
                *reinterpret_cast<uint2*>(codes + r * (I / 2) + 8 * blk[p]) = make_uint2(c0, c1);
            }
            sf[sf_offset(r, blk[p], I)] = static_cast<uint8_t>(s_code);   // pad rows: zero scales
        }
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
    const int G = H / 64;
    if (G <= 32) {   // 128-thread blocks (4 warps), one warp per token
        const int pad_blocks = (E + 3) / 4;
        const int64_t wanted = (warps_for_rows(T, G) + 3) / 4;
        const int64_t cap = static_cast<int64_t>(device_sm_count()) * 32;
        const int grid = pad_blocks + static_cast<int>(wanted < 1 ? 1 : (wanted < cap ? wanted : cap));
        e = launch_pdl(true, route_quant_scatter_kernel<1>, grid, 128, 0, st, x, T, H, E, k, ids, probs, offsets, b,
                       pad_blocks, capacity, err);
    } else {
        const int pad_blocks = (E + kWarpsPerBlock - 1) / kWarpsPerBlock;
        const int grid = pad_blocks + grid_for_warps(warps_for_rows(T, G));
        e = NVFP4_GPL_LAUNCH(true, G, route_quant_scatter_kernel, grid, st, x, T, H, E, k, ids, probs, offsets, b,
                             pad_blocks, capacity, err);
    }
    if (e != cudaSuccess) return e;
    // one block per (m-tile, chunk of K-blocks) of the capacity: chunks of 16 K-blocks, longer
    // while that leaves more than 4096 blocks; blocks past the used rows return at once.  Fewer,
    // longer blocks free the SMs sooner for FC1, which follows as a programmatic dependent (at
    // 4096 tokens 766 blocks of 16 give a 1.8% faster step than 3064 blocks of 4, at 16384
    // tokens 2302 of 16 a 2.5% faster one than 1151 of 32)
    const int64_t m_tiles = b.rows_cap / kTileM;
    const int W = H / 64;
    int chunk = 16;
    while (chunk < kTileMaxChunk && chunk < W && m_tiles * W / chunk > 4096) chunk *= 2;
    const dim3 tg(static_cast<unsigned>(m_tiles), static_cast<unsigned>((W + chunk - 1) / chunk));
    const size_t smem = sizeof(uint32_t) * kTileM * (chunk + 1);
    return launch_pdl(true, route_scale_tiles_kernel, tg, kTileM, smem, st, b.a_sf_rows, b.a_sf, H, chunk, offsets, E);
}

cudaError_t launch_route_sort_quant(const uint16_t* x, int64_t T, int H, int E, int k, const int32_t* ids,
                                    const float* probs, int32_t* offsets, const RouteBufs& b, int* err,
                                    cudaStream_t st) {
    return launch_route_sort_quant_cap(x, T, H, E, k, ids, probs, offsets, b, 0, err, st);
}

cudaError_t launch_requant(const uint16_t* h, const uint32_t* amax2, const int32_t* row_pair,
                           const int32_t* offsets, int E, int64_t rows_cap, int I, uint8_t* codes, uint8_t* sf,
                           float* g, int* err, cudaStream_t st, bool pdl) {
    const int P = block_lanes_passes(I);
    if (P > 0) {
        const int B = I / 16, R = 32 * P / B;
        const int grid = grid_for_warps((rows_cap + R - 1) / R);
        switch (P) {
            case 1: return launch_pdl(pdl, requant_blocks_kernel<1>, grid, 256, 0, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
            case 2: return launch_pdl(pdl, requant_blocks_kernel<2>, grid, 256, 0, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
            case 3:
                if (I == 768)
                    return launch_pdl(pdl, requant_blocks_kernel<3, 768>, grid, 256, 0, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
                if (I == 1536)
                    return launch_pdl(pdl, requant_blocks_kernel<3, 1536>, grid, 256, 0, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
                return launch_pdl(pdl, requant_blocks_kernel<3>, grid, 256, 0, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
            case 4: return launch_pdl(pdl, requant_blocks_kernel<4>, grid, 256, 0, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
            default: break;
        }
    }
    const int C = (I + 255) / 256;
    if (C <= kCoalescedMaxChunks) {
        const int grid = grid_for_warps(rows_cap);
#define NVFP4_REQUANT_C(CC) \
    case CC: return launch_pdl(pdl, requant_coalesced_kernel<CC>, grid, 256, 0, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
        switch (C) {
            NVFP4_REQUANT_C(1) NVFP4_REQUANT_C(2) NVFP4_REQUANT_C(3) NVFP4_REQUANT_C(4)
            NVFP4_REQUANT_C(5) NVFP4_REQUANT_C(6) NVFP4_REQUANT_C(7) NVFP4_REQUANT_C(8)
            default: break;
        }
#undef NVFP4_REQUANT_C
    }
    const int grid = grid_for_warps(warps_for_rows(rows_cap, I / 64));
    return NVFP4_GPL_LAUNCH(pdl, I / 64, requant_kernel, grid, st, h, amax2, row_pair, offsets, E, I, codes, sf, g, err);
}

}  // namespace nvfp4
