/*
 * nvfp4_moe.h -- C ABI of the batch-invariant NVFP4 W4A4 MoE expert forward
 * for GB300 (sm_103a).
 *
 * What is computed (sources; the pages are cited by title and section):
 *
 *  [miniTE/differs]  "miniTE diagnoses and narrows the cross-engine execution
 *      gap of NVFP4 RL" (onedev.kr/papers/1404), section "How it differs":
 *      two-level NVFP4 -- E2M1 codes, one E4M3 scale per 16 elements, an FP32
 *      outer scale per row g = max|row| / (6*448), round-to-nearest-even, no
 *      Hadamard transform, no stochastic rounding; g^x*g^w applied in an FP32
 *      epilogue before the BF16 cast; the router probability multiplies the
 *      SwiGLU activation before FC2; the expert combine order is preserved.
 *  [miniTE/use]  same page, section "How to use it": the quantiser writes the
 *      packed FP4 codes, block scales and outer scales into contiguous buffers
 *      the grouped GEMM consumes directly; expert boundaries are device
 *      offsets; sort+amax then pad(X, amax) then quantise (no separate
 *      activation scan); FC2 maxima come from the producer of the
 *      router-weighted activation; FC1 and FC2 have their own GEMM settings.
 *  [RL/4.4]  "Finishing RL training faster: bitwise consistency, high
 *      performance, agent-driven" (spke.com/ko/ai/article/3192), section 4.4
 *      "Expert GEMM: two layouts, same row result": per-token quantisation,
 *      a fixed per-row accumulation order, SiLU(gate)*up in FP32 rounded once.
 *  [RL/4.5]  same article, section 4.5 "Cross-GPU reduction": expert outputs
 *      summed in FP32 in top-k slot order.
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are device pointers; the caller allocates and owns
 *    every buffer.  The library never allocates or frees memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All GPU work is enqueued on it; no entry point synchronises
 *    except nvfp4_get_device_error.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns an error and enqueues nothing.  A failed launch
 *    returns NVFP4_ERR_CUDA.  Conditions only the GPU can see (an expert id
 *    out of range, a non-finite row maximum, a bounded wait that ran out) are
 *    recorded in a per-device error word read by nvfp4_get_device_error.
 *  - BF16 tensors are raw IEEE bfloat16 bit patterns (uint16).
 *
 * NVFP4 storage used by every entry point ("NVFP4 rows"):
 *  - codes  uint8 [rows_pad][cols/2]: element 2j of a row is the low nibble
 *           of byte j, element 2j+1 the high nibble; nibble = sign<<3 | E2M1
 *           magnitude index (0,0.5,1,1.5,2,3,4,6).
 *  - sf     uint8, nvfp4_sf_bytes(rows, cols) bytes: the E4M3 block scale of
 *           row r, block b (elements 16b..16b+15) is at byte
 *             ((r/128) * (cols/64) + b/4) * 512 + (r%32)*16 + ((r%128)/32)*4 + b%4
 *           i.e. 512-byte tiles of 128 rows x 64 columns laid out so one tile
 *           is what the tensor core's scale-factor copy takes for one MMA step.
 *  - g      float32 [rows]: the outer scale.
 *  - rows_pad = nvfp4_rows_padded(rows) = rows rounded up to 128.
 */
#ifndef NVFP4_MOE_H
#define NVFP4_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,          /* null pointer, negative size, misaligned pointer */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 2,    /* shape outside the supported set (see each call) */
    NVFP4_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below moe_workspace_bytes(...) */
    NVFP4_ERR_CUDA = 4,                 /* a CUDA runtime/driver call or launch failed */
    NVFP4_ERR_BAD_EXPERT_ID = 5,        /* device: a top-k id outside [0, E) */
    NVFP4_ERR_NONFINITE = 6,            /* device: a row maximum was Inf or NaN */
    NVFP4_ERR_DEVICE_TIMEOUT = 7,       /* device: a bounded pipeline wait ran out */
    NVFP4_ERR_CAPACITY = 8              /* device: an expert got more (token, slot) pairs than the
                                           fixed capacity; the excess pairs were dropped */
} nvfp4_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* nvfp4_status_string(int status);

/* rows rounded up to a multiple of 128 (the GEMM M tile). */
int64_t nvfp4_rows_padded(int64_t rows);

/* Bytes of the block-scale array of an NVFP4 matrix of rows x cols
 * (cols % 64 == 0): nvfp4_rows_padded(rows) * cols / 16.  0 on bad input. */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);

/*
 * nvfp4_quantize_rows -- two-level NVFP4 quantisation of each row of a BF16
 * matrix [miniTE/differs]: g = max|row| / 2688 (FP32 divide);
 * s_b = E4M3_rne(bmax_b / (g*6)) for each 16-element block; code =
 * E2M1_rne(x / (g*s_b)) with the sign of x; a zero row, or a block whose
 * divisor g*s_b is 0, gets zero codes.  Used for weight rows (one row per
 * output channel, along the reduction dimension) and for any activation rows.
 *
 *  x_dev      BF16 [rows][ld], 16-byte aligned, ld % 8 == 0, ld >= cols
 *  rows       >= 0;  cols % 64 == 0, 64 <= cols <= 8192
 *  codes_dev  uint8 [nvfp4_rows_padded(rows)][cols/2], 32-byte aligned
 *  sf_dev     nvfp4_sf_bytes(rows, cols) bytes, 16-byte aligned
 *  g_dev      float [rows]
 * The rows between rows and rows_pad get zero codes and zero scales.
 * Device error: NVFP4_ERR_NONFINITE if a row holds Inf/NaN.
 */
nvfp4_status nvfp4_quantize_rows(const void* x_dev, int64_t rows, int64_t cols, int64_t ld,
                                 void* codes_dev, void* sf_dev, float* g_dev, void* stream);

/* ------------------------------------------------------------------------
 * MoE layer.  Shapes: T tokens, H hidden, I expert intermediate (FC1 has 2I
 * outputs: gate rows 0..I-1 then up rows I..2I-1), E experts, top-k.
 * Supported: H % 256 == 0, 256 <= H <= 8192; I % 128 == 0, 128 <= I <= 8192;
 * 1 <= E <= 1024; 1 <= k <= min(E, 32); 0 <= T, T*k < 2^30.
 * --------------------------------------------------------------------- */

/* Quantised expert weights, as written by nvfp4_quantize_rows over the
 * [E*2I, H] view of W1 and the [E*H, I] view of W2. */
typedef struct {
    const void*  w1_codes;  /* uint8 [E*2I][H/2]            */
    const void*  w1_sf;     /* nvfp4_sf_bytes(E*2I, H) bytes */
    const float* w1_g;      /* [E*2I]                        */
    const void*  w2_codes;  /* uint8 [E*H][I/2]             */
    const void*  w2_sf;     /* nvfp4_sf_bytes(E*H, I) bytes  */
    const float* w2_g;      /* [E*H]                         */
    int32_t E, H, I;
} moe_nvfp4_weights;

/* Byte offsets of the sub-buffers of a MoE workspace (all 256-byte aligned).
 * The routed rows are expert-contiguous; expert e owns rows
 * [expert_offsets[e], expert_offsets[e+1]), a multiple of 128 rows whose
 * first count_e rows are its (token, slot) pairs in token-then-slot order
 * and the rest padding. */
typedef struct {
    int64_t T; int32_t H, I, E, k;
    int64_t rows_cap;     /* capacity of routed rows: every buffer below has this many */
    int64_t n_chunks;     /* 256-token chunks of the route sort */
    size_t a_codes;       /* uint8 [rows_cap][H/2]   quantised X rows (FC1 A operand) */
    size_t a_sf;          /* nvfp4_sf_bytes(rows_cap, H) */
    size_t a_g;           /* float [rows_cap]        g^x of each routed row */
    size_t row_pair;      /* int32 [rows_cap]        token*k + slot, -1 for a pad row */
    size_t row_prob;      /* float [rows_cap]        router probability of the row */
    size_t amax2;         /* uint32 [rows_cap]       bits of max|h| of the row (FC2 maxima) */
    size_t pair_row;      /* int32 [T*k]             routed row of each (token, slot), -1 if
                                                     the fixed-capacity layout dropped it */
    size_t a_sf_rows;     /* uint8 [rows_cap][H/16]  route-sort scratch: the routed rows' block
                                                     scales row-major, before they are arranged
                                                     into a_sf's tiles */
    size_t chunk_count;   /* int32 [E][n_chunks]     route-sort scratch */
    size_t chunk_base;    /* int32 [E][n_chunks]     route-sort scratch */
    size_t pair_rank;     /* int32 [T*k]             route-sort scratch */
    size_t expert_count;  /* int32 [E]               unpadded rows per expert */
    size_t route_end;     /* bytes used by moe_route_sort_amax (prefix of the workspace) */
    size_t h;             /* bf16 [rows_cap][I]      SwiGLU x prob (FC2 input before requant) */
    size_t a2_codes;      /* uint8 [rows_cap][I/2]   requantised h (FC2 A operand) */
    size_t a2_sf;         /* nvfp4_sf_bytes(rows_cap, I) */
    size_t a2_g;          /* float [rows_cap] */
    size_t y;             /* bf16 [rows_cap][H]      FC2 output per routed row (pad rows unwritten) */
    size_t total;         /* == moe_workspace_bytes(T, H, I, E, k) */
} moe_workspace_layout;

/* Fill *out with the workspace layout for this shape.  Host only. */
nvfp4_status moe_workspace_layout_query(int64_t T, int H, int I, int E, int k,
                                        moe_workspace_layout* out);

/* Workspace bytes a forward of this shape needs (0 on unsupported shape).
 * The size is a static capacity: it depends on the shape only, never on the
 * routing, so no host synchronisation is needed to size it. */
size_t moe_workspace_bytes(int64_t T, int H, int I, int E, int k);

/*
 * moe_route_sort_amax -- route sort + per-token amax + pad + NVFP4 quantise
 * of the FC1 input [miniTE/use].  Counting sort of the (token, slot) pairs by
 * expert, stable in token-then-slot order; each expert's rows padded to a
 * multiple of 128; each token row read once, its max|x| taken in the same
 * pass, quantised once (as nvfp4_quantize_rows) and written to its k routed
 * rows.  Also records each row's (token, slot) and router probability, each
 * (token, slot)'s row (pair_row), and zeroes the FC2 maxima.  Pad rows get
 * zero scales and g = 0.
 *
 *  x_dev           BF16 [T][H], 16-byte aligned
 *  topk_ids_dev    int32 [T][k], slot order = top-k order
 *  topk_w_dev      float [T][k], the router probability of each slot
 *  expert_offsets_dev  int32 [E+1], written: padded row starts, [E] = total rows
 *  ws_dev, ws_bytes    workspace of at least moe_workspace_bytes(T,H,I,E,k)
 *                  bytes (any I: only the prefix layout.route_end is touched),
 *                  256-byte aligned
 * Device errors: NVFP4_ERR_BAD_EXPERT_ID, NVFP4_ERR_NONFINITE.
 */
nvfp4_status moe_route_sort_amax(const void* x_dev, int64_t T, int H, int E, int k,
                                 const int32_t* topk_ids_dev, const float* topk_w_dev,
                                 int32_t* expert_offsets_dev,
                                 void* ws_dev, size_t ws_bytes, void* stream);

/*
 * moe_route_sort_amax_noalloc -- moe_route_sort_amax for callers that cannot
 * provide scratch memory.  The source pages have no counterpart to this
 * entry point: it is an interface addition of this library.
 *
 * Who needs it: callers whose device memory is planned once at start-up (a
 * serving engine that assigns every byte up front, an embedded runtime with
 * no allocator of its own), and hot paths that must not call cudaMalloc
 * because it can synchronise the device.  Such a caller has its inputs and
 * its output buffers but no spare scratch to hand over.
 *
 * What it does: exactly what moe_route_sort_amax does, with bit-identical
 * outputs.  Its scratch (per-chunk expert counts, chunk base rows, per-pair
 * ranks, per-expert counts) lives in a 2 MiB array inside the library, held
 * on every GPU that loads the library until the process exits.  Nothing is
 * allocated or freed by this call (no cudaMalloc, cudaFree or allocating
 * library routine).
 *
 *  x_dev, T, H, E, k, topk_ids_dev, topk_w_dev, expert_offsets_dev
 *                   as for moe_route_sort_amax
 *  out_dev          the routed-row outputs: the first
 *                   moe_workspace_layout.chunk_count bytes of a workspace laid
 *                   out as moe_workspace_layout_query(T, H, I, E, k) describes
 *                   (codes, scales, g^x, row pair, row probability, FC2 maxima,
 *                   pair rows, row-major scales; these offsets do not depend on
 *                   I), 256-byte aligned.  A full
 *                   workspace can be passed; its scratch part is not touched.
 *  out_bytes        size of out_dev; at least layout.chunk_count
 *
 * Limits and errors: shapes whose scratch would exceed 2 MiB
 * (8*E*ceil(T/256) + 4*T*k + 4*E bytes, each part rounded up to 256; e.g.
 * about 58,000 tokens at E = 128, k = 8) are rejected with
 * NVFP4_ERR_UNSUPPORTED_SHAPE before anything is launched; other argument
 * errors as for moe_route_sort_amax.
 *
 * Set-up and sharing: the first call on a device looks up the array's device
 * address (host-side, once per device, with that device current; again after a
 * device reset gives the device a new context); make that first call before any
 * stream capture.  Every call on a device shares the
 * one array and leaves its contents behind; no part of it needs to start at
 * zero.  Calls that can overlap on the GPU (on different streams without an
 * ordering between them) race on the array and must not be issued.
 */
nvfp4_status moe_route_sort_amax_noalloc(const void* x_dev, int64_t T, int H, int E, int k,
                                         const int32_t* topk_ids_dev, const float* topk_w_dev,
                                         int32_t* expert_offsets_dev, void* out_dev,
                                         size_t out_bytes, void* stream);

/*
 * moe_expert_forward_nvfp4 -- the expert forward after the route sort:
 * FC1 grouped GEMM (tcgen05 block-scaled FP4, FP32 accumulate) with the
 * epilogue v = (acc*g^x)*g^w, BF16 gate/up, h = bf16(f32(silu(gate)*up)*p)
 * and the row maxima of h; requantisation of h with those maxima; FC2
 * grouped GEMM with the same epilogue, BF16 y per routed row (each tile's
 * rows written contiguously); and the combine out[t] = bf16(sum over slots
 * 0..k-1 in order, FP32) of the rows pair_row names
 * [miniTE/differs, miniTE/use, RL/4.4, RL/4.5].  Equivalent to
 * moe_fc1_swiglu_nvfp4, moe_requant_nvfp4, moe_fc2_nvfp4, moe_combine_bf16 (bitwise).
 *
 *  w                   quantised weights (host struct, device pointers)
 *  T, k                as given to moe_route_sort_amax
 *  expert_offsets_dev  as written by moe_route_sort_amax
 *  out_dev             BF16 [T][H], 16-byte aligned
 *  ws_dev, ws_bytes    the workspace moe_route_sort_amax filled
 * Device error: NVFP4_ERR_DEVICE_TIMEOUT (a pipeline wait ran out).
 */
nvfp4_status moe_expert_forward_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k,
                                      const int32_t* expert_offsets_dev, void* out_dev,
                                      void* ws_dev, size_t ws_bytes, void* stream);

/*
 * moe_layer_forward_nvfp4 -- the whole hot path in one call: moe_route_sort_amax
 * followed by moe_expert_forward_nvfp4, with the same results bit for bit
 * (out, expert_offsets and the workspace).  One call lets the FC1 kernel be
 * launched as a programmatic dependent of the route sort's last kernel: its
 * set-up (barriers, TMEM, the SiLU range) overlaps that kernel's tail, and it
 * reads the routed rows only once the route sort has completed.
 *
 *  w, T, k, out_dev, ws_dev, ws_bytes   as for moe_expert_forward_nvfp4
 *  x_dev, topk_ids_dev, topk_w_dev      as for moe_route_sort_amax (H and E from w)
 *  expert_offsets_dev                   int32 [E+1], written as moe_route_sort_amax writes it
 * Every argument is checked before anything is launched; errors and device
 * errors as for the two calls.
 */
nvfp4_status moe_layer_forward_nvfp4(const moe_nvfp4_weights* w, const void* x_dev, int64_t T, int k,
                                     const int32_t* topk_ids_dev, const float* topk_w_dev,
                                     int32_t* expert_offsets_dev, void* out_dev, void* ws_dev,
                                     size_t ws_bytes, void* stream);

/* The four stages of moe_expert_forward_nvfp4, callable one by one (the
 * "unfused API").  fc1_debug_dev / fc2_debug_dev may be NULL; if given they
 * receive the FP32 pre-cast epilogue values v of every real routed row:
 * float [rows_cap][2I] (gate columns then up columns) and float
 * [rows_cap][H]; pad rows are not written.  They take the contiguous layout
 * that moe_route_sort_amax writes; a workspace filled by
 * moe_route_sort_amax_masked runs through moe_expert_forward_nvfp4_masked. */
nvfp4_status moe_fc1_swiglu_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k,
                                  const int32_t* expert_offsets_dev, void* ws_dev,
                                  size_t ws_bytes, float* fc1_debug_dev, void* stream);
/* moe_fc1_swiglu_save_nvfp4 -- moe_fc1_swiglu_nvfp4 for a forward whose backward
 * will run (moe_expert_backward_ste): the same h and FC2 maxima, and the BF16 gate
 * and up values that the SwiGLU ran on, which the backward takes its SwiGLU
 * derivative at ([miniTE/differs]: the backward works on saved BF16
 * values).  gu_save_dev: BF16 [rows_cap][2I] (gate columns then up columns) of
 * every real routed row, pad rows not written; device memory owned by the caller,
 * 4-byte aligned (16-byte for the backward that reads it).  Other arguments and
 * errors as for moe_fc1_swiglu_nvfp4 (contiguous layout only); NVFP4_ERR_INVALID_ARG
 * if gu_save_dev is NULL or misaligned. */
nvfp4_status moe_fc1_swiglu_save_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k,
                                       const int32_t* expert_offsets_dev, void* ws_dev,
                                       size_t ws_bytes, void* gu_save_dev, void* stream);
nvfp4_status moe_requant_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k,
                               const int32_t* expert_offsets_dev, void* ws_dev,
                               size_t ws_bytes, void* stream);
nvfp4_status moe_fc2_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k,
                           const int32_t* expert_offsets_dev, void* ws_dev,
                           size_t ws_bytes, float* fc2_debug_dev, void* stream);
nvfp4_status moe_combine_bf16(const moe_nvfp4_weights* w, int64_t T, int k, void* out_dev,
                              void* ws_dev, size_t ws_bytes, void* stream);

/* moe_fc2_requant_nvfp4 -- moe_requant_nvfp4 and moe_fc2_nvfp4 as one kernel: the FC2 input h
 * is requantised inside the FC2 kernel and never goes back through memory as NVFP4
 * ("miniTE diagnoses and narrows the cross-engine execution gap of NVFP4 RL", section
 * "Assumptions and limits": the online amax-quantisation-GEMM fusion).  Each FC2 work unit
 * quantises the 128 routed rows of its m-tile once into shared memory, with
 * g2 = amax2 / 2688 from the maxima FC1 reduced, and keeps them there while the W2 tiles of
 * its n-tiles stream through.  The codes, scales and outer scales are those
 * moe_requant_nvfp4 writes and the MMAs walk K in the same order, so y (and fc2_debug_dev)
 * are bitwise those of the two stages.  The workspace's requantised-operand buffers
 * (a2_codes, a2_sf, a2_g) are not written.  Reads h, amax2 and the row map that
 * moe_fc1_swiglu_nvfp4 and the route sort left in the workspace.
 * Supported for I <= moe_fc2_requant_max_intermediate() (768: two A buffers of 128 rows must
 * fit in shared memory beside the W2 stages and the staging of h) and E <= 512; other shapes
 * return NVFP4_ERR_UNSUPPORTED_SHAPE.  moe_expert_forward_nvfp4 runs the two separate stages,
 * which are faster on GB300 at the sizes measured (the quantisation inside FC2 is issue-bound
 * on the warps left beside FC2's own); this call gives the same bits with one launch less. */
nvfp4_status moe_fc2_requant_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k,
                                   const int32_t* expert_offsets_dev, void* ws_dev,
                                   size_t ws_bytes, float* fc2_debug_dev, void* stream);
/* Largest expert intermediate size moe_fc2_requant_nvfp4 takes (host only). */
int moe_fc2_requant_max_intermediate(void);

/* Fixed-capacity ("masked") layout -- a second way to lay the routed rows out: expert e owns
 * rows [e*capacity, (e+1)*capacity) whatever the batch, its pairs first (token, slot order),
 * then pad rows; expert_offsets[e] = e*capacity.  ("Finishing RL training faster: bitwise
 * consistency, high performance, agent-driven", section 4.4 "Expert GEMM: two layouts, same row
 * result": the rollout's masked per-expert layout and the trainer's contiguous one must give
 * bitwise-identical rows.)  Every routed row is computed exactly as in the contiguous layout, so
 * moe_expert_forward_nvfp4_masked returns the same output bits as moe_expert_forward_nvfp4 as
 * long as no expert gets more than `capacity` pairs; pairs past it are dropped, the device error
 * word records NVFP4_ERR_CAPACITY and the output is then unspecified.
 *  capacity   rows per expert, a multiple of 128, >= 128, E*capacity < 2^30
 * The workspace has E*capacity routed rows: size it with the _masked queries.  T == 0 writes
 * nothing. */
nvfp4_status moe_workspace_layout_query_masked(int64_t T, int H, int I, int E, int k, int capacity,
                                               moe_workspace_layout* layout);
size_t moe_workspace_bytes_masked(int64_t T, int H, int I, int E, int k, int capacity);
nvfp4_status moe_route_sort_amax_masked(const void* x_dev, int64_t T, int H, int E, int k,
                                        const int32_t* topk_ids_dev, const float* topk_w_dev, int capacity,
                                        int32_t* expert_offsets_dev, void* ws_dev, size_t ws_bytes, void* stream);
nvfp4_status moe_expert_forward_nvfp4_masked(const moe_nvfp4_weights* w, int64_t T, int k, int capacity,
                                             const int32_t* expert_offsets_dev, void* out_dev, void* ws_dev,
                                             size_t ws_bytes, void* stream);
/* moe_route_sort_amax_masked followed by moe_expert_forward_nvfp4_masked in one call, as
 * moe_layer_forward_nvfp4 is for the contiguous layout (FC1 launched as a programmatic
 * dependent of the route sort; every argument checked before anything is launched); the
 * same results bit for bit. */
nvfp4_status moe_layer_forward_nvfp4_masked(const moe_nvfp4_weights* w, const void* x_dev, int64_t T, int k,
                                            const int32_t* topk_ids_dev, const float* topk_w_dev, int capacity,
                                            int32_t* expert_offsets_dev, void* out_dev, void* ws_dev,
                                            size_t ws_bytes, void* stream);

/* moe_router_topk -- the router step that produces the inputs of
 * moe_route_sort_amax: logits[t, e] = sum_h x[t, h] * W_r[e, h] (BF16 inputs, FP32
 * tensor-core accumulation, K walked in one fixed order, so a token's logits, ids and
 * probabilities do not depend on T or on the other tokens), then the k largest logits
 * (larger first, lower expert id first on equal logits) and their probabilities, the
 * softmax over all experts renormalised over the k chosen (computed as the softmax of the
 * chosen, p_j = exp(l_j - l_1) / sum_i exp(l_i - l_1), FP32, sum in slot order).
 * ("Finishing RL training faster: bitwise consistency, high performance, agent-driven",
 * section 4.1 "Dense GEMM": one FP32-output router GEMM for every batch size; section 2:
 * top-k ties and order fixed.)
 *  x_dev           BF16 [T][H], 16-byte aligned; H % 64 == 0
 *  w_router_dev    BF16 [E][H] (row e = expert e), 16-byte aligned; E % 16 == 0, 16 <= E <= 256
 *  k               1 <= k <= min(E, 32)
 *  topk_ids_dev    int32 [T][k] out, slot order; 4-byte aligned
 *  topk_w_dev      float [T][k] out, 4-byte aligned
 *  logits_dev      float [T][E] out, 32-byte aligned, or NULL
 * The caller owns every buffer; nothing is allocated.  Non-finite logits are recorded as
 * NVFP4_ERR_NONFINITE (nvfp4_get_device_error). */
nvfp4_status moe_router_topk(const void* x_dev, int64_t T, int H, const void* w_router_dev, int E, int k,
                             int32_t* topk_ids_dev, float* topk_w_dev, float* logits_dev, void* stream);

/* ---- Straight-through (STE) backward ----------------------------------------------------
 * ("miniTE diagnoses and narrows the cross-engine execution gap of NVFP4 RL", section "How it
 * differs": the backward is a straight-through approximation, BF16 GEMMs on the saved original
 * BF16 activations and weights; no quantisation runs backward.)  Each quantiser is taken as the
 * identity and every other op is differentiated where it ran, with the rows of the forward's
 * contiguous layout (moe_route_sort_amax); pair(r) = token*k + slot, t(r), p(r) as there:
 *   dh[r]        = bf16( dOut[t(r)] W2[e] )                            BF16 GEMM, FP32 accumulate
 *   a, u         = bf16 of the forward's FC1 values of r (the gate/up the SwiGLU ran on)
 *   dgate, dup   = bf16( dh p u silu'(a) ), bf16( dh p silu(a) ),     silu(a) = a / (1 + e^-a),
 *                  silu'(a) = s (1 + a (1 - s)), s = 1 / (1 + e^-a)   (FP32)
 *   dprob[pair]  = sum_i dh_i silu(a_i) u_i                             (FP32)
 *   dxs[pair]    = bf16( [dgate, dup] W1[e] )                          BF16 GEMM
 *   dX[t]        = bf16( sum over slots 0..k-1 in order of dxs[t*k+j], FP32 )
 *   dW2[e]       = sum over e's rows of dOut[t(r)]^T h[r]               FP32
 *   dW1[e]       = sum over e's rows of [dgate, dup][r]^T x[t(r)]        FP32
 * A token's dX and dprob do not depend on the other tokens of the batch. */

/* The BF16 original weights, as given to the weight quantiser; the backward GEMMs read them in
 * place (MN-major operands):
 *   w1  BF16 [E][2I][H], gate rows then up rows per expert  (16-byte aligned)
 *   w2  BF16 [E][H][I]                                      (16-byte aligned) */
typedef struct {
    const void* w1;
    const void* w2;
    int32_t E, H, I;
} moe_bf16_weights_t;

/* Byte offsets of the backward workspace's scratch buffers (256-byte aligned); rows_cap is
 * the forward layout's. */
typedef struct {
    int64_t T; int32_t H, I, E, k;
    int64_t rows_cap;
    size_t dy_rows;   /* bf16 [rows_cap][H]  dOut gathered per routed row */
    size_t dh;        /* bf16 [rows_cap][I] */
    size_t dgu;       /* bf16 [rows_cap][2I] dgate then dup */
    size_t dx_pairs;  /* bf16 [T*k][H]       dX per (token, slot) */
    size_t x_rows;    /* bf16 [rows_cap][H]  x gathered per routed row */
    size_t real_end;  /* int32 [E]           end of each expert's real routed rows */
    size_t total;
} moe_backward_layout;

nvfp4_status moe_backward_layout_query(int64_t T, int H, int I, int E, int k, moe_backward_layout* layout);
size_t moe_backward_workspace_bytes(int64_t T, int H, int I, int E, int k);

/* moe_expert_backward_ste -- the gradients of one forward, from what it saved.
 *  w                    the BF16 originals (host struct, device pointers)
 *  T, k                 as given to the forward
 *  x_dev                BF16 [T][H], the forward's input; 16-byte aligned
 *  dout_dev             BF16 [T][H], the gradient of the forward's output; 16-byte aligned
 *  expert_offsets_dev   as moe_route_sort_amax wrote it for this forward (contiguous layout)
 *  fwd_ws_dev, fwd_ws_bytes  the forward's workspace after the forward (its row map, router
 *                       probabilities and h are read)
 *  gu_dev               BF16 [rows_cap][2I], what moe_fc1_swiglu_save_nvfp4 wrote to its
 *                       gu_save_dev in this forward (the BF16 gate/up of every real routed
 *                       row); 16-byte aligned
 *  dx_dev               BF16 [T][H] out; 16-byte aligned
 *  dw1_dev, dw2_dev     FP32 [E][2I][H] and [E][H][I] out (overwritten); 32-byte aligned
 *  dprob_dev            FP32 [T][k] out, the gradient of topk_w; 4-byte aligned
 *  bwd_ws_dev, bwd_ws_bytes  scratch, moe_backward_workspace_bytes(T, H, I, E, k) bytes,
 *                       256-byte aligned
 * Nothing is allocated and nothing synchronises; every output is written in stream order.
 * T == 0 zeroes dW1 and dW2.  Argument errors as for moe_expert_forward_nvfp4, and
 * NVFP4_ERR_UNSUPPORTED_SHAPE if rows_cap >= 2^30; device error NVFP4_ERR_DEVICE_TIMEOUT (a
 * pipeline wait ran out). */
nvfp4_status moe_expert_backward_ste(const moe_bf16_weights_t* w, int64_t T, int k, const void* x_dev,
                                     const void* dout_dev, const int32_t* expert_offsets_dev, const void* fwd_ws_dev,
                                     size_t fwd_ws_bytes, const void* gu_dev, void* dx_dev, float* dw1_dev,
                                     float* dw2_dev, float* dprob_dev, void* bwd_ws_dev, size_t bwd_ws_bytes,
                                     void* stream);

/* nvfp4_silu_table -- the SiLU that the FC1 epilogue applies to its BF16 gate values
 * ([RL/4.4]: SiLU(gate)*up in FP32), evaluated by the epilogue's own code for every input:
 * out_dev float [65536], entry i = silu(a) for the BF16 value a whose bit pattern is i, where
 * silu(a) = a / (1 + e^-a) rounded once (to nearest, ties to even) to FP32; silu(+-0) = +-0,
 * silu(+inf) = +inf, silu(-inf) and silu(NaN) are NaN.  The values come from a table that is
 * part of the library's device image (computed when the library is built, so no call has to
 * fill it first) and, outside 2^-24 <= |a| < 2^7, from closed forms that give the same bits.
 * out_dev: device memory, 4-byte aligned, 262144 bytes, owned by the caller.  Enqueued on
 * `stream` (one small kernel); returns NVFP4_ERR_CUDA if it cannot be. */
nvfp4_status nvfp4_silu_table(float* out_dev, void* stream);

/* The CUDA runtime error (a cudaError_t value) behind the calling thread's most recent
 * NVFP4_ERR_CUDA, or 0 if no call of this thread has returned NVFP4_ERR_CUDA.  Host only; it
 * neither synchronises nor clears anything. */
int nvfp4_last_cuda_error(void);
/* cudaGetErrorName of a cudaError_t value (static string, never NULL).  Host only. */
const char* nvfp4_cuda_error_name(int error);

/* Synchronise `stream`, then report and clear this device's error word:
 * *device_status receives NVFP4_OK or the first device error recorded since
 * the last call.  Returns NVFP4_ERR_CUDA if the synchronisation failed. */
nvfp4_status nvfp4_get_device_error(void* stream, int* device_status);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_MOE_H */
