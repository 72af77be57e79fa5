// Arguments of the straight-through backward (backward.cu), filled by the C ABI (api.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

struct BackwardArgs {
    int64_t T;
    int H, I, E, k;
    int64_t rows_cap;          // routed-row capacity of the forward's layout
    const uint16_t* w1t;       // BF16 [E][H][2I]: W1 transposed per expert
    const uint16_t* w2t;       // BF16 [E][I][H]: W2 transposed per expert
    const uint16_t* x;         // BF16 [T][H]
    const uint16_t* dout;      // BF16 [T][H]
    const int32_t* offsets;    // [E+1] padded expert row starts
    const int32_t* row_pair;   // [rows_cap] token*k + slot, -1 for a pad row
    const float* row_prob;     // [rows_cap]
    const uint16_t* h;         // BF16 [rows_cap][I], the forward's SwiGLU x prob
    const float* fc1_pre;      // FP32 [rows_cap][2I], the forward's FC1 values before the BF16 cast
    uint16_t* dx;              // BF16 [T][H]
    float* dw1;                // FP32 [E][2I][H]
    float* dw2;                // FP32 [E][H][I]
    float* dprob;              // FP32 [T*k]
    // scratch (the backward workspace)
    uint16_t* dy_rows;         // [rows_cap][H]
    uint16_t* dh;              // [rows_cap][I]
    uint16_t* dgu;             // [rows_cap][2I]
    uint16_t* dx_pairs;        // [T*k][H]
    uint16_t* dy_t;            // [H][rows_cap]
    uint16_t* h_t;             // [I][rows_cap]
    uint16_t* dgu_t;           // [2I][rows_cap]
    uint16_t* x_t;             // [H][rows_cap]
    int* err;
};

cudaError_t launch_moe_backward_ste(const BackwardArgs& a, cudaStream_t st);

// out[b][c][r] = in[b][r][c]; rows % 64 == 0, cols % 64 == 0, 16-byte aligned.
cudaError_t launch_transpose_bf16(const uint16_t* in, int64_t batch, int64_t rows, int64_t cols, uint16_t* out,
                                  cudaStream_t st);

}  // namespace nvfp4
