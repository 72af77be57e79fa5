// Arguments of the straight-through backward (backward.cu), filled by the C ABI (api.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

struct BackwardArgs {
    int64_t T;
    int H, I, E, k;
    int64_t rows_cap;          // routed-row capacity of the forward's layout
    const uint16_t* w1;        // BF16 [E][2I][H]: the original W1 (gate rows, then up rows)
    const uint16_t* w2;        // BF16 [E][H][I]: the original W2
    const uint16_t* x;         // BF16 [T][H]
    const uint16_t* dout;      // BF16 [T][H]
    const int32_t* offsets;    // [E+1] padded expert row starts
    const int32_t* row_pair;   // [rows_cap] token*k + slot, -1 for a pad row
    const float* row_prob;     // [rows_cap]
    const uint16_t* h;         // BF16 [rows_cap][I], the forward's SwiGLU x prob
    const uint16_t* gu;        // BF16 [rows_cap][2I], the forward's gate/up (the values its SwiGLU ran on)
    uint16_t* dx;              // BF16 [T][H]
    float* dw1;                // FP32 [E][2I][H]
    float* dw2;                // FP32 [E][H][I]
    float* dprob;              // FP32 [T*k]
    // scratch (the backward workspace)
    uint16_t* dy_rows;         // [rows_cap][H]
    uint16_t* dh;              // [rows_cap][I]
    uint16_t* dgu;             // [rows_cap][2I]
    uint16_t* dx_pairs;        // [T*k][H]
    uint16_t* x_rows;          // [rows_cap][H]: x gathered per routed row
    int32_t* real_end;         // [E]: end of each expert's real routed rows
    int* err;
};

cudaError_t launch_moe_backward_ste(const BackwardArgs& a, cudaStream_t st);

}  // namespace nvfp4
