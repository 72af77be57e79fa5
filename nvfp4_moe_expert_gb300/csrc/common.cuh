// Shared definitions of the CUDA path: constants of the NVFP4 layout, the
// device error word protocol and the host-side launchers each .cu provides.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nvfp4_moe.h"

namespace nvfp4 {

constexpr int kBlock = 16;          // elements per E4M3 block scale
constexpr int kTileM = 128;         // GEMM M tile = row padding of each expert
constexpr int kSfAtomBytes = 512;   // one 128-row x 64-column scale tile
constexpr float kOuterDivisor = 2688.0f;   // 6 * 448

// Byte offset of the E4M3 scale of (row r, block b) in a matrix with `cols` columns.
__host__ __device__ inline size_t sf_offset(int64_t r, int64_t b, int64_t cols) {
    return static_cast<size_t>(((r >> 7) * (cols >> 6) + (b >> 2)) * kSfAtomBytes + (r & 31) * 16 +
                               ((r & 127) >> 5) * 4 + (b & 3));
}

// Byte of block scale (row r, 16-element block b) in the row-major scale layout of the routed
// activation operands: [rows][cols/16].
__host__ __device__ inline size_t sf_row_offset(int64_t r, int64_t b, int64_t cols) {
    return static_cast<size_t>(r * (cols / 16) + b);
}

// Record a device-side error (first one wins).
__device__ __forceinline__ void set_device_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch.  Inside one library call, every kernel after
// the first is launched with programmatic stream serialisation, so its CTAs may
// be scheduled while the previous kernel (also this library's) is finishing.
// Every kernel calls pdl_wait() before its first access to global memory that
// an earlier kernel may still be writing (it returns once the previous kernel
// has completed and its writes are visible; at once for a normal launch) and
// then pdl_launch_dependents() so that the next kernel can be scheduled early
// too.  The first kernel of a call is launched normally, so it is ordered after
// whatever the caller queued before (a programmatic launch is not ordered after a
// host-to-device copy); a later kernel may therefore read the call's inputs
// before its own wait once the kernel before it has passed its wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Cycles a pipeline wait may spin before it reports NVFP4_ERR_DEVICE_TIMEOUT (~2 s).
constexpr long long kWaitBudgetCycles = 4000000000LL;

// ---- host launchers (each defined in the .cu that holds the kernel) ----
struct RouteBufs {
    uint8_t* a_codes;
    uint8_t* a_sf;
    uint8_t* a_sf_rows;  // [rows_cap][H/16] the scatter's scales, row-major, before the tile step
    float* a_g;
    int32_t* row_pair;
    float* row_prob;
    uint32_t* amax2;
    int32_t* pair_row;   // [T*k] routed row of each (token, slot), -1 if dropped
    int32_t* chunk_count;
    int32_t* chunk_base;
    int32_t* pair_rank;
    int32_t* expert_count;
    int64_t n_chunks;
    int64_t rows_cap;
    int direct_rows;   // set by the route launcher: pair_rank holds destination rows
};

cudaError_t launch_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                                 uint8_t* sf, float* g, int* err, cudaStream_t st);

cudaError_t launch_route_sort_quant(const uint16_t* x, int64_t T, int H, int E, int k, const int32_t* ids,
                                    const float* probs, int32_t* offsets, const RouteBufs& b, int* err,
                                    cudaStream_t st);

cudaError_t launch_requant(const uint16_t* h, const uint32_t* amax2, const int32_t* row_pair,
                           const int32_t* offsets, int E, int64_t rows_cap, int I, uint8_t* codes, uint8_t* sf,
                           float* g, int* err, cudaStream_t st, bool pdl);

struct GemmArgs {
    // operands
    const uint8_t* a_codes;   // [rows_cap][K/2]
    const uint8_t* a_sf;
    const float* a_g;         // per routed row
    const uint8_t* b_codes;   // [E*Nw][K/2]
    const uint8_t* b_sf;
    const float* b_g;         // [E*Nw]
    int64_t rows_cap;
    int K;                    // reduction length (H for FC1, I for FC2)
    int Nw;                   // weight rows per expert (2I for FC1, H for FC2)
    int E;
    const int32_t* offsets;   // [E+1] padded expert row starts
    const int32_t* row_pair;  // token*k + slot or -1
    const float* row_prob;
    // FC1 outputs
    int I;
    uint16_t* h;              // [rows_cap][I]
    uint32_t* amax2;          // [rows_cap]
    // FC2 outputs
    int H;
    uint16_t* y;              // [rows_cap][H], per routed row
    float* debug;             // optional pre-cast FP32 values
    uint16_t* gu_save;        // optional FC1 BF16 gate/up [rows_cap][2I] (the values SwiGLU runs on)
    int* err;
};

cudaError_t launch_fc1(const GemmArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_fc2(const GemmArgs& a, cudaStream_t st, bool pdl);
// FC2 with the requantisation of h fused in (reads h, amax2 and row_pair; a_codes/a_sf/a_g
// unused); supports I <= fc2_requant_max_i() and E <= fc2_requant_max_e().
cudaError_t launch_fc2_requant(const GemmArgs& a, cudaStream_t st, bool pdl);
int fc2_requant_max_i();
int fc2_requant_max_e();
// Copy the FC1 epilogue's 65536-entry SiLU table (FP32, by BF16 bit pattern) to `out`.
cudaError_t copy_silu_table(float* out, cudaStream_t st);

// rows: the y row of each (token, slot) (rows[t*k+s], -1 for none), or nullptr for y in
// (token, slot) order.
cudaError_t launch_combine(const uint16_t* y, const int32_t* rows, int64_t T, int k, int H, uint16_t* out,
                           cudaStream_t st, bool pdl);

int device_sm_count();

// Device address of this device's error word (nullptr if it cannot be looked up).
int* device_error_word();

// The calling thread's current CUDA context (nullptr if it cannot be read).  Device
// addresses of the library's __device__ variables are cached per device together with the
// context they were looked up in, and looked up again when the context changes (a device
// reset tears the old one down and loads the library's module again elsewhere).
void* current_context();

}  // namespace nvfp4
