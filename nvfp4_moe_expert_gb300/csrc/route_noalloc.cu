// moe_route_sort_amax_noalloc: the route sort + per-token amax + pad +
// quantise of moe_route_sort_amax, with its scratch (per-chunk expert counts,
// chunk base rows, per-pair ranks, per-expert counts) in a fixed device array
// owned by this library instead of in caller-provided memory.
//
// It exists for callers that cannot provide scratch memory: code whose device
// memory is planned once at start-up (a serving engine that assigns every
// byte up front, an embedded runtime without an allocator of its own), and
// hot paths that must not call cudaMalloc because it can synchronise the
// device.  Such a caller passes only its inputs and the output buffers.
#include <mutex>

#include "common.cuh"

namespace nvfp4 {
namespace {

// Largest scratch one call may use; shapes that need more are rejected.
constexpr size_t kRouteScratchBytes = size_t(2) << 20;   // 2 MiB

// The scratch array.  Every GPU that loads the library holds it until the
// process exits.  All calls on a device share it and it keeps the last call's
// contents; nothing in it has to start at zero, because each call writes every
// word it later reads.  Calls whose executions overlap on the GPU (different
// streams, no ordering between them) race on it.
static __device__ __align__(256) uint8_t g_route_scratch[kRouteScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
uint8_t* g_scratch_addr[kMaxDevices];
void* g_scratch_ctx[kMaxDevices];

// Device address of g_route_scratch on device `dev` (which must be current).
// In host code the array's name is only a host-side stand-in, so the address
// is looked up once per device and cached with the context it was looked up
// in; after a device reset (a new context, the library's module loaded again)
// it is looked up anew instead of reusing an address that no longer exists.
uint8_t* scratch_address(int dev) {
    void* ctx = current_context();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_addr[dev] = static_cast<uint8_t*>(p);
        g_scratch_ctx[dev] = ctx;
    }
    return g_scratch_addr[dev];
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status moe_route_sort_amax_noalloc(const void* x_dev, int64_t T, int H, int E, int k,
                                                    const int32_t* topk_ids_dev, const float* topk_w_dev,
                                                    int32_t* expert_offsets_dev, void* out_dev, size_t out_bytes,
                                                    void* stream) {
    moe_workspace_layout L;
    if (moe_workspace_layout_query(T, H, 128, E, k, &L) != NVFP4_OK) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!expert_offsets_dev || !out_dev) return NVFP4_ERR_INVALID_ARG;
    if (T > 0 && (!x_dev || !topk_ids_dev || !topk_w_dev)) return NVFP4_ERR_INVALID_ARG;
    const auto aligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
    if (!aligned(x_dev, 16) || !aligned(out_dev, 256) || !aligned(topk_ids_dev, 4) || !aligned(topk_w_dev, 4) ||
        !aligned(expert_offsets_dev, 4))
        return NVFP4_ERR_INVALID_ARG;
    // the outputs are the routed rows, which come first in the workspace layout
    if (out_bytes < L.chunk_count) return NVFP4_ERR_WORKSPACE_TOO_SMALL;

    const size_t cc_bytes = align256(static_cast<size_t>(E) * L.n_chunks * 4);
    const size_t pr_bytes = align256(static_cast<size_t>(T) * k * 4);
    const size_t ec_bytes = align256(static_cast<size_t>(E) * 4);
    if (2 * cc_bytes + pr_bytes + ec_bytes > kRouteScratchBytes) return NVFP4_ERR_UNSUPPORTED_SHAPE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    uint8_t* scratch = scratch_address(dev);
    int* err = device_error_word();
    if (!scratch || !err) return NVFP4_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(out_dev);
    RouteBufs b;
    b.a_codes = ws + L.a_codes;
    b.a_sf = ws + L.a_sf;
    b.a_g = reinterpret_cast<float*>(ws + L.a_g);
    b.row_pair = reinterpret_cast<int32_t*>(ws + L.row_pair);
    b.row_prob = reinterpret_cast<float*>(ws + L.row_prob);
    b.amax2 = reinterpret_cast<uint32_t*>(ws + L.amax2);
    b.pair_row = reinterpret_cast<int32_t*>(ws + L.pair_row);
    b.a_sf_rows = ws + L.a_sf_rows;
    b.rows_cap = L.rows_cap;
    b.chunk_count = reinterpret_cast<int32_t*>(scratch);
    b.chunk_base = reinterpret_cast<int32_t*>(scratch + cc_bytes);
    b.pair_rank = reinterpret_cast<int32_t*>(scratch + 2 * cc_bytes);
    b.expert_count = reinterpret_cast<int32_t*>(scratch + 2 * cc_bytes + pr_bytes);
    b.n_chunks = L.n_chunks;
    const cudaError_t e = launch_route_sort_quant(static_cast<const uint16_t*>(x_dev), T, H, E, k, topk_ids_dev,
                                                  topk_w_dev, expert_offsets_dev, b, err,
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
