// C ABI of the NVFP4 MoE expert forward: argument validation, workspace
// layout, per-device state (error word, SM count) and the launch sequences.
// The operations themselves are documented in include/nvfp4_moe.h.
#include <cstring>
#include <mutex>

#include "backward.cuh"
#include "common.cuh"

namespace nvfp4 {

// First device-side error since the last nvfp4_get_device_error (0 = none).
__device__ int g_device_error;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int* g_err_ptr[kMaxDevices];
void* g_err_ctx[kMaxDevices];
int g_sm_count[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        }
    });
    return fn;
}

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return (d >= 0 && d < kMaxDevices) ? d : -1;
}

// Device address of this device's error word (looked up once per device and context).
int* device_error_ptr() {
    const int d = current_device();
    if (d < 0) return nullptr;
    void* ctx = current_context();
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_err_ptr[d] || g_err_ctx[d] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[d] = static_cast<int*>(p);
        g_err_ctx[d] = ctx;
    }
    return g_err_ptr[d];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool moe_shape_ok(int64_t T, int H, int I, int E, int k) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return false;
    if (H < 256 || H > 8192 || H % 256) return false;
    if (I < 128 || I > 8192 || I % 128) return false;
    if (T * static_cast<int64_t>(k) >= (int64_t(1) << 30)) return false;
    return true;
}

// capacity > 0: the fixed-capacity layout, E*capacity routed rows (expert e at e*capacity).
void compute_layout(int64_t T, int H, int I, int E, int k, moe_workspace_layout* L, int capacity = 0) {
    std::memset(L, 0, sizeof(*L));
    L->T = T;
    L->H = H;
    L->I = I;
    L->E = E;
    L->k = k;
    const int64_t R = T * k;
    const int64_t live_experts = R < E ? R : E;
    L->rows_cap = capacity > 0 ? static_cast<int64_t>(E) * capacity
                               : (R + live_experts * (kTileM - 1) + kTileM - 1) / kTileM * kTileM;
    L->n_chunks = (T + 255) / 256;
    const int64_t rc = L->rows_cap;
    size_t o = 0;
    auto take = [&o](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L->a_codes = take(rc * H / 2);
    L->a_sf = take(rc * H / 16);
    L->a_g = take(rc * 4);
    L->row_pair = take(rc * 4);
    L->row_prob = take(rc * 4);
    L->amax2 = take(rc * 4);
    L->pair_row = take(R * 4);
    L->a_sf_rows = take(rc * H / 16);
    L->chunk_count = take(static_cast<size_t>(E) * L->n_chunks * 4);
    L->chunk_base = take(static_cast<size_t>(E) * L->n_chunks * 4);
    L->pair_rank = take(R * 4);
    L->expert_count = take(static_cast<size_t>(E) * 4);
    L->route_end = o;
    L->h = take(rc * I * 2);
    L->a2_codes = take(rc * I / 2);
    L->a2_sf = take(rc * I / 16);
    L->a2_g = take(rc * 4);
    L->y = take(rc * H * 2);
    L->total = o;
}

// Scratch of the straight-through backward (sizes from the forward's contiguous layout).
void compute_backward_layout(int64_t T, int H, int I, int E, int k, moe_backward_layout* B) {
    moe_workspace_layout L;
    compute_layout(T, H, I, E, k, &L);
    std::memset(B, 0, sizeof(*B));
    B->T = T;
    B->H = H;
    B->I = I;
    B->E = E;
    B->k = k;
    const int64_t rc = L.rows_cap;
    B->rows_cap = rc;
    size_t o = 0;
    auto take = [&o](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    B->dy_rows = take(rc * H * 2);
    B->dh = take(rc * I * 2);
    B->dgu = take(rc * 2 * I * 2);
    B->dx_pairs = take(T * k * H * 2);
    B->x_rows = take(rc * H * 2);
    B->real_end = take(static_cast<size_t>(E) * 4);
    B->total = o;
}

// The CUDA error behind the calling thread's last NVFP4_ERR_CUDA (cudaSuccess if none yet).
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

nvfp4_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return NVFP4_OK;
    t_last_cuda_error = e;
    return NVFP4_ERR_CUDA;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Shared validation of the calls that run on a filled workspace.
bool capacity_ok(int E, int capacity) {
    return capacity >= kTileM && capacity % kTileM == 0 && static_cast<int64_t>(E) * capacity < (int64_t(1) << 30);
}

nvfp4_status check_forward_args(const moe_nvfp4_weights* w, int64_t T, int k, const void* ws, size_t ws_bytes,
                                moe_workspace_layout* L, int capacity = 0) {
    if (!w || !ws) return NVFP4_ERR_INVALID_ARG;
    if (!w->w1_codes || !w->w1_sf || !w->w1_g || !w->w2_codes || !w->w2_sf || !w->w2_g) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(w->w1_codes, 16) || !aligned(w->w1_sf, 16) || !aligned(w->w2_codes, 16) || !aligned(w->w2_sf, 16) ||
        !aligned(ws, 256))
        return NVFP4_ERR_INVALID_ARG;
    if (!moe_shape_ok(T, w->H, w->I, w->E, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (capacity != 0 && !capacity_ok(w->E, capacity)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    compute_layout(T, w->H, w->I, w->E, k, L, capacity);
    if (ws_bytes < L->total) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    return NVFP4_OK;
}

GemmArgs fc1_args(const moe_nvfp4_weights* w, const int32_t* offsets, void* ws, const moe_workspace_layout& L,
                  float* debug, int* err) {
    GemmArgs a{};
    a.a_codes = at<uint8_t>(ws, L.a_codes);
    a.a_sf = at<uint8_t>(ws, L.a_sf);
    a.a_g = at<float>(ws, L.a_g);
    a.b_codes = static_cast<const uint8_t*>(w->w1_codes);
    a.b_sf = static_cast<const uint8_t*>(w->w1_sf);
    a.b_g = w->w1_g;
    a.rows_cap = L.rows_cap;
    a.K = w->H;
    a.Nw = 2 * w->I;
    a.E = w->E;
    a.offsets = offsets;
    a.row_pair = at<int32_t>(ws, L.row_pair);
    a.row_prob = at<float>(ws, L.row_prob);
    a.I = w->I;
    a.h = at<uint16_t>(ws, L.h);
    a.amax2 = at<uint32_t>(ws, L.amax2);
    a.H = w->H;
    a.y = nullptr;
    a.debug = debug;
    a.err = err;
    return a;
}

GemmArgs fc2_args(const moe_nvfp4_weights* w, const int32_t* offsets, void* ws, const moe_workspace_layout& L,
                  float* debug, int* err) {
    GemmArgs a{};
    a.a_codes = at<uint8_t>(ws, L.a2_codes);
    a.a_sf = at<uint8_t>(ws, L.a2_sf);
    a.a_g = at<float>(ws, L.a2_g);
    a.b_codes = static_cast<const uint8_t*>(w->w2_codes);
    a.b_sf = static_cast<const uint8_t*>(w->w2_sf);
    a.b_g = w->w2_g;
    a.rows_cap = L.rows_cap;
    a.K = w->I;
    a.Nw = w->H;
    a.E = w->E;
    a.offsets = offsets;
    a.row_pair = at<int32_t>(ws, L.row_pair);
    a.row_prob = at<float>(ws, L.row_prob);
    a.I = w->I;
    a.h = nullptr;
    a.amax2 = nullptr;
    a.H = w->H;
    a.y = at<uint16_t>(ws, L.y);
    a.debug = debug;
    a.err = err;
    return a;
}

}  // namespace

int* device_error_word() { return device_error_ptr(); }

void* current_context() {
    CtxGetCurrentFn fn = ctx_get_current_fn();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

int device_sm_count() {
    const int d = current_device();
    if (d < 0) return 1;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_sm_count[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n < 1) n = 1;
        g_sm_count[d] = n;
    }
    return g_sm_count[d];
}

}  // namespace nvfp4

using namespace nvfp4;

namespace nvfp4 {
// defined in quant.cu: the route sort with an optional fixed capacity per expert
cudaError_t launch_route_sort_quant_cap(const uint16_t* x, int64_t T, int H, int E, int k, const int32_t* ids,
                                        const float* probs, int32_t* offsets, const RouteBufs& b, int capacity,
                                        int* err, cudaStream_t st);
// defined in router.cu
cudaError_t launch_router_topk(const uint16_t* x, int64_t T, int H, const uint16_t* w, int E, int k, int32_t* ids,
                               float* probs, float* logits, int* err, cudaStream_t st);
}  // namespace nvfp4

extern "C" {

const char* nvfp4_status_string(int status) {
    switch (status) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
        case NVFP4_ERR_UNSUPPORTED_SHAPE: return "NVFP4_ERR_UNSUPPORTED_SHAPE";
        case NVFP4_ERR_WORKSPACE_TOO_SMALL: return "NVFP4_ERR_WORKSPACE_TOO_SMALL";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
        case NVFP4_ERR_BAD_EXPERT_ID: return "NVFP4_ERR_BAD_EXPERT_ID";
        case NVFP4_ERR_NONFINITE: return "NVFP4_ERR_NONFINITE";
        case NVFP4_ERR_DEVICE_TIMEOUT: return "NVFP4_ERR_DEVICE_TIMEOUT";
        case NVFP4_ERR_CAPACITY: return "NVFP4_ERR_CAPACITY";
        default: return "NVFP4_UNKNOWN_STATUS";
    }
}

int64_t nvfp4_rows_padded(int64_t rows) {
    if (rows < 0) return 0;
    return (rows + kTileM - 1) / kTileM * kTileM;
}

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols <= 0 || cols % 64) return 0;
    return static_cast<size_t>(nvfp4_rows_padded(rows)) * static_cast<size_t>(cols / 16);
}

nvfp4_status nvfp4_quantize_rows(const void* x_dev, int64_t rows, int64_t cols, int64_t ld, void* codes_dev,
                                 void* sf_dev, float* g_dev, void* stream) {
    if (rows < 0 || cols < 64 || cols > 8192 || cols % 64 || ld < cols || ld % 8) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return NVFP4_OK;
    if (!x_dev || !codes_dev || !sf_dev || !g_dev) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x_dev, 16) || !aligned(codes_dev, 32) || !aligned(sf_dev, 16) || !aligned(g_dev, 4))
        return NVFP4_ERR_INVALID_ARG;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    return from_cuda(launch_quantize_rows(static_cast<const uint16_t*>(x_dev), rows, cols, ld,
                                          static_cast<uint8_t*>(codes_dev), static_cast<uint8_t*>(sf_dev), g_dev, err,
                                          static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_workspace_layout_query(int64_t T, int H, int I, int E, int k, moe_workspace_layout* out) {
    if (!out) return NVFP4_ERR_INVALID_ARG;
    if (!moe_shape_ok(T, H, I, E, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    compute_layout(T, H, I, E, k, out);
    return NVFP4_OK;
}

size_t moe_workspace_bytes(int64_t T, int H, int I, int E, int k) {
    if (!moe_shape_ok(T, H, I, E, k)) return 0;
    moe_workspace_layout L;
    compute_layout(T, H, I, E, k, &L);
    return L.total;
}

static nvfp4_status route_impl(const void* x_dev, int64_t T, int H, int E, int k, const int32_t* topk_ids_dev,
                               const float* topk_w_dev, int32_t* expert_offsets_dev, void* ws_dev, size_t ws_bytes,
                               int capacity, void* stream) {
    if (!moe_shape_ok(T, H, 128, E, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (capacity != 0 && !capacity_ok(E, capacity)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!expert_offsets_dev || !ws_dev) return NVFP4_ERR_INVALID_ARG;
    if (T > 0 && (!x_dev || !topk_ids_dev || !topk_w_dev)) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x_dev, 16) || !aligned(ws_dev, 256) || !aligned(topk_ids_dev, 4) || !aligned(topk_w_dev, 4) ||
        !aligned(expert_offsets_dev, 4))
        return NVFP4_ERR_INVALID_ARG;
    moe_workspace_layout L;
    compute_layout(T, H, 128, E, k, &L, capacity);
    if (ws_bytes < L.route_end) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    RouteBufs b;
    b.a_codes = at<uint8_t>(ws_dev, L.a_codes);
    b.a_sf = at<uint8_t>(ws_dev, L.a_sf);
    b.a_g = at<float>(ws_dev, L.a_g);
    b.row_pair = at<int32_t>(ws_dev, L.row_pair);
    b.row_prob = at<float>(ws_dev, L.row_prob);
    b.amax2 = at<uint32_t>(ws_dev, L.amax2);
    b.pair_row = at<int32_t>(ws_dev, L.pair_row);
    b.a_sf_rows = at<uint8_t>(ws_dev, L.a_sf_rows);
    b.rows_cap = L.rows_cap;
    b.chunk_count = at<int32_t>(ws_dev, L.chunk_count);
    b.chunk_base = at<int32_t>(ws_dev, L.chunk_base);
    b.pair_rank = at<int32_t>(ws_dev, L.pair_rank);
    b.expert_count = at<int32_t>(ws_dev, L.expert_count);
    b.n_chunks = L.n_chunks;
    return from_cuda(launch_route_sort_quant_cap(static_cast<const uint16_t*>(x_dev), T, H, E, k, topk_ids_dev,
                                                 topk_w_dev, expert_offsets_dev, b, capacity, err,
                                                 static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_route_sort_amax(const void* x_dev, int64_t T, int H, int E, int k, const int32_t* topk_ids_dev,
                                 const float* topk_w_dev, int32_t* expert_offsets_dev, void* ws_dev, size_t ws_bytes,
                                 void* stream) {
    return route_impl(x_dev, T, H, E, k, topk_ids_dev, topk_w_dev, expert_offsets_dev, ws_dev, ws_bytes, 0, stream);
}

nvfp4_status moe_route_sort_amax_masked(const void* x_dev, int64_t T, int H, int E, int k,
                                        const int32_t* topk_ids_dev, const float* topk_w_dev, int capacity,
                                        int32_t* expert_offsets_dev, void* ws_dev, size_t ws_bytes, void* stream) {
    if (capacity == 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    return route_impl(x_dev, T, H, E, k, topk_ids_dev, topk_w_dev, expert_offsets_dev, ws_dev, ws_bytes, capacity,
                      stream);
}

nvfp4_status moe_workspace_layout_query_masked(int64_t T, int H, int I, int E, int k, int capacity,
                                               moe_workspace_layout* out) {
    if (!out) return NVFP4_ERR_INVALID_ARG;
    if (!moe_shape_ok(T, H, I, E, k) || !capacity_ok(E, capacity)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    compute_layout(T, H, I, E, k, out, capacity);
    return NVFP4_OK;
}

size_t moe_workspace_bytes_masked(int64_t T, int H, int I, int E, int k, int capacity) {
    if (!moe_shape_ok(T, H, I, E, k) || !capacity_ok(E, capacity)) return 0;
    moe_workspace_layout L;
    compute_layout(T, H, I, E, k, &L, capacity);
    return L.total;
}

static nvfp4_status moe_fc1_swiglu_nvfp4_impl(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                                  void* ws_dev, size_t ws_bytes, float* fc1_debug_dev, void* stream, bool pdl, int capacity = 0,
                                  uint16_t* gu_save = nullptr) {
    moe_workspace_layout L;
    const nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L, capacity);
    if (s != NVFP4_OK) return s;
    if (!expert_offsets_dev) return NVFP4_ERR_INVALID_ARG;
    if (T == 0) return NVFP4_OK;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    GemmArgs a = fc1_args(w, expert_offsets_dev, ws_dev, L, fc1_debug_dev, err);
    a.gu_save = gu_save;
    return from_cuda(launch_fc1(a, static_cast<cudaStream_t>(stream), pdl));
}

static nvfp4_status moe_requant_nvfp4_impl(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                               void* ws_dev, size_t ws_bytes, void* stream, bool pdl, int capacity = 0) {
    moe_workspace_layout L;
    const nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L, capacity);
    if (s != NVFP4_OK) return s;
    if (!expert_offsets_dev) return NVFP4_ERR_INVALID_ARG;
    if (T == 0) return NVFP4_OK;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    return from_cuda(launch_requant(at<uint16_t>(ws_dev, L.h), at<uint32_t>(ws_dev, L.amax2),
                                    at<int32_t>(ws_dev, L.row_pair), expert_offsets_dev, w->E, L.rows_cap, w->I,
                                    at<uint8_t>(ws_dev, L.a2_codes), at<uint8_t>(ws_dev, L.a2_sf),
                                    at<float>(ws_dev, L.a2_g), err, static_cast<cudaStream_t>(stream), pdl));
}

static nvfp4_status moe_fc2_nvfp4_impl(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                           void* ws_dev, size_t ws_bytes, float* fc2_debug_dev, void* stream, bool pdl, int capacity = 0) {
    moe_workspace_layout L;
    const nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L, capacity);
    if (s != NVFP4_OK) return s;
    if (!expert_offsets_dev) return NVFP4_ERR_INVALID_ARG;
    if (T == 0) return NVFP4_OK;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    return from_cuda(launch_fc2(fc2_args(w, expert_offsets_dev, ws_dev, L, fc2_debug_dev, err),
                                static_cast<cudaStream_t>(stream), pdl));
}

static nvfp4_status moe_fc2_requant_nvfp4_impl(const moe_nvfp4_weights* w, int64_t T, int k,
                                               const int32_t* expert_offsets_dev, void* ws_dev, size_t ws_bytes,
                                               float* fc2_debug_dev, void* stream, bool pdl, int capacity = 0) {
    moe_workspace_layout L;
    const nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L, capacity);
    if (s != NVFP4_OK) return s;
    if (w->I > fc2_requant_max_i() || w->E > fc2_requant_max_e()) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!expert_offsets_dev) return NVFP4_ERR_INVALID_ARG;
    if (T == 0) return NVFP4_OK;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    GemmArgs a = fc2_args(w, expert_offsets_dev, ws_dev, L, fc2_debug_dev, err);
    a.h = at<uint16_t>(ws_dev, L.h);             // the FC2 input before requantisation, and its maxima
    a.amax2 = at<uint32_t>(ws_dev, L.amax2);
    return from_cuda(launch_fc2_requant(a, static_cast<cudaStream_t>(stream), pdl));
}

static nvfp4_status moe_combine_bf16_impl(const moe_nvfp4_weights* w, int64_t T, int k, void* out_dev, void* ws_dev,
                              size_t ws_bytes, void* stream, bool pdl, int capacity = 0) {
    moe_workspace_layout L;
    const nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L, capacity);
    if (s != NVFP4_OK) return s;
    if (T == 0) return NVFP4_OK;
    if (!out_dev || !aligned(out_dev, 16)) return NVFP4_ERR_INVALID_ARG;
    return from_cuda(launch_combine(at<uint16_t>(ws_dev, L.y), at<int32_t>(ws_dev, L.pair_row), T, k, w->H,
                                    static_cast<uint16_t*>(out_dev),
                                    static_cast<cudaStream_t>(stream), pdl));
}

// FC1, the FC2 input's requantisation, FC2, the combine; every kernel after FC1 starts early
// (programmatic dependent launch) and waits on its predecessor in the device.  The forward runs
// requant and FC2 as two kernels: on GB300 at the measured sizes that is faster than the fused
// moe_fc2_requant_nvfp4 (same bits), whose in-kernel quantisation is issue-bound on the few
// warps the FC2 kernel's registers and shared memory leave for it.
static nvfp4_status forward_stages(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* offs, void* out_dev,
                                   void* ws_dev, size_t ws_bytes, void* stream, int capacity, bool pdl_fc1 = false) {
    nvfp4_status s = moe_fc1_swiglu_nvfp4_impl(w, T, k, offs, ws_dev, ws_bytes, nullptr, stream, pdl_fc1, capacity);
    if (s != NVFP4_OK) return s;
    s = moe_requant_nvfp4_impl(w, T, k, offs, ws_dev, ws_bytes, stream, true, capacity);
    if (s != NVFP4_OK) return s;
    s = moe_fc2_nvfp4_impl(w, T, k, offs, ws_dev, ws_bytes, nullptr, stream, true, capacity);
    if (s != NVFP4_OK) return s;
    return moe_combine_bf16_impl(w, T, k, out_dev, ws_dev, ws_bytes, stream, true, capacity);
}

// The stage entry points: each one's kernel is ordered after all earlier work on the stream.
nvfp4_status moe_fc1_swiglu_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                                  void* ws_dev, size_t ws_bytes, float* fc1_debug_dev, void* stream) {
    return moe_fc1_swiglu_nvfp4_impl(w, T, k, expert_offsets_dev, ws_dev, ws_bytes, fc1_debug_dev, stream, false);
}

nvfp4_status moe_fc1_swiglu_save_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                                       void* ws_dev, size_t ws_bytes, void* gu_save_dev, void* stream) {
    if (!gu_save_dev || !aligned(gu_save_dev, 4)) return NVFP4_ERR_INVALID_ARG;
    return moe_fc1_swiglu_nvfp4_impl(w, T, k, expert_offsets_dev, ws_dev, ws_bytes, nullptr, stream, false, 0,
                                     static_cast<uint16_t*>(gu_save_dev));
}

nvfp4_status moe_requant_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                               void* ws_dev, size_t ws_bytes, void* stream) {
    return moe_requant_nvfp4_impl(w, T, k, expert_offsets_dev, ws_dev, ws_bytes, stream, false);
}

nvfp4_status moe_fc2_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                           void* ws_dev, size_t ws_bytes, float* fc2_debug_dev, void* stream) {
    return moe_fc2_nvfp4_impl(w, T, k, expert_offsets_dev, ws_dev, ws_bytes, fc2_debug_dev, stream, false);
}

nvfp4_status moe_combine_bf16(const moe_nvfp4_weights* w, int64_t T, int k, void* out_dev, void* ws_dev,
                              size_t ws_bytes, void* stream) {
    return moe_combine_bf16_impl(w, T, k, out_dev, ws_dev, ws_bytes, stream, false);
}

nvfp4_status moe_fc2_requant_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                                   void* ws_dev, size_t ws_bytes, float* fc2_debug_dev, void* stream) {
    return moe_fc2_requant_nvfp4_impl(w, T, k, expert_offsets_dev, ws_dev, ws_bytes, fc2_debug_dev, stream, false);
}

int moe_fc2_requant_max_intermediate(void) { return fc2_requant_max_i(); }

nvfp4_status moe_expert_forward_nvfp4(const moe_nvfp4_weights* w, int64_t T, int k, const int32_t* expert_offsets_dev,
                                      void* out_dev, void* ws_dev, size_t ws_bytes, void* stream) {
    moe_workspace_layout L;
    nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L);
    if (s != NVFP4_OK) return s;
    if (T == 0) return NVFP4_OK;
    if (!expert_offsets_dev || !out_dev || !aligned(out_dev, 16)) return NVFP4_ERR_INVALID_ARG;
    return forward_stages(w, T, k, expert_offsets_dev, out_dev, ws_dev, ws_bytes, stream, 0);
}

// Route sort + quantise and the expert forward in one call: every argument of both is checked
// before anything is launched, and FC1 is launched as a programmatic dependent of the route's
// last kernel (its set-up overlaps that kernel's tail; its reads of the routed rows wait for
// the route to complete), which the two separate calls cannot do.
nvfp4_status moe_layer_forward_nvfp4(const moe_nvfp4_weights* w, const void* x_dev, int64_t T, int k,
                                     const int32_t* topk_ids_dev, const float* topk_w_dev,
                                     int32_t* expert_offsets_dev, void* out_dev, void* ws_dev, size_t ws_bytes,
                                     void* stream) {
    moe_workspace_layout L;
    nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L);
    if (s != NVFP4_OK) return s;
    if (T > 0 && (!out_dev || !aligned(out_dev, 16))) return NVFP4_ERR_INVALID_ARG;
    s = route_impl(x_dev, T, w->H, w->E, k, topk_ids_dev, topk_w_dev, expert_offsets_dev, ws_dev, ws_bytes, 0,
                   stream);
    if (s != NVFP4_OK || T == 0) return s;
    return forward_stages(w, T, k, expert_offsets_dev, out_dev, ws_dev, ws_bytes, stream, 0, true);
}

nvfp4_status moe_router_topk(const void* x_dev, int64_t T, int H, const void* w_router_dev, int E, int k,
                             int32_t* topk_ids_dev, float* topk_w_dev, float* logits_dev, void* stream) {
    if (T < 0 || H <= 0 || H % 64 != 0 || H > (1 << 20) || E < 16 || E > 256 || E % 16 != 0 || k < 1 || k > E ||
        k > 32)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return NVFP4_OK;
    if (!x_dev || !w_router_dev || !topk_ids_dev || !topk_w_dev) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x_dev, 16) || !aligned(w_router_dev, 16) || !aligned(topk_ids_dev, 4) || !aligned(topk_w_dev, 4) ||
        (logits_dev && !aligned(logits_dev, 32)))
        return NVFP4_ERR_INVALID_ARG;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    return from_cuda(launch_router_topk(static_cast<const uint16_t*>(x_dev), T, H,
                                        static_cast<const uint16_t*>(w_router_dev), E, k, topk_ids_dev, topk_w_dev,
                                        logits_dev, err, static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_expert_forward_nvfp4_masked(const moe_nvfp4_weights* w, int64_t T, int k, int capacity,
                                             const int32_t* expert_offsets_dev, void* out_dev, void* ws_dev,
                                             size_t ws_bytes, void* stream) {
    if (capacity == 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    moe_workspace_layout L;
    nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L, capacity);
    if (s != NVFP4_OK) return s;
    if (T == 0) return NVFP4_OK;
    if (!expert_offsets_dev || !out_dev || !aligned(out_dev, 16)) return NVFP4_ERR_INVALID_ARG;
    return forward_stages(w, T, k, expert_offsets_dev, out_dev, ws_dev, ws_bytes, stream, capacity);
}

nvfp4_status moe_layer_forward_nvfp4_masked(const moe_nvfp4_weights* w, const void* x_dev, int64_t T, int k,
                                            const int32_t* topk_ids_dev, const float* topk_w_dev, int capacity,
                                            int32_t* expert_offsets_dev, void* out_dev, void* ws_dev,
                                            size_t ws_bytes, void* stream) {
    if (capacity == 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    moe_workspace_layout L;
    nvfp4_status s = check_forward_args(w, T, k, ws_dev, ws_bytes, &L, capacity);
    if (s != NVFP4_OK) return s;
    if (T > 0 && (!out_dev || !aligned(out_dev, 16))) return NVFP4_ERR_INVALID_ARG;
    s = route_impl(x_dev, T, w->H, w->E, k, topk_ids_dev, topk_w_dev, expert_offsets_dev, ws_dev, ws_bytes,
                   capacity, stream);
    if (s != NVFP4_OK || T == 0) return s;
    return forward_stages(w, T, k, expert_offsets_dev, out_dev, ws_dev, ws_bytes, stream, capacity, true);
}

nvfp4_status moe_backward_layout_query(int64_t T, int H, int I, int E, int k, moe_backward_layout* out) {
    if (!out) return NVFP4_ERR_INVALID_ARG;
    if (!moe_shape_ok(T, H, I, E, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    compute_backward_layout(T, H, I, E, k, out);
    return NVFP4_OK;
}

size_t moe_backward_workspace_bytes(int64_t T, int H, int I, int E, int k) {
    if (!moe_shape_ok(T, H, I, E, k)) return 0;
    moe_backward_layout B;
    compute_backward_layout(T, H, I, E, k, &B);
    return B.total;
}

nvfp4_status moe_expert_backward_ste(const moe_bf16_weights_t* w, int64_t T, int k, const void* x_dev,
                                     const void* dout_dev, const int32_t* expert_offsets_dev, const void* fwd_ws_dev,
                                     size_t fwd_ws_bytes, const void* gu_dev, void* dx_dev, float* dw1_dev,
                                     float* dw2_dev, float* dprob_dev, void* bwd_ws_dev, size_t bwd_ws_bytes,
                                     void* stream) {
    if (!w) return NVFP4_ERR_INVALID_ARG;
    if (!moe_shape_ok(T, w->H, w->I, w->E, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!w->w1 || !w->w2 || !dw1_dev || !dw2_dev) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(w->w1, 16) || !aligned(w->w2, 16) || !aligned(dw1_dev, 32) || !aligned(dw2_dev, 32))
        return NVFP4_ERR_INVALID_ARG;
    const int H = w->H, I = w->I, E = w->E;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(dw1_dev, 0, static_cast<size_t>(E) * 2 * I * H * 4, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dw2_dev, 0, static_cast<size_t>(E) * H * I * 4, st);
        return from_cuda(e);
    }
    if (!x_dev || !dout_dev || !expert_offsets_dev || !fwd_ws_dev || !gu_dev || !dx_dev || !dprob_dev ||
        !bwd_ws_dev)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x_dev, 16) || !aligned(dout_dev, 16) || !aligned(expert_offsets_dev, 4) || !aligned(fwd_ws_dev, 256) ||
        !aligned(gu_dev, 16) || !aligned(dx_dev, 16) || !aligned(dprob_dev, 4) || !aligned(bwd_ws_dev, 256))
        return NVFP4_ERR_INVALID_ARG;
    moe_workspace_layout L;
    compute_layout(T, H, I, E, k, &L);
    // the backward's GEMMs address routed rows as int32 tensor-map coordinates
    if (L.rows_cap >= (int64_t(1) << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    moe_backward_layout B;
    compute_backward_layout(T, H, I, E, k, &B);
    if (fwd_ws_bytes < L.total || bwd_ws_bytes < B.total) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    int* err = device_error_ptr();
    if (!err) return NVFP4_ERR_CUDA;
    void* fws = const_cast<void*>(fwd_ws_dev);
    BackwardArgs a{};
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = k;
    a.rows_cap = L.rows_cap;
    a.w1 = static_cast<const uint16_t*>(w->w1);
    a.w2 = static_cast<const uint16_t*>(w->w2);
    a.x = static_cast<const uint16_t*>(x_dev);
    a.dout = static_cast<const uint16_t*>(dout_dev);
    a.offsets = expert_offsets_dev;
    a.row_pair = at<int32_t>(fws, L.row_pair);
    a.row_prob = at<float>(fws, L.row_prob);
    a.h = at<uint16_t>(fws, L.h);
    a.gu = static_cast<const uint16_t*>(gu_dev);
    a.dx = static_cast<uint16_t*>(dx_dev);
    a.dw1 = dw1_dev;
    a.dw2 = dw2_dev;
    a.dprob = dprob_dev;
    a.dy_rows = at<uint16_t>(bwd_ws_dev, B.dy_rows);
    a.dh = at<uint16_t>(bwd_ws_dev, B.dh);
    a.dgu = at<uint16_t>(bwd_ws_dev, B.dgu);
    a.dx_pairs = at<uint16_t>(bwd_ws_dev, B.dx_pairs);
    a.x_rows = at<uint16_t>(bwd_ws_dev, B.x_rows);
    a.real_end = at<int32_t>(bwd_ws_dev, B.real_end);
    a.err = err;
    return from_cuda(launch_moe_backward_ste(a, st));
}

int nvfp4_last_cuda_error(void) { return static_cast<int>(t_last_cuda_error); }

const char* nvfp4_cuda_error_name(int error) { return cudaGetErrorName(static_cast<cudaError_t>(error)); }

nvfp4_status nvfp4_silu_table(float* out_dev, void* stream) {
    if (!out_dev || !aligned(out_dev, 4)) return NVFP4_ERR_INVALID_ARG;
    return from_cuda(copy_silu_table(out_dev, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_get_device_error(void* stream, int* device_status) {
    if (!device_status) return NVFP4_ERR_INVALID_ARG;
    *device_status = NVFP4_OK;
    if (from_cuda(cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != NVFP4_OK) return NVFP4_ERR_CUDA;
    int v = 0;
    if (from_cuda(cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int))) != NVFP4_OK) return NVFP4_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (from_cuda(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int))) != NVFP4_OK) return NVFP4_ERR_CUDA;
    }
    *device_status = v;
    return NVFP4_OK;
}

}  // extern "C"
