"""Python binding of libnvfp4moe.so, the GB300 (sm_103a) NVFP4 W4A4 MoE expert forward.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels; PyTorch provides device memory and the current stream.  The
entry points have the names of the C ABI in ``include/nvfp4_moe.h``:

    nvfp4_quantize_rows, moe_route_sort_amax, moe_expert_forward_nvfp4, moe_layer_forward_nvfp4,
    moe_fc1_swiglu_nvfp4, moe_fc1_swiglu_save_nvfp4, moe_requant_nvfp4, moe_fc2_nvfp4, moe_fc2_requant_nvfp4, moe_combine_bf16,
    moe_workspace_bytes, moe_workspace_layout_query, nvfp4_sf_bytes,
    nvfp4_rows_padded, nvfp4_get_device_error, nvfp4_status_string, nvfp4_silu_table,
    moe_router_topk, the fixed-capacity moe_*_masked calls, and the
    straight-through backward: moe_backward_layout_query,
    moe_backward_workspace_bytes, moe_expert_backward_ste

There is no CPU fallback: if the library is missing or a call fails, an
exception is raised.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4moe.so")

NVFP4_OK = 0
STATUS_NAMES = {
    0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED_SHAPE",
    3: "NVFP4_ERR_WORKSPACE_TOO_SMALL", 4: "NVFP4_ERR_CUDA", 5: "NVFP4_ERR_BAD_EXPERT_ID",
    6: "NVFP4_ERR_NONFINITE", 7: "NVFP4_ERR_DEVICE_TIMEOUT", 8: "NVFP4_ERR_CAPACITY",
}


class NVFP4Error(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}{detail}")


class moe_nvfp4_weights(ctypes.Structure):
    _fields_ = [
        ("w1_codes", ctypes.c_void_p), ("w1_sf", ctypes.c_void_p), ("w1_g", ctypes.c_void_p),
        ("w2_codes", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p), ("w2_g", ctypes.c_void_p),
        ("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
    ]


class moe_workspace_layout(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
        ("E", ctypes.c_int32), ("k", ctypes.c_int32),
        ("rows_cap", ctypes.c_int64), ("n_chunks", ctypes.c_int64),
    ] + [(n, ctypes.c_size_t) for n in (
        "a_codes", "a_sf", "a_g", "row_pair", "row_prob", "amax2", "pair_row", "a_sf_rows", "chunk_count", "chunk_base",
        "pair_rank", "expert_count", "route_end", "h", "a2_codes", "a2_sf", "a2_g", "y", "total")]


class moe_bf16_weights_t(ctypes.Structure):
    _fields_ = [("w1", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32)]


class moe_backward_layout(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
        ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("rows_cap", ctypes.c_int64),
    ] + [(n, ctypes.c_size_t) for n in (
        "dy_rows", "dh", "dgu", "dx_pairs", "x_rows", "real_end", "total")]


_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "nvfp4_status_string": (ctypes.c_char_p, [_I32]),
    "nvfp4_rows_padded": (_I64, [_I64]),
    "nvfp4_sf_bytes": (_SZ, [_I64, _I64]),
    "nvfp4_quantize_rows": (_I32, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
    "moe_workspace_layout_query": (_I32, [_I64, _I32, _I32, _I32, _I32, ctypes.POINTER(moe_workspace_layout)]),
    "moe_workspace_bytes": (_SZ, [_I64, _I32, _I32, _I32, _I32]),
    "moe_route_sort_amax": (_I32, [_P, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_forward_nvfp4": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _P, _P, _P, _SZ, _P]),
    "moe_fc1_swiglu_nvfp4": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _P, _P, _SZ, _P, _P]),
    "moe_fc1_swiglu_save_nvfp4": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _P, _P, _SZ, _P, _P]),
    "moe_layer_forward_nvfp4": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _P, _I64, _I32, _P, _P, _P, _P, _P, _SZ,
                                       _P]),
    "moe_layer_forward_nvfp4_masked": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _P, _I64, _I32, _P, _P, _I32, _P,
                                              _P, _P, _SZ, _P]),
    "moe_requant_nvfp4": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _P, _P, _SZ, _P]),
    "moe_fc2_nvfp4": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _P, _P, _SZ, _P, _P]),
    "moe_combine_bf16": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _P, _P, _SZ, _P]),
    "moe_fc2_requant_nvfp4": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _P, _P, _SZ, _P, _P]),
    "moe_fc2_requant_max_intermediate": (_I32, []),
    "nvfp4_get_device_error": (_I32, [_P, ctypes.POINTER(ctypes.c_int)]),
    "nvfp4_silu_table": (_I32, [_P, _P]),
    "nvfp4_last_cuda_error": (_I32, []),
    "nvfp4_cuda_error_name": (ctypes.c_char_p, [_I32]),
    "moe_route_sort_amax_noalloc": (_I32, [_P, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_router_topk": (_I32, [_P, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P]),
    "moe_workspace_layout_query_masked": (_I32, [_I64, _I32, _I32, _I32, _I32, _I32,
                                                 ctypes.POINTER(moe_workspace_layout)]),
    "moe_workspace_bytes_masked": (_SZ, [_I64, _I32, _I32, _I32, _I32, _I32]),
    "moe_route_sort_amax_masked": (_I32, [_P, _I64, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _SZ, _P]),
    "moe_expert_forward_nvfp4_masked": (_I32, [ctypes.POINTER(moe_nvfp4_weights), _I64, _I32, _I32, _P, _P, _P,
                                               _SZ, _P]),
    "moe_backward_layout_query": (_I32, [_I64, _I32, _I32, _I32, _I32, ctypes.POINTER(moe_backward_layout)]),
    "moe_backward_workspace_bytes": (_SZ, [_I64, _I32, _I32, _I32, _I32]),
    "moe_expert_backward_ste": (_I32, [ctypes.POINTER(moe_bf16_weights_t), _I64, _I32, _P, _P, _P, _P, _SZ, _P,
                                       _P, _P, _P, _P, _P, _SZ, _P]),
}

_lib = None


def lib():
    """The loaded library (loaded on first use; raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m nvfp4_moe_expert_gb300.build` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(fn, status):
    if status != NVFP4_OK:
        detail = ""
        if status == 4 and _lib is not None:          # NVFP4_ERR_CUDA: name the CUDA error behind it
            code = _lib.nvfp4_last_cuda_error()
            detail = f" ({_lib.nvfp4_cuda_error_name(code).decode()}, {code})"
        raise NVFP4Error(fn, status, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# ---------------------------------------------------------------- host queries
def nvfp4_status_string(status):
    return lib().nvfp4_status_string(status).decode()


def nvfp4_rows_padded(rows):
    return lib().nvfp4_rows_padded(rows)


def nvfp4_sf_bytes(rows, cols):
    return lib().nvfp4_sf_bytes(rows, cols)


def moe_workspace_bytes(T, H, I, E, k):
    return lib().moe_workspace_bytes(T, H, I, E, k)


def moe_workspace_layout_query(T, H, I, E, k):
    L = moe_workspace_layout()
    _check("moe_workspace_layout_query", lib().moe_workspace_layout_query(T, H, I, E, k, ctypes.byref(L)))
    return L


# ---------------------------------------------------------------- quantiser
def nvfp4_quantize_rows(x, codes=None, sf=None, g=None, stream=None):
    """NVFP4-quantise each row of a BF16 CUDA matrix [rows, cols]; returns (codes, sf, g)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    if not x.is_cuda or (x.shape[0] > 0 and x.stride(1) != 1):
        raise ValueError("x must be a CUDA tensor with contiguous rows")
    rows, cols = x.shape
    rp = nvfp4_rows_padded(rows)
    dev = x.device
    if codes is None:
        codes = torch.empty((rp, cols // 2), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty(max(nvfp4_sf_bytes(rows, cols), 1), dtype=torch.uint8, device=dev)
    if g is None:
        g = torch.empty(rows, dtype=torch.float32, device=dev)
    _check("nvfp4_quantize_rows", lib().nvfp4_quantize_rows(
        _ptr(x), rows, cols, x.stride(0), _ptr(codes), _ptr(sf), _ptr(g), _stream(stream)))
    return codes, sf, g


def nvfp4_silu_table(out=None, stream=None):
    """The SiLU the FC1 epilogue applies, evaluated by its own code for every BF16 input:
    float32 [65536] on the current device, entry i = silu of the BF16 value with bit pattern
    i, rounded once to FP32."""
    if out is None:
        out = torch.empty(65536, dtype=torch.float32, device="cuda")
    _need_cuda(out)
    if out.dtype != torch.float32 or out.numel() != 65536:
        raise ValueError("out must be a float32 tensor of 65536 elements")
    _check("nvfp4_silu_table", lib().nvfp4_silu_table(_ptr(out), _stream(stream)))
    return out


def nvfp4_get_device_error(stream=None):
    st = ctypes.c_int(0)
    _check("nvfp4_get_device_error", lib().nvfp4_get_device_error(_stream(stream), ctypes.byref(st)))
    return st.value


# ---------------------------------------------------------------- MoE
class MoEWeights:
    """Quantised expert weights (device tensors) and the C struct pointing at them."""

    def __init__(self, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, E, H, I):
        self.tensors = (w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g)
        self.E, self.H, self.I = E, H, I
        self.struct = moe_nvfp4_weights(*[t.data_ptr() for t in self.tensors], E, H, I)

    def ref(self):
        return ctypes.byref(self.struct)


def quantize_moe_weights(w1, w2, stream=None):
    """w1 bf16 [E, 2I, H] (gate rows then up rows), w2 bf16 [E, H, I] -> MoEWeights."""
    E, two_i, H = w1.shape
    I = two_i // 2
    if tuple(w2.shape) != (E, H, I):
        raise ValueError("w2 must be [E, H, I]")
    c1, s1, g1 = nvfp4_quantize_rows(w1.reshape(E * two_i, H), stream=stream)
    c2, s2, g2 = nvfp4_quantize_rows(w2.reshape(E * H, I), stream=stream)
    return MoEWeights(c1, s1, g1, c2, s2, g2, E, H, I)


def alloc_workspace(T, H, I, E, k, device="cuda"):
    n = moe_workspace_bytes(T, H, I, E, k)
    if n == 0:
        raise NVFP4Error("moe_workspace_bytes", 2)
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_route_sort_amax(x, topk_ids, topk_w, E, expert_offsets, ws, stream=None):
    """Route sort + per-token amax + pad + NVFP4 quantise of x [T, H] into ws."""
    _need_cuda(x, topk_ids, topk_w, expert_offsets, ws)
    if x.dtype != torch.bfloat16 or topk_ids.dtype != torch.int32 or topk_w.dtype != torch.float32:
        raise ValueError("x bf16, topk_ids int32, topk_w float32 expected")
    T, H = x.shape
    k = topk_ids.shape[1]
    _check("moe_route_sort_amax", lib().moe_route_sort_amax(
        _ptr(x), T, H, E, k, _ptr(topk_ids), _ptr(topk_w), _ptr(expert_offsets), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_route_sort_amax_noalloc(x, topk_ids, topk_w, E, expert_offsets, out, stream=None):
    """moe_route_sort_amax with its scratch inside the library: `out` only has to hold
    the routed-row outputs (the first layout.chunk_count bytes of a workspace)."""
    _need_cuda(x, topk_ids, topk_w, expert_offsets, out)
    T, H = x.shape
    k = topk_ids.shape[1]
    _check("moe_route_sort_amax_noalloc", lib().moe_route_sort_amax_noalloc(
        _ptr(x), T, H, E, k, _ptr(topk_ids), _ptr(topk_w), _ptr(expert_offsets), _ptr(out),
        out.numel(), _stream(stream)))


def moe_router_topk(x, w_router, k, with_logits=False, stream=None):
    """Router step: (topk_ids int32 [T, k], topk_w float32 [T, k], logits float32 [T, E] or None)
    of BF16 activations x [T, H] and BF16 router weights w_router [E, H]."""
    _need_cuda(x, w_router)
    if x.dtype != torch.bfloat16 or w_router.dtype != torch.bfloat16:
        raise ValueError("x and w_router must be bf16")
    T, H = x.shape
    E = w_router.shape[0]
    ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device) if with_logits else None
    _check("moe_router_topk", lib().moe_router_topk(
        _ptr(x), T, H, _ptr(w_router), E, k, _ptr(ids), _ptr(w),
        _ptr(logits) if logits is not None else None, _stream(stream)))
    return ids, w, logits


def moe_workspace_layout_query_masked(T, H, I, E, k, capacity):
    L = moe_workspace_layout()
    _check("moe_workspace_layout_query_masked",
           lib().moe_workspace_layout_query_masked(T, H, I, E, k, capacity, ctypes.byref(L)))
    return L


def alloc_workspace_masked(T, H, I, E, k, capacity, device="cuda"):
    n = lib().moe_workspace_bytes_masked(T, H, I, E, k, capacity)
    if n == 0:
        raise NVFP4Error("moe_workspace_bytes_masked", 2)
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_route_sort_amax_masked(x, topk_ids, topk_w, E, capacity, expert_offsets, ws, stream=None):
    """Route sort into the fixed-capacity layout (expert e at rows [e*capacity, ...))."""
    _need_cuda(x, topk_ids, topk_w, expert_offsets, ws)
    T, H = x.shape
    k = topk_ids.shape[1]
    _check("moe_route_sort_amax_masked", lib().moe_route_sort_amax_masked(
        _ptr(x), T, H, E, k, _ptr(topk_ids), _ptr(topk_w), capacity, _ptr(expert_offsets), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_expert_forward_nvfp4_masked(weights, T, k, capacity, expert_offsets, out, ws, stream=None):
    _need_cuda(expert_offsets, out, ws)
    _check("moe_expert_forward_nvfp4_masked", lib().moe_expert_forward_nvfp4_masked(
        weights.ref(), T, k, capacity, _ptr(expert_offsets), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_expert_forward_nvfp4(weights, T, k, expert_offsets, out, ws, stream=None):
    _need_cuda(expert_offsets, out, ws)
    _check("moe_expert_forward_nvfp4", lib().moe_expert_forward_nvfp4(
        weights.ref(), T, k, _ptr(expert_offsets), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_forward_nvfp4(weights, x, topk_ids, topk_w, expert_offsets, out, ws, stream=None):
    """moe_route_sort_amax + moe_expert_forward_nvfp4 in one call (FC1 chained to the route
    sort by programmatic launch); the same results bit for bit."""
    _need_cuda(x, topk_ids, topk_w, expert_offsets, out, ws)
    if x.dtype != torch.bfloat16 or topk_ids.dtype != torch.int32 or topk_w.dtype != torch.float32:
        raise ValueError("x bf16, topk_ids int32, topk_w float32 expected")
    T, H = x.shape
    if H != weights.H or out.dtype != torch.bfloat16 or tuple(out.shape) != (T, H):
        raise ValueError(f"x and out must be bfloat16 [T, {weights.H}]")
    _check("moe_layer_forward_nvfp4", lib().moe_layer_forward_nvfp4(
        weights.ref(), _ptr(x), T, topk_ids.shape[1], _ptr(topk_ids), _ptr(topk_w), _ptr(expert_offsets),
        _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_forward_nvfp4_masked(weights, x, topk_ids, topk_w, capacity, expert_offsets, out, ws, stream=None):
    """moe_route_sort_amax_masked + moe_expert_forward_nvfp4_masked in one call."""
    _need_cuda(x, topk_ids, topk_w, expert_offsets, out, ws)
    if x.dtype != torch.bfloat16 or topk_ids.dtype != torch.int32 or topk_w.dtype != torch.float32:
        raise ValueError("x bf16, topk_ids int32, topk_w float32 expected")
    T, H = x.shape
    if H != weights.H or out.dtype != torch.bfloat16 or tuple(out.shape) != (T, H):
        raise ValueError(f"x and out must be bfloat16 [T, {weights.H}]")
    _check("moe_layer_forward_nvfp4_masked", lib().moe_layer_forward_nvfp4_masked(
        weights.ref(), _ptr(x), T, topk_ids.shape[1], _ptr(topk_ids), _ptr(topk_w), capacity,
        _ptr(expert_offsets), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_fc1_swiglu_nvfp4(weights, T, k, expert_offsets, ws, debug=None, stream=None):
    _need_cuda(expert_offsets, ws, debug)
    _check("moe_fc1_swiglu_nvfp4", lib().moe_fc1_swiglu_nvfp4(
        weights.ref(), T, k, _ptr(expert_offsets), _ptr(ws), ws.numel(), _ptr(debug), _stream(stream)))


def moe_fc1_swiglu_save_nvfp4(weights, T, k, expert_offsets, ws, gu_save, stream=None):
    """FC1 + SwiGLU x prob that also saves the BF16 gate/up [rows_cap, 2I] for the backward."""
    if gu_save.dtype != torch.bfloat16 or gu_save.dim() != 2 or gu_save.shape[1] != 2 * weights.I:
        raise ValueError("gu_save must be a bfloat16 [rows_cap, 2I] tensor")
    _need_cuda(expert_offsets, ws, gu_save)
    _check("moe_fc1_swiglu_save_nvfp4", lib().moe_fc1_swiglu_save_nvfp4(
        weights.ref(), T, k, _ptr(expert_offsets), _ptr(ws), ws.numel(), _ptr(gu_save), _stream(stream)))


def moe_requant_nvfp4(weights, T, k, expert_offsets, ws, stream=None):
    _need_cuda(expert_offsets, ws)
    _check("moe_requant_nvfp4", lib().moe_requant_nvfp4(
        weights.ref(), T, k, _ptr(expert_offsets), _ptr(ws), ws.numel(), _stream(stream)))


def moe_fc2_nvfp4(weights, T, k, expert_offsets, ws, debug=None, stream=None):
    _need_cuda(expert_offsets, ws, debug)
    _check("moe_fc2_nvfp4", lib().moe_fc2_nvfp4(
        weights.ref(), T, k, _ptr(expert_offsets), _ptr(ws), ws.numel(), _ptr(debug), _stream(stream)))


def moe_fc2_requant_nvfp4(weights, T, k, expert_offsets, ws, debug=None, stream=None):
    """Requantisation of h fused into FC2 (one kernel; y bitwise that of the two stages)."""
    _need_cuda(expert_offsets, ws, debug)
    _check("moe_fc2_requant_nvfp4", lib().moe_fc2_requant_nvfp4(
        weights.ref(), T, k, _ptr(expert_offsets), _ptr(ws), ws.numel(), _ptr(debug), _stream(stream)))


def moe_fc2_requant_max_intermediate():
    return lib().moe_fc2_requant_max_intermediate()


def moe_combine_bf16(weights, T, k, out, ws, stream=None):
    _need_cuda(out, ws)
    _check("moe_combine_bf16", lib().moe_combine_bf16(
        weights.ref(), T, k, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


# ---------------------------------------------------------------- straight-through backward
class MoEWeightsBF16:
    """The BF16 original expert weights for the backward (w1 [E, 2I, H], w2 [E, H, I], as
    given to quantize_moe_weights; the backward's GEMMs read them in place) and the C struct
    pointing at them."""

    def __init__(self, w1, w2):
        if w1.dtype != torch.bfloat16 or w2.dtype != torch.bfloat16 or w1.dim() != 3 or w2.dim() != 3:
            raise ValueError("w1, w2 must be 3-D bfloat16 tensors")
        self.E, two_i, self.H = w1.shape
        self.I = two_i // 2
        if tuple(w2.shape) != (self.E, self.H, self.I):
            raise ValueError(f"w2 must be [E, H, I] = {(self.E, self.H, self.I)}, got {tuple(w2.shape)}")
        self.w1 = w1.contiguous()
        self.w2 = w2.contiguous()
        _need_cuda(self.w1, self.w2)
        self.struct = moe_bf16_weights_t(self.w1.data_ptr(), self.w2.data_ptr(), self.E, self.H, self.I)

    def ref(self):
        return ctypes.byref(self.struct)


def moe_backward_layout_query(T, H, I, E, k):
    L = moe_backward_layout()
    _check("moe_backward_layout_query", lib().moe_backward_layout_query(T, H, I, E, k, ctypes.byref(L)))
    return L


def alloc_backward_workspace(T, H, I, E, k, device="cuda"):
    n = lib().moe_backward_workspace_bytes(T, H, I, E, k)
    if n == 0:
        raise NVFP4Error("moe_backward_workspace_bytes", 2)
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_expert_backward_ste(wt, T, k, x, dout, expert_offsets, ws, gu, dx, dw1, dw2, dprob, bws,
                            stream=None):
    """STE gradients (dx, dw1, dw2, dprob written in place) of the forward whose route
    sort filled `ws` / `expert_offsets` and whose FC1 stage (moe_fc1_swiglu_save_nvfp4)
    saved the BF16 gate/up `gu` [rows_cap, 2I]."""
    E, H, I = wt.E, wt.H, wt.I
    want = ((x, torch.bfloat16, (T, H)), (dout, torch.bfloat16, (T, H)), (dx, torch.bfloat16, (T, H)),
            (dw1, torch.float32, (E, 2 * I, H)), (dw2, torch.float32, (E, H, I)), (dprob, torch.float32, (T, k)),
            (expert_offsets, torch.int32, (E + 1,)))
    for t, dt, shape in want:
        if T > 0 or t is dw1 or t is dw2:
            if t.dtype != dt or tuple(t.shape) != shape:
                raise ValueError(f"expected {dt} {shape}, got {t.dtype} {tuple(t.shape)}")
    if T > 0:
        rows_cap = moe_workspace_layout_query(T, H, I, E, k).rows_cap
        if gu.dtype != torch.bfloat16 or tuple(gu.shape) != (rows_cap, 2 * I):
            raise ValueError(f"gu must be the bfloat16 [{rows_cap}, {2 * I}] gate/up FC1 saved")
    _need_cuda(x, dout, expert_offsets, ws, gu, dx, dw1, dw2, dprob, bws)
    _check("moe_expert_backward_ste", lib().moe_expert_backward_ste(
        wt.ref(), T, k, _ptr(x), _ptr(dout), _ptr(expert_offsets), _ptr(ws), ws.numel(), _ptr(gu),
        _ptr(dx), _ptr(dw1), _ptr(dw2), _ptr(dprob), _ptr(bws), bws.numel(), _stream(stream)))


class MoELayer:
    """Convenience wrapper: owns quantised weights and a workspace sized per call.

    ``forward(..., save_for_backward=True)`` runs the forward stage by stage and keeps
    what the straight-through backward reads (the route, h, FC1's FP32 values);
    ``backward(dout)`` then returns (dx, dw1, dw2, dprob).

    The BF16 weights are the master copy and the layer keeps their NVFP4 quantisation in
    step with them ("Finishing RL training faster: bitwise consistency, high performance,
    agent-driven", section 3.1: the inference kernels define the forward values and the
    backward must belong to the same weights):

    * a forward re-quantises the weights when they were changed through an in-place op on
      the tensors themselves (``w.add_(...)``, ``w.copy_(...)``: torch's version counter) or
      when a tensor's storage was swapped (``w.data = ...``: its data pointer);
    * a write that bypasses the version counter, such as ``w.data.add_(...)`` in a
      hand-written optimizer step, is not seen: call ``refresh_weights()`` after it;
    * ``backward`` raises if the weights were changed or refreshed after the forward it
      belongs to, so one forward/backward pair never mixes two weight versions."""

    def __init__(self, w1, w2, stream=None):
        self._w_bf16 = (w1, w2)
        self._saved = None
        self._ws = {}
        self._gen = 0
        self._quantize(stream)

    def _weight_version(self):
        return tuple((t._version, t.data_ptr()) for t in self._w_bf16)

    def _quantize(self, stream=None):
        self.weights = quantize_moe_weights(*self._w_bf16, stream=stream)
        self.E, self.H, self.I = self.weights.E, self.weights.H, self.weights.I
        self._wver = self._weight_version()
        self._gen += 1

    def _refresh_if_changed(self, stream=None):
        if self._weight_version() != self._wver:
            self._quantize(stream)

    def refresh_weights(self, stream=None):
        """Quantise the BF16 weights again (after a write the version counter cannot see)."""
        self._quantize(stream)

    def workspace(self, T, k, device):
        key = (T, k)
        if key not in self._ws:
            self._ws.clear()
            self._ws[key] = alloc_workspace(T, self.H, self.I, self.E, k, device)
        return self._ws[key]

    def forward(self, x, topk_ids, topk_w, out=None, stream=None, save_for_backward=False):
        self._refresh_if_changed(stream)
        T, H = x.shape
        k = topk_ids.shape[1]
        ws = self.workspace(T, k, x.device)
        offs = torch.empty(self.E + 1, dtype=torch.int32, device=x.device)
        if out is None:
            out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
        if not save_for_backward:
            self._saved = None
            moe_layer_forward_nvfp4(self.weights, x, topk_ids, topk_w, offs, out, ws, stream=stream)
            return out
        moe_route_sort_amax(x, topk_ids, topk_w, self.E, offs, ws, stream=stream)
        L = moe_workspace_layout_query(T, self.H, self.I, self.E, k)
        gu = torch.empty((L.rows_cap, 2 * self.I), dtype=torch.bfloat16, device=x.device)
        moe_fc1_swiglu_save_nvfp4(self.weights, T, k, offs, ws, gu, stream=stream)
        moe_requant_nvfp4(self.weights, T, k, offs, ws, stream=stream)
        moe_fc2_nvfp4(self.weights, T, k, offs, ws, stream=stream)
        moe_combine_bf16(self.weights, T, k, out, ws, stream=stream)
        self._saved = (x, offs, ws, gu, T, k, (self._wver, self._gen))
        return out

    def backward(self, dout, stream=None):
        """(dx bf16 [T, H], dw1 f32 [E, 2I, H], dw2 f32 [E, H, I], dprob f32 [T, k]) of the
        last forward run with save_for_backward=True."""
        if self._saved is None:
            raise RuntimeError("backward needs a forward with save_for_backward=True")
        x, offs, ws, gu, T, k, (wver, gen) = self._saved
        if self._weight_version() != wver or self._gen != gen:
            raise RuntimeError("the weights changed after the forward this backward belongs to")
        wt = MoEWeightsBF16(*self._w_bf16)
        dev = x.device
        dx = torch.empty((T, self.H), dtype=torch.bfloat16, device=dev)
        dw1 = torch.empty((self.E, 2 * self.I, self.H), dtype=torch.float32, device=dev)
        dw2 = torch.empty((self.E, self.H, self.I), dtype=torch.float32, device=dev)
        dprob = torch.empty((T, k), dtype=torch.float32, device=dev)
        bws = alloc_backward_workspace(T, self.H, self.I, self.E, k, dev)
        moe_expert_backward_ste(wt, T, k, x, dout, offs, ws, gu, dx, dw1, dw2, dprob, bws,
                                stream=stream)
        return dx, dw1, dw2, dprob


# ---------------------------------------------------------------- layout helpers
def sf_byte_index(rows, cols):
    """numpy int64 [rows, cols/16]: byte offset of each block scale in the library's
    scale-factor layout (512-byte tiles of 128 rows x 64 columns)."""
    import numpy as np
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(cols // 16, dtype=np.int64)[None, :]
    return ((r >> 7) * (cols >> 6) + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)


def sf_to_rows(sf, rows, cols):
    """Library scale-factor bytes (numpy uint8) -> plain [rows, cols/16] E4M3 codes."""
    return sf[sf_byte_index(rows, cols)]


def sf_from_rows(scales, cols, rows_pad=None):
    """Plain [rows, cols/16] E4M3 codes -> library scale-factor bytes (numpy uint8)."""
    import numpy as np
    rows = scales.shape[0]
    rows_pad = nvfp4_rows_padded(rows) if rows_pad is None else rows_pad
    out = np.zeros(rows_pad * cols // 16, dtype=np.uint8)
    out[sf_byte_index(rows, cols)] = scales
    return out
