"""The C-ABI library loads, exports every symbol include/*.h declares, and its
host-side queries and argument validation behave as documented.  No kernel is
launched here: every call below is rejected (or answered) on the host."""

import ctypes
import glob
import os
import re

import numpy as np
import pytest

import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return M.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b((?:nvfp4|moe)_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"nvfp4_quantize_rows", "moe_route_sort_amax", "moe_expert_forward_nvfp4"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in M.STATUS_NAMES.items():
        assert M.nvfp4_status_string(code) == name
    assert M.nvfp4_status_string(99) == "NVFP4_UNKNOWN_STATUS"


def test_sizes(lib):
    assert M.nvfp4_rows_padded(0) == 0
    assert M.nvfp4_rows_padded(1) == 128
    assert M.nvfp4_rows_padded(128) == 128
    assert M.nvfp4_rows_padded(129) == 256
    assert M.nvfp4_sf_bytes(1, 64) == 128 * 4
    assert M.nvfp4_sf_bytes(300, 2048) == 384 * 128
    assert M.nvfp4_sf_bytes(10, 100) == 0


def test_sf_index_is_a_permutation():
    for rows, cols in ((128, 64), (256, 2048), (384, 768)):
        idx = M.sf_byte_index(rows, cols)
        assert np.array_equal(np.sort(idx.ravel()), np.arange(rows * cols // 16))
        # the first 128-row x 64-column tile is the 32x16-byte block the tensor-core copy takes
        assert idx[0, 0] == 0 and idx[0, 1] == 1 and idx[32, 0] == 4 and idx[1, 0] == 16
        if cols > 64:
            assert idx[0, 4] == 512


def test_workspace_layout(lib):
    L = M.moe_workspace_layout_query(4096, 2048, 768, 128, 8)
    assert L.rows_cap % 128 == 0 and L.rows_cap >= 4096 * 8
    assert L.rows_cap <= 4096 * 8 + 128 * 128
    offs = [L.a_codes, L.a_sf, L.a_g, L.row_pair, L.row_prob, L.amax2, L.pair_row, L.a_sf_rows, L.chunk_count,
            L.chunk_base,
            L.pair_rank, L.expert_count, L.route_end, L.h, L.a2_codes, L.a2_sf, L.a2_g, L.y, L.total]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs)
    assert L.total == M.moe_workspace_bytes(4096, 2048, 768, 128, 8)
    assert L.a_sf - L.a_codes >= L.rows_cap * 1024
    assert L.total - L.y >= L.rows_cap * 2048 * 2
    assert L.chunk_count - L.pair_row >= 4096 * 8 * 4
    # the capacity only counts experts that can be live
    small = M.moe_workspace_layout_query(1, 2048, 768, 128, 8)
    assert small.rows_cap == 1024


@pytest.mark.parametrize("shape", [(0, 2048, 768, 0, 8), (4, 2000, 768, 8, 2), (4, 2048, 100, 8, 2),
                                   (4, 2048, 768, 8, 9), (4, 2048, 768, 2000, 2), (-1, 256, 128, 8, 2)])
def test_unsupported_shapes(lib, shape):
    assert M.moe_workspace_bytes(*shape) == 0
    L = M.moe_workspace_layout()
    assert lib.moe_workspace_layout_query(*shape, ctypes.byref(L)) == 2


def test_quantize_rows_validation(lib):
    p = ctypes.c_void_p(256)
    # bad shapes
    assert lib.nvfp4_quantize_rows(p, 4, 100, 100, p, p, p, None) == 2
    assert lib.nvfp4_quantize_rows(p, 4, 128, 64, p, p, p, None) == 2
    assert lib.nvfp4_quantize_rows(p, 4, 16384, 16384, p, p, p, None) == 2
    # null / misaligned pointers
    assert lib.nvfp4_quantize_rows(None, 4, 128, 128, p, p, p, None) == 1
    assert lib.nvfp4_quantize_rows(ctypes.c_void_p(258), 4, 128, 128, p, p, p, None) == 1
    # codes are written with 32-byte stores: a 16- but not 32-byte aligned buffer is refused
    assert lib.nvfp4_quantize_rows(p, 4, 128, 128, ctypes.c_void_p(272), p, p, None) == 1
    # zero rows is a no-op
    assert lib.nvfp4_quantize_rows(None, 0, 128, 128, None, None, None, None) == 0


def test_router_validation(lib):
    p = ctypes.c_void_p(4096)
    ok = lambda T, H, E, k, x=p, w=p, ids=p, pw=p, lg=None: lib.moe_router_topk(x, T, H, w, E, k, ids, pw, lg, None)
    assert ok(0, 256, 16, 4) == 0                         # nothing to do, nothing launched
    assert ok(8, 250, 16, 4) == 2                         # H % 64
    assert ok(8, 256, 8, 4) == 2 and ok(8, 256, 24, 4) == 2 and ok(8, 256, 272, 4) == 2   # E
    assert ok(8, 256, 16, 0) == 2 and ok(8, 256, 16, 17) == 2 and ok(8, 256, 64, 33) == 2  # k
    assert ok(8, 256, 16, 4, x=None) == 1
    assert ok(8, 256, 16, 4, x=ctypes.c_void_p(4104)) == 1              # 8-byte aligned x
    assert ok(8, 256, 16, 4, lg=ctypes.c_void_p(4112)) == 1             # logits need 32 bytes


def test_masked_layout_validation(lib):
    p = ctypes.c_void_p(4096)
    L = M.moe_workspace_layout()
    assert lib.moe_workspace_layout_query_masked(100, 256, 128, 8, 2, 256, ctypes.byref(L)) == 0
    assert L.rows_cap == 8 * 256                          # E * capacity rows, expert e at e * capacity
    assert lib.moe_workspace_bytes_masked(100, 256, 128, 8, 2, 256) == L.total
    assert lib.moe_workspace_bytes_masked(100, 256, 128, 8, 2, 200) == 0       # not a multiple of 128
    assert lib.moe_workspace_layout_query_masked(100, 256, 128, 8, 2, 0, ctypes.byref(L)) == 2
    assert lib.moe_route_sort_amax_masked(p, 16, 256, 8, 2, p, p, 64, p, p, 1 << 30, None) == 2
    assert lib.moe_route_sort_amax_masked(p, 16, 256, 8, 2, p, p, 128, p, None, 1 << 30, None) == 1
    small = lib.moe_workspace_bytes_masked(16, 256, 128, 8, 2, 128)
    route_end = M.moe_workspace_layout_query_masked(16, 256, 128, 8, 2, 128).route_end
    assert small > route_end
    assert lib.moe_route_sort_amax_masked(p, 16, 256, 8, 2, p, p, 128, p, p, route_end - 1, None) == 3
    assert M.nvfp4_status_string(8) == "NVFP4_ERR_CAPACITY"


def test_route_validation(lib):
    p = ctypes.c_void_p(4096)
    ok_ws = M.moe_workspace_layout_query(16, 256, 128, 8, 2).route_end
    assert lib.moe_route_sort_amax(p, 16, 256, 8, 2, p, p, p, None, ok_ws, None) == 1
    assert lib.moe_route_sort_amax(p, 16, 256, 8, 2, p, p, p, p, ok_ws - 1, None) == 3
    assert lib.moe_route_sort_amax(p, 16, 250, 8, 2, p, p, p, p, ok_ws, None) == 2
    assert lib.moe_route_sort_amax(p, 16, 256, 8, 2, p, p, p, ctypes.c_void_p(4097), ok_ws, None) == 1


def test_forward_validation(lib):
    p = 4096
    w = M.moe_nvfp4_weights(p, p, p, p, p, p, 8, 256, 128)
    need = M.moe_workspace_bytes(16, 256, 128, 8, 2)
    ws = ctypes.c_void_p(4096)
    f = lib.moe_expert_forward_nvfp4
    assert f(None, 16, 2, ws, ws, ws, need, None) == 1
    assert f(ctypes.byref(w), 16, 2, ws, ws, ws, need - 1, None) == 3
    assert f(ctypes.byref(w), 16, 9, ws, ws, ws, need, None) == 2
    bad = M.moe_nvfp4_weights(p, p, 0, p, p, p, 8, 256, 128)
    assert f(ctypes.byref(bad), 16, 2, ws, ws, ws, need, None) == 1
    odd = M.moe_nvfp4_weights(p + 8, p, p, p, p, p, 8, 256, 128)
    assert f(ctypes.byref(odd), 16, 2, ws, ws, ws, need, None) == 1
    # T = 0 is a valid empty call
    need0 = M.moe_workspace_bytes(0, 256, 128, 8, 2)
    assert f(ctypes.byref(w), 0, 2, ws, ws, ws, need0, None) == 0
    for stage in (lib.moe_fc1_swiglu_nvfp4, lib.moe_fc2_nvfp4):
        assert stage(ctypes.byref(w), 16, 2, ws, ws, need - 1, None, None) == 3
    assert lib.moe_requant_nvfp4(ctypes.byref(w), 16, 2, ws, ws, need - 1, None) == 3
    assert lib.moe_combine_bf16(ctypes.byref(w), 16, 2, ws, ws, need - 1, None) == 3
    # the one-call layer checks the forward's and the route sort's arguments before launching
    layer = lib.moe_layer_forward_nvfp4
    assert layer(None, ws, 16, 2, ws, ws, ws, ws, ws, need, None) == 1
    assert layer(ctypes.byref(w), ws, 16, 2, ws, ws, ws, ws, ws, need - 1, None) == 3
    assert layer(ctypes.byref(w), ws, 16, 2, ws, ws, ws, ctypes.c_void_p(4104), ws, need, None) == 1  # out
    assert layer(ctypes.byref(w), ws, 16, 2, None, ws, ws, ws, ws, need, None) == 1                   # ids
    assert layer(ctypes.byref(w), ctypes.c_void_p(4100), 16, 2, ws, ws, ws, ws, ws, need, None) == 1  # x
    assert layer(ctypes.byref(w), ws, 16, 9, ws, ws, ws, ws, ws, need, None) == 2
    lm = lib.moe_layer_forward_nvfp4_masked
    need_m = lib.moe_workspace_bytes_masked(16, 256, 128, 8, 2, 128)
    assert lm(ctypes.byref(w), ws, 16, 2, ws, ws, 0, ws, ws, ws, need_m, None) == 2          # capacity 0
    assert lm(ctypes.byref(w), ws, 16, 2, ws, ws, 100, ws, ws, ws, need_m, None) == 2        # not a multiple of 128
    assert lm(ctypes.byref(w), ws, 16, 2, ws, ws, 128, ws, ws, ws, need_m - 1, None) == 3
    assert lm(ctypes.byref(w), ws, 16, 2, None, ws, 128, ws, ws, ws, need_m, None) == 1      # ids
    save = lib.moe_fc1_swiglu_save_nvfp4
    assert save(ctypes.byref(w), 16, 2, ws, ws, need, None, None) == 1               # no gate/up buffer
    assert save(ctypes.byref(w), 16, 2, ws, ws, need, ctypes.c_void_p(4098), None) == 1   # misaligned
    assert save(ctypes.byref(w), 16, 2, ws, ws, need - 1, ws, None) == 3


def test_backward_layout(lib):
    T, H, I, E, k = 4096, 2048, 768, 128, 8
    B_ = M.moe_backward_layout_query(T, H, I, E, k)
    L = M.moe_workspace_layout_query(T, H, I, E, k)
    assert B_.rows_cap == L.rows_cap
    offs = [B_.dy_rows, B_.dh, B_.dgu, B_.dx_pairs, B_.x_rows, B_.real_end, B_.total]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    rc = L.rows_cap
    sizes = [rc * H * 2, rc * I * 2, rc * 2 * I * 2, T * k * H * 2, rc * H * 2, E * 4]
    assert all(b - a >= n for a, b, n in zip(offs[:-1], offs[1:], sizes))
    assert B_.total == lib.moe_backward_workspace_bytes(T, H, I, E, k)
    assert lib.moe_backward_workspace_bytes(T, 2000, I, E, k) == 0


def test_backward_validation(lib):
    p = 4096
    w = M.moe_bf16_weights_t(p, p, 8, 256, 128)
    fwd = M.moe_workspace_bytes(16, 256, 128, 8, 2)
    bwd = lib.moe_backward_workspace_bytes(16, 256, 128, 8, 2)
    q = ctypes.c_void_p(p)
    f = lambda w_=ctypes.byref(w), T=16, k=2, dw=q, fws=fwd, bws=bwd, x=q: lib.moe_expert_backward_ste(  # noqa: E731
        w_, T, k, x, q, q, q, fws, q, q, dw, dw, q, q, bws, None)
    assert f(w_=None) == 1
    assert f(k=9) == 2
    assert f(fws=fwd - 1) == 3 and f(bws=bwd - 1) == 3
    assert f(dw=ctypes.c_void_p(p + 16)) == 1               # weight gradients are stored 32 bytes at a time
    assert f(x=None) == 1
    assert f(x=ctypes.c_void_p(p + 8)) == 1
    assert lib.moe_expert_backward_ste(ctypes.byref(M.moe_bf16_weights_t(0, p, 8, 256, 128)), 16, 2, q, q, q, q,
                                       fwd, q, q, q, q, q, q, bwd, None) == 1
    # T*k just under 2^30 passes the shape check, but its rows_cap reaches 2^30
    big_T = (1 << 30) // 2 - 1
    assert lib.moe_expert_backward_ste(ctypes.byref(w), big_T, 2, q, q, q, q, 1 << 62, q, q, q, q, q, q, 1 << 62,
                                       None) == 2
    assert lib.moe_expert_backward_ste(ctypes.byref(M.moe_bf16_weights_t(p, p + 8, 8, 256, 128)), 16, 2, q, q, q,
                                       q, fwd, q, q, q, q, q, q, bwd, None) == 1     # weights 16-byte aligned


def test_device_error_requires_pointer(lib):
    assert lib.nvfp4_get_device_error(None, None) == 1


def test_product_path_has_no_oracle_import():
    # the binding and the CUDA sources never reach into the oracle
    for path in glob.glob(os.path.join(ROOT, "nvfp4_moe_expert_gb300", "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            src = open(path).read()
            assert "oracle" not in src.replace("the oracle", ""), path


def test_backward_binding_checks_tensors(lib):
    import torch
    E, H, I, T, k = 4, 256, 128, 8, 2
    wt = type("W", (), {"E": E, "H": H, "I": I})()
    bf, f32 = torch.bfloat16, torch.float32
    ok = dict(x=torch.zeros(T, H, dtype=bf), dout=torch.zeros(T, H, dtype=bf),
              offs=torch.zeros(E + 1, dtype=torch.int32), ws=torch.zeros(16, dtype=torch.uint8),
              gu=torch.zeros(M.moe_workspace_layout_query(T, H, I, E, k).rows_cap, 2 * I, dtype=bf),
              dx=torch.zeros(T, H, dtype=bf),
              dw1=torch.zeros(E, 2 * I, H), dw2=torch.zeros(E, H, I), dprob=torch.zeros(T, k))

    def call(**kw):
        a = dict(ok, **kw)
        M.moe_expert_backward_ste(wt, T, k, a["x"], a["dout"], a["offs"], a["ws"], a["gu"], a["dx"], a["dw1"],
                                  a["dw2"], a["dprob"], a["ws"])
    with pytest.raises(ValueError, match="float32"):
        call(dw1=torch.zeros(E, 2 * I, H, dtype=bf))
    with pytest.raises(ValueError, match=r"\(8, 2\)"):
        call(dprob=torch.zeros(T, k + 1))
    with pytest.raises(ValueError, match="gu must be"):
        call(gu=torch.zeros(256, 2 * I, dtype=f32))                    # the FP32 values: refused
    with pytest.raises(ValueError, match="gu must be"):
        call(gu=torch.zeros(4, 2 * I, dtype=bf))                       # fewer rows than rows_cap
    with pytest.raises(ValueError, match="CUDA"):      # right shapes, but host tensors: refused before any call
        call()


def test_layer_weight_versions():
    # host logic of MoELayer's weight-version checks, with the quantisation stubbed out
    import torch
    layer = M.MoELayer.__new__(M.MoELayer)
    calls = []

    def fake_quantize(stream=None):
        calls.append(1)
        layer._wt = None
        layer._wver = layer._weight_version()
        layer._gen += 1

    layer._quantize = fake_quantize
    layer._gen = 0
    layer._w_bf16 = (torch.zeros(2, 4), torch.zeros(2, 4))
    layer._quantize()
    layer._refresh_if_changed()
    assert len(calls) == 1                           # unchanged weights: nothing to do
    layer._w_bf16[0].add_(1.0)                       # an optimizer step updates a weight in place
    layer._refresh_if_changed()
    assert len(calls) == 2 and layer._wver == layer._weight_version()
    layer._w_bf16[1].data = torch.ones(2, 4)         # storage swapped: seen through the data pointer
    layer._refresh_if_changed()
    assert len(calls) == 3
    # a write through .data bypasses the version counter: not seen until refresh_weights()
    layer._w_bf16[0].data.add_(1.0)
    layer._refresh_if_changed()
    assert len(calls) == 3
    layer._saved = (None, None, None, None, 0, 1, (layer._wver, layer._gen))
    layer.refresh_weights()
    assert len(calls) == 4
    with pytest.raises(RuntimeError, match="weights changed"):   # refreshed after its forward
        layer.backward(None)
    # a backward whose forward saw an older version refuses to run
    layer._saved = (None, None, None, None, 0, 1, (layer._wver, layer._gen))
    layer._w_bf16[1].mul_(2.0)
    with pytest.raises(RuntimeError, match="weights changed"):
        layer.backward(None)
