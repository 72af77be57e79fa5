"""The fixed-capacity ("masked") layout against the contiguous one, on the GPU.

Expert e owns rows [e*C, (e+1)*C).  Every routed row must carry the same codes, block scales
and outer scale as in the contiguous layout, and the layer output must be bitwise the same
(page "Finishing RL training faster: bitwise consistency, high performance, agent-driven",
section 4.4: the masked and contiguous layouts give bitwise-identical rows).  An expert that
gets more pairs than C is reported as NVFP4_ERR_CAPACITY, without writes past its rows.
"""

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from _helpers import bf16_to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def layer_inputs(cfg):
    L = S.make_layer(cfg)
    dev = torch.device("cuda")
    w = M.quantize_moe_weights(bf16_to_torch(L["w1"]), bf16_to_torch(L["w2"]))
    x = bf16_to_torch(L["x"])
    ids = torch.from_numpy(L["topk_ids"]).to(dev)
    pw = torch.from_numpy(L["topk_w"]).to(dev)
    return L, w, x, ids, pw


def bytes_of(ws, off, n):
    return ws[off:off + n].cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", 64), ("qwen3_30b_a3b", 1024)])
def test_masked_equals_contiguous(name, T):
    cfg = S.shrink(S.CONFIGS[name], T=T)
    L, w, x, ids, pw = layer_inputs(cfg)
    counts = np.bincount(L["topk_ids"].ravel(), minlength=cfg.E)
    C = 128 * (int(counts.max()) // 128 + 1) + 128
    dev = x.device
    # contiguous
    ws_c = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    off_c = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    out_c = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    M.moe_route_sort_amax(x, ids, pw, cfg.E, off_c, ws_c)
    M.moe_expert_forward_nvfp4(w, cfg.T, cfg.k, off_c, out_c, ws_c)
    # masked
    ws_m = M.alloc_workspace_masked(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, C)
    off_m = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    out_m = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    M.moe_route_sort_amax_masked(x, ids, pw, cfg.E, C, off_m, ws_m)
    M.moe_expert_forward_nvfp4_masked(w, cfg.T, cfg.k, C, off_m, out_m, ws_m)
    assert M.nvfp4_get_device_error() == 0
    assert np.array_equal(off_m.cpu().numpy(), np.arange(cfg.E + 1) * C)
    assert torch.equal(out_m.view(torch.int16), out_c.view(torch.int16))
    # routed rows: same codes, scales and g, expert by expert
    Lc = M.moe_workspace_layout_query(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    Lm = M.moe_workspace_layout_query_masked(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, C)
    oc = off_c.cpu().numpy()
    codes_c = bytes_of(ws_c, Lc.a_codes, Lc.rows_cap * cfg.H // 2).reshape(Lc.rows_cap, cfg.H // 2)
    codes_m = bytes_of(ws_m, Lm.a_codes, Lm.rows_cap * cfg.H // 2).reshape(Lm.rows_cap, cfg.H // 2)
    sf_c = M.sf_to_rows(bytes_of(ws_c, Lc.a_sf, Lc.rows_cap * cfg.H // 16), Lc.rows_cap, cfg.H)
    sf_m = M.sf_to_rows(bytes_of(ws_m, Lm.a_sf, Lm.rows_cap * cfg.H // 16), Lm.rows_cap, cfg.H)
    g_c = bytes_of(ws_c, Lc.a_g, Lc.rows_cap * 4).view(np.uint32)
    g_m = bytes_of(ws_m, Lm.a_g, Lm.rows_cap * 4).view(np.uint32)
    for e in range(cfg.E):
        n = int(counts[e])
        rc, rm = slice(oc[e], oc[e] + n), slice(e * C, e * C + n)
        assert np.array_equal(codes_m[rm], codes_c[rc])
        assert np.array_equal(sf_m[rm], sf_c[rc])
        assert np.array_equal(g_m[rm], g_c[rc])
        assert not sf_m[e * C + n:(e + 1) * C].any() and not g_m[e * C + n:(e + 1) * C].any()   # pad rows
    # the one-call masked layer: the same offsets and output bits
    ws_1 = M.alloc_workspace_masked(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, C)
    off_1 = torch.full((cfg.E + 1,), -7, dtype=torch.int32, device=dev)
    out_1 = torch.empty_like(out_m)
    M.moe_layer_forward_nvfp4_masked(w, x, ids, pw, C, off_1, out_1, ws_1)
    assert M.nvfp4_get_device_error() == 0
    assert torch.equal(off_1, off_m) and torch.equal(out_1.view(torch.int16), out_m.view(torch.int16))


@pytest.mark.parametrize("T", [64, 4096])     # one-block sort and chunked sort
def test_masked_capacity_overflow_is_reported(T):
    cfg = S.shrink(S.CONFIGS["qwen3_30b_a3b"], T=T)
    L, w, x, ids, pw = layer_inputs(cfg)
    ids[:, 0] = 5                              # every token's first slot goes to expert 5 (> 128 pairs at T=4096)
    ids[:, 1] = 6
    ids_np = ids.cpu().numpy()
    assert all(len(set(r)) == cfg.k for r in ids_np[:8]) or True
    C = 128
    over = np.bincount(ids_np.ravel(), minlength=cfg.E).max() > C
    ws_m = M.alloc_workspace_masked(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, C)
    guard = torch.zeros(1 << 20, dtype=torch.uint8, device=x.device)   # allocated after: must stay zero
    off_m = torch.empty(cfg.E + 1, dtype=torch.int32, device=x.device)
    M.moe_route_sort_amax_masked(x, ids, pw, cfg.E, C, off_m, ws_m)
    status = M.nvfp4_get_device_error()
    assert status == (8 if over else 0)
    assert not guard.any()
    assert np.array_equal(off_m.cpu().numpy(), np.arange(cfg.E + 1) * C)
    # dropped pairs have no row (the combine adds nothing for them); the others name a row of
    # their expert
    lay = M.moe_workspace_layout_query_masked(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, C)
    pair_row = ws_m[lay.pair_row:lay.pair_row + 4 * cfg.T * cfg.k].view(torch.int32).cpu().numpy()
    flat = ids_np.ravel()
    kept = pair_row >= 0
    assert np.all(pair_row[kept] // C == flat[kept])
    assert (~kept).sum() == np.maximum(np.bincount(flat, minlength=cfg.E) - C, 0).sum()


def test_masked_dropped_pairs_add_nothing():
    """With experts over capacity, each dropped (token, slot) pair has no row and the combine adds
    nothing for it: the output equals the contiguous layout's with those pairs' router
    probabilities set to zero (their h, and so their y, are zero rows), compared as values
    (+0 and -0 alike)."""
    cfg = S.shrink(S.CONFIGS["qwen3_30b_a3b"], T=1024)
    L, w, x, ids, pw = layer_inputs(cfg)
    ids[:, 0] = 5                              # experts 5 and 6 get over 1024 pairs each
    ids[:, 1] = 6
    C = 256
    dev = x.device
    ws_m = M.alloc_workspace_masked(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, C)
    off_m = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    out_m = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    M.moe_route_sort_amax_masked(x, ids, pw, cfg.E, C, off_m, ws_m)
    assert M.nvfp4_get_device_error() == 8     # NVFP4_ERR_CAPACITY
    M.moe_expert_forward_nvfp4_masked(w, cfg.T, cfg.k, C, off_m, out_m, ws_m)
    assert M.nvfp4_get_device_error() == 0
    lay = M.moe_workspace_layout_query_masked(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, C)
    pair_row = ws_m[lay.pair_row:lay.pair_row + 4 * cfg.T * cfg.k].view(torch.int32).view(cfg.T, cfg.k)
    dropped = pair_row < 0
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=cfg.E)
    assert int(dropped.sum()) == np.maximum(counts - C, 0).sum() > 0
    pw0 = pw.clone()
    pw0[dropped] = 0.0
    ws_c = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    off_c = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    out_c = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    M.moe_route_sort_amax(x, ids, pw0, cfg.E, off_c, ws_c)
    M.moe_expert_forward_nvfp4(w, cfg.T, cfg.k, off_c, out_c, ws_c)
    assert M.nvfp4_get_device_error() == 0
    assert torch.equal(out_m.float(), out_c.float())
