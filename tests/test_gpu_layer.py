"""End-to-end parity of the GPU layer (moe_route_sort_amax + moe_expert_forward_nvfp4)
with the oracle: output relative L2 <= 1e-2, FC2 requantisation code flips
<= 0.1%, the forward identical to the four stages called one by one and the
one-call layer (moe_layer_forward_nvfp4) identical to the two calls, and FC2
with the requantisation fused in (moe_fc2_requant_nvfp4) identical to the two
stages it replaces.
At the full 2048/768/128/top-8 size with 4096 tokens the oracle checks a
sample of routed rows and tokens."""

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import formats as F
from oracle import moe as OM
from oracle import quant as Q
from _helpers import FC2_CODE_FLIP_RATE, LAYER_REL_L2, bf16_to_torch, rel_l2, torch_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def gpu_layer(L, E, stages=False):
    T, H = L["x"].shape
    k = L["topk_ids"].shape[1]
    w = M.quantize_moe_weights(bf16_to_torch(L["w1"]), bf16_to_torch(L["w2"]))
    I = w.I
    ws = M.alloc_workspace(T, H, I, E, k)
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    M.moe_route_sort_amax(bf16_to_torch(L["x"]), torch.from_numpy(L["topk_ids"]).cuda(),
                          torch.from_numpy(L["topk_w"]).cuda(), E, offs, ws)
    if stages:
        M.moe_fc1_swiglu_nvfp4(w, T, k, offs, ws)
        M.moe_requant_nvfp4(w, T, k, offs, ws)
        M.moe_fc2_nvfp4(w, T, k, offs, ws)
        M.moe_combine_bf16(w, T, k, out, ws)
    else:
        M.moe_expert_forward_nvfp4(w, T, k, offs, out, ws)
    assert M.nvfp4_get_device_error() == 0
    return out, ws, offs, M.moe_workspace_layout_query(T, H, I, E, k)


def a2_codes_by_pair(ws, lay, offs, T, k, I):
    rc = lay.rows_cap
    used = int(offs.cpu().numpy()[-1])          # rows past expert_offsets[E] were never written
    pair = ws[lay.row_pair:lay.row_pair + 4 * rc].view(torch.int32).cpu().numpy()
    pair[used:] = -1
    codes = ws[lay.a2_codes:lay.a2_codes + rc * I // 2].cpu().numpy().reshape(rc, I // 2)
    out = np.zeros((T * k, I // 2), np.uint8)
    real = pair >= 0
    out[pair[real]] = codes[real]
    return out


@pytest.mark.parametrize("cfg", [
    S.CONFIGS["tiny"],
    S.LayerConfig("tiny_skew", H=256, I=128, E=8, k=2, T=200, routing="zipf", outlier_frac=0.02),
    S.LayerConfig("mid", H=1024, I=384, E=16, k=4, T=300),
    S.LayerConfig("qwen_slice", H=2048, I=768, E=128, k=8, T=96),
], ids=lambda c: c.name)
def test_layer_vs_oracle(cfg):
    L = S.make_layer(cfg)
    out, _, _, _ = gpu_layer(L, cfg.E)
    wq = OM.quantize_weights(L["w1"], L["w2"])
    ref, inter = OM.moe_forward(L["x"], L["topk_ids"], L["topk_w"], wq, keep=True)
    got = torch_to_bf16_bits(out)
    assert rel_l2(F.bf16_bits_to_f32(got), F.bf16_bits_to_f32(ref)) <= LAYER_REL_L2
    # the requantised FC2 operand: written to the workspace by the staged path (the fused FC2
    # keeps it in shared memory), whose output is bitwise the fused one
    out_s, ws, offs, lay = gpu_layer(L, cfg.E, stages=True)
    assert np.array_equal(torch_to_bf16_bits(out_s), got)
    ref_codes = Q.pack_nibbles(inter["hq"][0])
    gpu_codes = a2_codes_by_pair(ws, lay, offs, cfg.T, cfg.k, cfg.I)
    flips = (Q.unpack_nibbles(ref_codes) != Q.unpack_nibbles(gpu_codes)).mean()
    assert flips <= FC2_CODE_FLIP_RATE, flips


FUSED_CASES = [
    S.LayerConfig("mid", H=1024, I=384, E=16, k=4, T=300),
    S.LayerConfig("one_ntile", H=256, I=128, E=8, k=2, T=700),
    S.LayerConfig("narrow_i", H=512, I=256, E=4, k=2, T=2000, routing="zipf"),
    S.LayerConfig("skew", H=2048, I=768, E=32, k=4, T=900, routing="zipf", outlier_frac=0.01),
    S.LayerConfig("qwen_many_mtiles", H=2048, I=768, E=128, k=8, T=3000, routing="zipf", outlier_frac=0.01),
    S.LayerConfig("qwen_few_mtiles", H=2048, I=768, E=128, k=8, T=40),
]


@pytest.mark.parametrize("cfg", FUSED_CASES, ids=lambda c: c.name)
def test_fused_fc2_stage_equals_requant_then_fc2(cfg):
    """moe_fc2_requant_nvfp4 (the FC2 input quantised inside the FC2 kernel, never written to
    memory) against the two stages it replaces (requant writes A2, FC2 reads it back): y for
    every (token, slot) and FC2's FP32 pre-cast values bit for bit, over shapes whose m-tile
    counts make the fused kernel group n-tiles differently, with partial K blocks (I = 384),
    one n-tile (H = 256), Zipf routing and outlier channels; and the whole forward against the
    four stages called one by one."""
    L = S.make_layer(cfg)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    w = M.quantize_moe_weights(bf16_to_torch(L["w1"]), bf16_to_torch(L["w2"]))
    ws = M.alloc_workspace(T, H, I, E, k)
    lay = M.moe_workspace_layout_query(T, H, I, E, k)
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    M.moe_route_sort_amax(bf16_to_torch(L["x"]), torch.from_numpy(L["topk_ids"]).cuda(),
                          torch.from_numpy(L["topk_w"]).cuda(), E, offs, ws)
    M.moe_fc1_swiglu_nvfp4(w, T, k, offs, ws)
    y_view = ws[lay.y:lay.y + 2 * lay.rows_cap * H]          # per routed row; pad rows unwritten
    d1 = torch.full((lay.rows_cap, H), float("nan"), device="cuda")
    d2 = torch.full((lay.rows_cap, H), float("nan"), device="cuda")
    M.moe_requant_nvfp4(w, T, k, offs, ws)
    y_view.zero_()
    M.moe_fc2_nvfp4(w, T, k, offs, ws, debug=d1)
    y1 = y_view.clone()
    for _ in range(2):                  # twice: the second call starts from the first one's leftovers
        y_view.zero_()
        M.moe_fc2_requant_nvfp4(w, T, k, offs, ws, debug=d2)
        assert M.nvfp4_get_device_error() == 0
        assert torch.equal(y1, y_view)
        assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))     # NaN-filled pad rows alike
    a = torch_to_bf16_bits(gpu_layer(L, E)[0])
    b = torch_to_bf16_bits(gpu_layer(L, E, stages=True)[0])
    assert np.array_equal(a, b)


def test_fused_fc2_rejects_wide_intermediate():
    cfg = S.LayerConfig("wide", H=256, I=1024, E=2, k=1, T=8)
    assert M.moe_fc2_requant_max_intermediate() == 768
    w = M.quantize_moe_weights(torch.zeros((2, 2048, 256), dtype=torch.bfloat16, device="cuda"),
                               torch.zeros((2, 256, 1024), dtype=torch.bfloat16, device="cuda"))
    ws = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    offs = torch.zeros(cfg.E + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(M.NVFP4Error, match="UNSUPPORTED_SHAPE"):
        M.moe_fc2_requant_nvfp4(w, cfg.T, cfg.k, offs, ws)


@pytest.mark.parametrize("cfg", [
    S.LayerConfig("one_block_sort", H=256, I=128, E=8, k=2, T=300, seed=11),                 # <= 8192 pairs
    S.LayerConfig("chunked_sort", H=2048, I=768, E=128, k=8, T=1500, seed=12, routing="zipf"),
    S.LayerConfig("empty", H=256, I=128, E=8, k=2, T=0, seed=13),
], ids=lambda c: c.name)
def test_layer_call_equals_route_then_forward(cfg):
    # the one-call layer (FC1 chained to the route sort by programmatic launch) gives the two
    # calls' output, offsets and routed rows bit for bit
    L = S.make_layer(cfg)
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    out2, ws2, offs2, lay = gpu_layer(L, E)
    w = M.quantize_moe_weights(bf16_to_torch(L["w1"]), bf16_to_torch(L["w2"]))
    ws = M.alloc_workspace(T, H, cfg.I, E, k)
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    M.moe_layer_forward_nvfp4(w, bf16_to_torch(L["x"]), torch.from_numpy(L["topk_ids"]).cuda(),
                              torch.from_numpy(L["topk_w"]).cuda(), offs, out, ws)
    assert M.nvfp4_get_device_error() == 0
    assert torch.equal(offs, offs2)
    assert np.array_equal(torch_to_bf16_bits(out), torch_to_bf16_bits(out2))
    if T:
        rows = int(offs[-1].item())
        pair = ws[lay.row_pair:lay.row_pair + 4 * rows].view(torch.int32)
        assert torch.equal(pair, ws2[lay.row_pair:lay.row_pair + 4 * rows].view(torch.int32))
        real = pair >= 0                              # pad rows of h are never written
        for name, width in (("a_codes", H // 2), ("h", 2 * cfg.I)):
            a = ws[getattr(lay, name):getattr(lay, name) + rows * width].view(rows, width)
            b = ws2[getattr(lay, name):getattr(lay, name) + rows * width].view(rows, width)
            assert torch.equal(a[real], b[real]), name


def test_run_to_run_deterministic():
    cfg = S.LayerConfig("skew", H=2048, I=768, E=32, k=4, T=700, routing="zipf", outlier_frac=0.01)
    L = S.make_layer(cfg)
    a = torch_to_bf16_bits(gpu_layer(L, cfg.E)[0])
    b = torch_to_bf16_bits(gpu_layer(L, cfg.E)[0])
    assert np.array_equal(a, b)


def test_dense_special_case_on_gpu():
    # one expert, top-1, probability 1: the layer is a quantised SwiGLU MLP
    cfg = S.LayerConfig("dense", H=512, I=256, E=1, k=1, T=130)
    L = S.make_layer(cfg)
    out = torch_to_bf16_bits(gpu_layer(L, 1)[0])
    ref = OM.dense_swiglu_mlp_f64(F.bf16_bits_to_f32(L["x"]), F.bf16_bits_to_f32(L["w1"][0]),
                                  F.bf16_bits_to_f32(L["w2"][0]))
    assert rel_l2(F.bf16_bits_to_f32(out), ref) < 0.30
    wq = OM.quantize_weights(L["w1"], L["w2"])
    assert rel_l2(F.bf16_bits_to_f32(out), F.bf16_bits_to_f32(OM.moe_forward(
        L["x"], L["topk_ids"], L["topk_w"], wq))) <= LAYER_REL_L2


def test_qwen3_30b_a3b_full_size_sampled():
    """4096 tokens, 2048/768, 128 experts, top-8: every routed row of a few experts
    and the full output of a few tokens against the oracle."""
    cfg = S.CONFIGS["qwen3_30b_a3b"]
    L = S.make_layer(cfg)
    out, ws, offs, lay = gpu_layer(L, cfg.E)
    got = torch_to_bf16_bits(out)
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(cfg.T, 6, replace=False))
    wq = OM.quantize_weights(L["w1"], L["w2"])
    ref = OM.moe_forward(L["x"][toks], L["topk_ids"][toks], L["topk_w"][toks], wq)
    assert rel_l2(F.bf16_bits_to_f32(got[toks]), F.bf16_bits_to_f32(ref)) <= LAYER_REL_L2
    # per-slot FC2 outputs of every pair routed to experts {0, 77, 127}
    rc = lay.rows_cap
    y = ws[lay.y:lay.y + rc * cfg.H * 2].view(torch.int16).cpu().numpy().view(np.uint16).reshape(rc, cfg.H)
    pair_row = ws[lay.pair_row:lay.pair_row + 4 * cfg.T * cfg.k].view(torch.int32).cpu().numpy()
    pair_row = pair_row.reshape(cfg.T, cfg.k)
    for e in (0, 77, 127):
        t_e, s_e = np.nonzero(L["topk_ids"] == e)
        sub_ids = np.zeros((len(t_e), 1), np.int32) + e
        sub_w = L["topk_w"][t_e, s_e][:, None]
        _, inter = OM.moe_forward(L["x"][t_e], sub_ids, sub_w, wq, keep=True)
        y_e = y[pair_row[t_e, s_e]]
        assert rel_l2(F.bf16_bits_to_f32(y_e), F.bf16_bits_to_f32(inter["y"][:, 0])) <= LAYER_REL_L2
