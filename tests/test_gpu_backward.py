"""GPU parity of the straight-through backward (moe_expert_backward_ste) with the oracle
(oracle/backward.py).

Inputs are seeded (moe_synth): BF16 x, W1, W2, dOut and the routing.  The saved activations
the backward reads (the forward's BF16 gate/up and h) are the oracle forward's, put into the
GPU workspace rows through the GPU route sort's row map; pad rows hold NaN, so a pad row that
leaks into a gradient shows.  Tolerances:

* against the oracle with BF16 stages (dh, [dgate, dup], each slot's dX and dX rounded where
  the GPU rounds them): the two sides differ only by FP32 against FP64 sums before the same
  roundings, which now and then moves a BF16 rounding by one unit; at least 90% of dX is
  bitwise equal (a missing or misplaced rounding moves about half of it) and the relative L2
  is <= 6e-4 for dX and <= 3e-4 for dW1 and dprob (a misplaced rounding costs about 1e-3);
  dW2 (no rounded operand) <= 1e-5;
* against the exact FP64 oracle: relative L2 <= 2 sqrt(n) 2^-9/sqrt(3) for a result behind n
  BF16 roundings (dX 4, dW1 2, dprob 1), about the BF16-backward figure the miniTE page
  reports (0.001663);
* an expert without pairs gets exactly zero weight gradients, T = 0 zeroes them, and a
  token's dX and dprob are bitwise the same in a smaller batch.
"""

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import backward as OB
from oracle import formats as F
from oracle import moe as OM
from _helpers import bf16_to_torch, rel_l2, torch_to_bf16_bits

pytestmark = pytest.mark.gpu

STAGED_REL_L2 = {"dx": 6e-4, "dw1": 3e-4, "dprob": 3e-4}
STAGED_DX_EQUAL = 0.9
DW2_REL_L2 = 1e-5
_U = 2.0 ** -9 / np.sqrt(3)
EXACT_REL_L2 = {"dx": 2 * np.sqrt(4) * _U, "dw1": 2 * np.sqrt(2) * _U, "dprob": 2 * _U, "dw2": 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def _f(bits):
    return F.bf16_bits_to_f32(bits).astype(np.float64)


def make_case(H, I, E, k, T, seed, routing="uniform", unused_experts=0, ids=None):
    """Seeded inputs; the last `unused_experts` experts get no pairs; `ids` replaces the
    routing's expert ids (the probabilities stay the seeded ones)."""
    cfg = S.LayerConfig("bwd", H=H, I=I, E=E, k=k, T=T, seed=seed, routing=routing)
    x = S.make_x(cfg)
    ids_r, p = S.make_routing(S.shrink(cfg, E=E - unused_experts))
    ids = ids_r if ids is None else np.ascontiguousarray(ids, dtype=ids_r.dtype)
    w1, w2 = S.make_weights(cfg)
    dout = S.make_grad_out(cfg)
    wq = OM.quantize_weights(w1, w2)
    _, inter = OM.moe_forward(x, ids, p, wq, keep=True)
    gu = inter["gu"].reshape(T, k, 2 * I)          # the forward's BF16 gate/up per (token, slot)
    h = inter["h"].reshape(T, k, I)                # the forward's BF16 SwiGLU x prob
    return dict(x=x, ids=ids, p=p, w1=w1, w2=w2, dout=dout, gu=gu, h=h, H=H, I=I, E=E, k=k, T=T)


def gpu_backward(c):
    """Route on the GPU, place the saved activations, run the backward; numpy results."""
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    x = bf16_to_torch(c["x"])
    ws = M.alloc_workspace(T, H, I, E, k)
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    M.moe_route_sort_amax(x, torch.from_numpy(c["ids"]).cuda(), torch.from_numpy(c["p"]).cuda(), E, offs, ws)
    torch.cuda.synchronize()
    L = M.moe_workspace_layout_query(T, H, I, E, k)
    rc = L.rows_cap
    used = int(offs[-1].item())
    pair = ws[L.row_pair:L.row_pair + 4 * rc].view(torch.int32).cpu().numpy().copy()
    pair[used:] = -1
    real = pair >= 0
    h_rows = np.full((rc, I), 0x7FC0, np.uint16)                 # NaN in pad rows
    h_rows[real] = c["h"].reshape(T * k, I)[pair[real]]
    ws[L.h:L.h + rc * I * 2].copy_(torch.from_numpy(h_rows.view(np.uint8).ravel()).cuda())
    gu_rows = np.full((rc, 2 * I), 0x7FC0, np.uint16)              # NaN in pad rows
    gu_rows[real] = c["gu"].reshape(T * k, 2 * I)[pair[real]]
    gu = bf16_to_torch(gu_rows)
    wt = M.MoEWeightsBF16(bf16_to_torch(c["w1"]), bf16_to_torch(c["w2"]))
    dx = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dw1 = torch.full((E, 2 * I, H), float("nan"), device="cuda")
    dw2 = torch.full((E, H, I), float("nan"), device="cuda")
    dprob = torch.empty((T, k), dtype=torch.float32, device="cuda")
    bws = M.alloc_backward_workspace(T, H, I, E, k)
    M.moe_expert_backward_ste(wt, T, k, x, bf16_to_torch(c["dout"]), offs, ws, gu, dx, dw1, dw2, dprob, bws)
    assert M.nvfp4_get_device_error() == 0
    return dict(dx=_f(torch_to_bf16_bits(dx)), dx_bits=torch_to_bf16_bits(dx), dw1=dw1.cpu().numpy(),
                dw2=dw2.cpu().numpy(), dprob=dprob.cpu().numpy())


def oracle_backward(c, bf16_stages):
    return OB.moe_backward_ste(_f(c["dout"]), _f(c["x"]), c["ids"], c["p"], _f(c["w1"]), _f(c["w2"]),
                               _f(c["gu"]), _f(c["h"]), bf16_stages=bf16_stages)


CASES = [
    dict(H=256, I=128, E=9, k=2, T=300, seed=1, unused_experts=1),          # N = 128 tiles, an empty expert
    dict(H=512, I=256, E=16, k=4, T=200, seed=2, routing="zipf"),           # N = 256 tiles, skewed routing
    dict(H=256, I=384, E=4, k=2, T=150, seed=3),                            # I % 256 = 128
    dict(H=256, I=128, E=300, k=2, T=200, seed=7, unused_experts=40),       # many experts, most with a
                                                                            # few rows, 40+ empty
]


@pytest.mark.parametrize("case", CASES, ids=["h256_i128_e9", "h512_i256_e16_zipf", "h256_i384_e4",
                                             "h256_i128_e300"])
def test_backward_matches_oracle(case):
    c = make_case(**case)
    g = gpu_backward(c)
    st = oracle_backward(c, bf16_stages=True)
    ex = oracle_backward(c, bf16_stages=False)
    report = {}
    for name in ("dx", "dw1", "dprob"):
        assert np.all(np.isfinite(g[name])), name
        report[name] = (rel_l2(g[name], st[name]), rel_l2(g[name], ex[name]))
    report["dx_equal"] = float(np.mean(g["dx"] == st["dx"]))
    print("backward parity", case, report)
    assert report["dx_equal"] >= STAGED_DX_EQUAL, report
    for name in ("dx", "dw1", "dprob"):
        assert report[name][0] <= STAGED_REL_L2[name], (name, report)
        assert report[name][1] <= EXACT_REL_L2[name], (name, report)
    assert rel_l2(g["dw2"], ex["dw2"]) <= DW2_REL_L2
    # experts without pairs
    counts = np.bincount(c["ids"].ravel(), minlength=c["E"])
    for e in np.nonzero(counts == 0)[0]:
        assert np.all(g["dw1"][e] == 0) and np.all(g["dw2"][e] == 0)


def test_backward_whole_stage_tails():
    # experts with exactly 128, 64 and 192 real rows (K stages of 64 rows end on a real row)
    # and 0, 64 and 64 pad rows (a stage of pad rows only is skipped; h's pad rows are NaN)
    T, k, E = 192, 2, 4
    ids = np.zeros((T, k), np.int32)
    ids[128:, 0] = 1
    ids[:, 1] = 2
    c = make_case(H=256, I=128, E=E, k=k, T=T, seed=6, ids=ids)
    assert list(np.bincount(ids.ravel(), minlength=E)) == [128, 64, 192, 0]
    g = gpu_backward(c)
    ex = oracle_backward(c, bf16_stages=False)
    for name in ("dx", "dw1", "dprob"):
        assert np.all(np.isfinite(g[name])), name
        assert rel_l2(g[name], ex[name]) <= EXACT_REL_L2[name], (name, rel_l2(g[name], ex[name]))
    assert rel_l2(g["dw2"], ex["dw2"]) <= DW2_REL_L2
    assert np.all(g["dw1"][3] == 0) and np.all(g["dw2"][3] == 0)


def test_backward_batch_invariance():
    c = make_case(H=256, I=128, E=8, k=2, T=300, seed=4)
    g = gpu_backward(c)
    for T2 in (1, 77, 128):
        c2 = dict(c, T=T2, x=c["x"][:T2], ids=c["ids"][:T2], p=c["p"][:T2], dout=c["dout"][:T2],
                  gu=c["gu"][:T2], h=c["h"][:T2])
        g2 = gpu_backward(c2)
        assert np.array_equal(g2["dx_bits"], g["dx_bits"][:T2])
        assert np.array_equal(g2["dprob"].view(np.uint32), g["dprob"][:T2].view(np.uint32))


def test_backward_empty_batch_zeroes_weight_gradients():
    E, H, I, k = 4, 256, 128, 2
    wt = M.MoEWeightsBF16(torch.zeros((E, 2 * I, H), dtype=torch.bfloat16, device="cuda"),
                          torch.zeros((E, H, I), dtype=torch.bfloat16, device="cuda"))
    dw1 = torch.full((E, 2 * I, H), float("nan"), device="cuda")
    dw2 = torch.full((E, H, I), float("nan"), device="cuda")
    e0 = torch.empty(0, device="cuda")
    ws = M.alloc_workspace(0, H, I, E, k)
    M.moe_expert_backward_ste(wt, 0, k, e0, e0, torch.zeros(E + 1, dtype=torch.int32, device="cuda"), ws, e0,
                              e0, dw1, dw2, e0, ws)
    torch.cuda.synchronize()
    assert bool((dw1 == 0).all()) and bool((dw2 == 0).all())


def test_layer_forward_backward_pipeline():
    # the GPU forward saves its own activations; its gradients agree with the oracle's
    # (fed with the oracle forward's activations) within the exact-reading bounds
    c = make_case(H=512, I=256, E=16, k=4, T=256, seed=5, routing="zipf")
    layer = M.MoELayer(bf16_to_torch(c["w1"]), bf16_to_torch(c["w2"]))
    x = bf16_to_torch(c["x"])
    ids = torch.from_numpy(c["ids"]).cuda()
    p = torch.from_numpy(c["p"]).cuda()
    out_saved = layer.forward(x, ids, p, save_for_backward=True)
    dx, dw1, dw2, dprob = layer.backward(bf16_to_torch(c["dout"]))
    assert M.nvfp4_get_device_error() == 0
    out_plain = layer.forward(x, ids, p)
    assert torch.equal(out_saved, out_plain)
    ex = oracle_backward(c, bf16_stages=False)
    got = dict(dx=_f(torch_to_bf16_bits(dx)), dw1=dw1.cpu().numpy(), dw2=dw2.cpu().numpy(),
               dprob=dprob.cpu().numpy())
    for name in ("dx", "dw1", "dprob"):
        assert rel_l2(got[name], ex[name]) <= EXACT_REL_L2[name], (name, rel_l2(got[name], ex[name]))
    assert rel_l2(got["dw2"], ex["dw2"]) <= 1e-3     # h itself comes from the GPU forward here


def test_backward_qwen3_30b_a3b_full_size_sampled():
    """The backward at the size the bench times (4096 tokens, H 2048, I 768, 128 experts, top-8):
    dW1 and dW2 of three experts over all their pairs, and dX and dprob of six tokens, against the
    oracle fed with the GPU forward's own saved gate/up and h (so the backward alone is checked).
    An expert's weight gradients sum over its own pairs only, and a token's dX and dprob over its
    own k pairs, so each sample is the oracle on that expert's pairs or that token's slots."""
    cfg = S.CONFIGS["qwen3_30b_a3b"]
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    Lay = S.make_layer(cfg)
    dout_bits = S.make_grad_out(cfg)
    w = M.quantize_moe_weights(bf16_to_torch(Lay["w1"]), bf16_to_torch(Lay["w2"]))
    x = bf16_to_torch(Lay["x"])
    ws = M.alloc_workspace(T, H, I, E, k)
    lay = M.moe_workspace_layout_query(T, H, I, E, k)
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    M.moe_route_sort_amax(x, torch.from_numpy(Lay["topk_ids"]).cuda(), torch.from_numpy(Lay["topk_w"]).cuda(), E,
                          offs, ws)
    rc = lay.rows_cap
    gu = torch.empty((rc, 2 * I), dtype=torch.bfloat16, device="cuda")
    M.moe_fc1_swiglu_save_nvfp4(w, T, k, offs, ws, gu)
    wt = M.MoEWeightsBF16(bf16_to_torch(Lay["w1"]), bf16_to_torch(Lay["w2"]))
    dx = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dw1 = torch.full((E, 2 * I, H), float("nan"), device="cuda")
    dw2 = torch.full((E, H, I), float("nan"), device="cuda")
    dprob = torch.empty((T, k), dtype=torch.float32, device="cuda")
    bws = M.alloc_backward_workspace(T, H, I, E, k)
    M.moe_expert_backward_ste(wt, T, k, x, bf16_to_torch(dout_bits), offs, ws, gu, dx, dw1, dw2, dprob, bws)
    assert M.nvfp4_get_device_error() == 0
    # the saved values of every (token, slot): the BF16 gate/up the SwiGLU ran on, and h
    pair_row = ws[lay.pair_row:lay.pair_row + 4 * T * k].view(torch.int32).cpu().numpy().reshape(T, k)
    gu_bits = torch_to_bf16_bits(gu)
    h_rows = ws[lay.h:lay.h + 2 * rc * I].view(torch.int16).cpu().numpy().view(np.uint16).reshape(rc, I)

    def saved(t, s):
        rows = pair_row[t, s]
        return gu_bits[rows], h_rows[rows]

    ids, p = Lay["topk_ids"], Lay["topk_w"]
    dw1_g, dw2_g = dw1.cpu().numpy(), dw2.cpu().numpy()
    for e in (0, 77, 127):
        t_e, s_e = np.nonzero(ids == e)
        gu_e, h_e = saved(t_e, s_e)
        args = (_f(dout_bits[t_e]), _f(Lay["x"][t_e]), np.zeros((len(t_e), 1), np.int32), p[t_e, s_e][:, None],
                _f(Lay["w1"][e:e + 1]), _f(Lay["w2"][e:e + 1]), _f(gu_e[:, None]), _f(h_e[:, None]))
        st = OB.moe_backward_ste(*args, bf16_stages=True)
        ex = OB.moe_backward_ste(*args, bf16_stages=False)
        assert rel_l2(dw1_g[e], st["dw1"][0]) <= STAGED_REL_L2["dw1"], e
        assert rel_l2(dw2_g[e], ex["dw2"][0]) <= DW2_REL_L2, e
    toks = np.sort(np.random.default_rng(1).choice(T, 6, replace=False))
    dx_g = _f(torch_to_bf16_bits(dx))
    dprob_g = dprob.cpu().numpy()
    got_dx, ref_dx, got_p, ref_p = [], [], [], []
    for t in toks:
        e_t = ids[t]
        gu_t, h_t = saved(np.full(k, t), np.arange(k))
        st = OB.moe_backward_ste(_f(dout_bits[t:t + 1]), _f(Lay["x"][t:t + 1]), np.arange(k, dtype=np.int32)[None],
                                 p[t:t + 1], _f(Lay["w1"][e_t]), _f(Lay["w2"][e_t]), _f(gu_t[None]), _f(h_t[None]),
                                 bf16_stages=True)
        got_dx.append(dx_g[t]), ref_dx.append(st["dx"][0]), got_p.append(dprob_g[t]), ref_p.append(st["dprob"][0])
    got_dx, ref_dx = np.array(got_dx), np.array(ref_dx)
    assert np.mean(got_dx == ref_dx) >= STAGED_DX_EQUAL
    assert rel_l2(got_dx, ref_dx) <= STAGED_REL_L2["dx"]
    assert rel_l2(np.array(got_p), np.array(ref_p)) <= STAGED_REL_L2["dprob"]
