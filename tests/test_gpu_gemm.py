"""GPU parity of each expert-forward stage given identical quantised inputs:

* FC1 (tcgen05 block-scaled FP4 grouped GEMM + FP32 epilogue): pre-cast FP32
  values within relative L2 1e-5 of the oracle's exact FP64 values, BF16
  gate/up within 1 ulp; SwiGLU x prob bit-exact wherever gate and up agree,
  and elsewhere every element within the bound the gate/up difference
  propagates to (tests/_helpers.h_bound); the row maxima equal max|h|.
* requantisation of a seeded synthetic FC2 input: bit-exact.
* FC2 on that input: pre-cast within 1e-5, BF16 y within 1 ulp.
* combine of a seeded synthetic y: bit-exact.

Shapes cover one and several K stages, a partial last K stage (I = 128, 384),
several n tiles, many m tiles per expert (Zipf routing) and many near-empty
experts (128 experts, few tokens)."""

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import formats as F
from oracle import moe as OM
from oracle import quant as Q
from _helpers import (GEMM_BF16_ULP, GEMM_REL_L2, bf16_to_torch, bf16_ulp_distance, h_bound, rel_l2,
                      torch_to_bf16_bits)

pytestmark = pytest.mark.gpu

CASES = [
    S.LayerConfig("tiny", H=256, I=128, E=8, k=2, T=64),
    S.LayerConfig("mid", H=1024, I=384, E=16, k=4, T=300),
    S.LayerConfig("many_experts", H=2048, I=768, E=128, k=8, T=128),
    S.LayerConfig("skew", H=2048, I=768, E=16, k=2, T=2000, routing="zipf", outlier_frac=0.01),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def ws_view(ws, off, n, dtype):
    nbytes = n * torch.empty(0, dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


class Run:
    """One layer on the GPU, kept stage by stage."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.L = S.make_layer(cfg)
        c = cfg
        self.w = M.quantize_moe_weights(bf16_to_torch(self.L["w1"]), bf16_to_torch(self.L["w2"]))
        self.ws = M.alloc_workspace(c.T, c.H, c.I, c.E, c.k)
        self.lay = M.moe_workspace_layout_query(c.T, c.H, c.I, c.E, c.k)
        self.offs = torch.empty(c.E + 1, dtype=torch.int32, device="cuda")
        M.moe_route_sort_amax(bf16_to_torch(self.L["x"]), torch.from_numpy(self.L["topk_ids"]).cuda(),
                              torch.from_numpy(self.L["topk_w"]).cuda(), c.E, self.offs, self.ws)
        self.off_np = self.offs.cpu().numpy()
        rc = self.lay.rows_cap
        self.pair = ws_view(self.ws, self.lay.row_pair, rc, torch.int32).cpu().numpy()
        # rows past expert_offsets[E] are capacity the route sort never touched
        self.real = np.nonzero(self.pair[:self.off_np[-1]] >= 0)[0]
        self.expert = np.searchsorted(self.off_np, self.real, side="right") - 1
        self.wq = OM.quantize_weights(self.L["w1"], self.L["w2"])

    def view(self, name, n, dtype):
        return ws_view(self.ws, getattr(self.lay, name), n, dtype)


@pytest.fixture(scope="module", params=CASES, ids=lambda c: c.name)
def run(request):
    return Run(request.param)


def test_fc1_stage(run):
    c = run.cfg
    rc = run.lay.rows_cap
    dbg = torch.zeros((rc, 2 * c.I), dtype=torch.float32, device="cuda")
    M.moe_fc1_swiglu_nvfp4(run.w, c.T, c.k, run.offs, run.ws, debug=dbg)
    assert M.nvfp4_get_device_error() == 0
    v_gpu = dbg.cpu().numpy()[run.real]
    h_gpu = run.view("h", rc * c.I, torch.int16).cpu().numpy().view(np.uint16).reshape(rc, c.I)[run.real]
    amax2 = run.view("amax2", rc, torch.int32).cpu().numpy().view(np.uint32)[run.real]

    xq = Q.quantize_rows(F.bf16_bits_to_f32(run.L["x"]))
    toks, slots = run.pair[run.real] // c.k, run.pair[run.real] % c.k
    v_ref = np.zeros_like(v_gpu, dtype=np.float64)
    for e in np.unique(run.expert):
        sel = run.expert == e
        (c1, s1, g1), _ = run.wq.expert(int(e))
        t = toks[sel]
        v_ref[sel] = OM.epilogue_f64(OM.qgemm_f64(xq[0][t], xq[1][t], c1, s1), xq[2][t], g1)
    assert rel_l2(v_gpu, v_ref) <= GEMM_REL_L2
    gu_gpu = F.round_to_bf16_bits(v_gpu)
    gu_ref = F.round_to_bf16_bits(v_ref)
    assert bf16_ulp_distance(gu_gpu, gu_ref).max() <= GEMM_BF16_ULP

    # SwiGLU x prob: bit-exact wherever the gate and up values the two sides cast agree
    h_ref = OM.swiglu_prob(gu_ref[:, :c.I], gu_ref[:, c.I:], run.L["topk_w"][toks, slots])
    same = (gu_gpu[:, :c.I] == gu_ref[:, :c.I]) & (gu_gpu[:, c.I:] == gu_ref[:, c.I:])
    assert same.mean() > 0.9
    assert np.array_equal(h_gpu[same], h_ref[same])
    # where gate or up differ (by their 1-ulp cast difference), every element of h stays
    # within the bound that difference propagates to through silu(gate)*up*p
    diff = ~same
    f = F.bf16_bits_to_f32
    pr = np.broadcast_to(run.L["topk_w"][toks, slots][:, None], same.shape)
    bound = h_bound(f(gu_gpu[:, :c.I])[diff], f(gu_gpu[:, c.I:])[diff], f(gu_ref[:, :c.I])[diff],
                    f(gu_ref[:, c.I:])[diff], pr[diff], f(h_gpu)[diff], f(h_ref)[diff])
    err = np.abs(f(h_gpu)[diff].astype(np.float64) - f(h_ref)[diff])
    assert (err <= bound).all(), float((err / bound).max())
    # FC2 maxima: the producer's max|h| over each row
    hmax = np.abs(F.bf16_bits_to_f32(h_gpu)).max(axis=1)
    assert np.array_equal(amax2, hmax.view(np.uint32))


def test_fc1_save_matches_debug(run):
    # the training forward's FC1 saves the BF16 gate/up its SwiGLU ran on: bitwise the BF16
    # rounding of the FP32 epilogue values, with h and the FC2 maxima unchanged; pad rows and
    # rows past expert_offsets[E] keep what they held
    c = run.cfg
    rc = run.lay.rows_cap
    dbg = torch.zeros((rc, 2 * c.I), dtype=torch.float32, device="cuda")
    M.moe_fc1_swiglu_nvfp4(run.w, c.T, c.k, run.offs, run.ws, debug=dbg)
    h0 = run.view("h", rc * c.I, torch.int16).cpu().numpy()[:run.off_np[-1] * c.I].copy()
    a0 = run.view("amax2", rc, torch.int32).cpu().numpy()[run.real].copy()
    gu = torch.full((rc, 2 * c.I), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.moe_fc1_swiglu_save_nvfp4(run.w, c.T, c.k, run.offs, run.ws, gu)
    assert M.nvfp4_get_device_error() == 0
    gu_bits = torch_to_bf16_bits(gu)
    assert np.array_equal(gu_bits[run.real], F.round_to_bf16_bits(dbg.cpu().numpy()[run.real]))
    untouched = np.ones(rc, bool)
    untouched[run.real] = False
    assert np.array_equal(gu_bits[untouched], np.full((untouched.sum(), 2 * c.I), 0x7FC0, np.uint16))
    h1 = run.view("h", rc * c.I, torch.int16).cpu().numpy()[:run.off_np[-1] * c.I]
    assert np.array_equal(h0, h1)
    assert np.array_equal(a0, run.view("amax2", rc, torch.int32).cpu().numpy()[run.real])


def _synthetic_h(run, seed):
    c = run.cfg
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((len(run.real), c.I)).astype(np.float32)
    h *= np.exp2(rng.uniform(-8, 2, (len(run.real), 1))).astype(np.float32)
    h[:, rng.choice(c.I, 2, replace=False)] *= 16
    return S.f32_to_bf16_bits(h)


def test_requant_and_fc2_stage(run):
    c = run.cfg
    rc = run.lay.rows_cap
    h = _synthetic_h(run, seed=c.T)
    full = np.zeros((rc, c.I), np.uint16)
    full[run.real] = h
    run.view("h", rc * c.I, torch.int16).copy_(torch.from_numpy(full.view(np.int16).ravel()).cuda())
    amax = np.zeros(rc, np.float32)
    amax[run.real] = np.abs(F.bf16_bits_to_f32(h)).max(axis=1)
    run.view("amax2", rc, torch.int32).copy_(torch.from_numpy(amax.view(np.int32)).cuda())
    M.moe_requant_nvfp4(run.w, c.T, c.k, run.offs, run.ws)
    dbg = torch.zeros((rc, c.H), dtype=torch.float32, device="cuda")
    M.moe_fc2_nvfp4(run.w, c.T, c.k, run.offs, run.ws, debug=dbg)
    assert M.nvfp4_get_device_error() == 0

    # requantisation: bit-exact
    hc, hs, hg = Q.quantize_rows(F.bf16_bits_to_f32(h))
    a2c = run.view("a2_codes", rc * c.I // 2, torch.uint8).cpu().numpy().reshape(rc, c.I // 2)
    a2s = run.view("a2_sf", rc * c.I // 16, torch.uint8).cpu().numpy()
    a2g = run.view("a2_g", rc, torch.float32).cpu().numpy()
    assert np.array_equal(a2c[run.real], Q.pack_nibbles(hc))
    assert np.array_equal(M.sf_to_rows(a2s, rc, c.I)[run.real], hs)
    assert np.array_equal(a2g[run.real].view(np.uint32), hg.view(np.uint32))
    pads = np.nonzero(run.pair[:run.off_np[-1]] < 0)[0]
    assert not M.sf_to_rows(a2s, rc, c.I)[pads].any() and not a2g[pads].any()

    # FC2 on identical quantised inputs
    v_gpu = dbg.cpu().numpy()[run.real]
    v_ref = np.zeros_like(v_gpu, dtype=np.float64)
    for e in np.unique(run.expert):
        sel = run.expert == e
        _, (c2, s2, g2) = run.wq.expert(int(e))
        v_ref[sel] = OM.epilogue_f64(OM.qgemm_f64(hc[sel], hs[sel], c2, s2), hg[sel], g2)
    assert rel_l2(v_gpu, v_ref) <= GEMM_REL_L2
    y = run.view("y", rc * c.H, torch.int16).cpu().numpy().view(np.uint16).reshape(rc, c.H)
    y_rows = y[run.real]                                               # y is per routed row
    assert np.array_equal(y_rows, F.round_to_bf16_bits(v_gpu))        # the kernel's own cast
    assert bf16_ulp_distance(y_rows, F.round_to_bf16_bits(v_ref)).max() <= GEMM_BF16_ULP


# Requant lane mappings: a batch of R rows per warp in P passes of 32 blocks (I = 128: R 4,
# P 1; 256: R 2, P 1; 384: R 4, P 3; 1024: P 2; 1536: P 3; 2048: P 4), the coalesced
# warp-per-row kernel (640: five passes would be needed) and the lane-owns-groups kernel
# (2304 > 2048).  Rows include zeros, values whose divisors fall below the Markstein range
# (the IEEE-division fallback) and one row each with an infinity and a NaN (zero codes,
# scales and g, flagged as non-finite).
@pytest.mark.parametrize("I", [128, 256, 384, 640, 1024, 1536, 2048, 2304])
def test_requant_lane_mappings(I):
    c = S.LayerConfig(f"rq{I}", H=256, I=I, E=4, k=2, T=150)
    run = Run(c)
    rc = run.lay.rows_cap
    rng = np.random.default_rng(I)
    n = len(run.real)
    h = rng.standard_normal((n, I)).astype(np.float32)
    h *= np.exp2(rng.uniform(-8, 2, (n, 1))).astype(np.float32)
    h[0] = 0.0
    h[1] *= np.float32(2.0 ** -110)                  # g*6 and g*s below 2^-60
    h[2, : I // 2] *= np.float32(2.0 ** -120)       # BF16 subnormals beside normal values
    bits = S.f32_to_bf16_bits(h)
    bad = {3: 0x7F80, 4: 0x7FC0}                      # +inf, NaN
    for row, b in bad.items():
        bits[row, 7] = b
    full = np.zeros((rc, I), np.uint16)
    full[run.real] = bits
    run.view("h", rc * I, torch.int16).copy_(torch.from_numpy(full.view(np.int16).ravel()).cuda())
    f = F.bf16_bits_to_f32(bits)
    amax = np.zeros(rc, np.float32)
    with np.errstate(invalid="ignore"):
        amax[run.real] = np.where(np.isnan(f).any(axis=1), np.float32(np.nan), np.abs(f).max(axis=1))
    run.view("amax2", rc, torch.int32).copy_(torch.from_numpy(amax.view(np.int32)).cuda())
    assert M.nvfp4_get_device_error() == 0
    M.moe_requant_nvfp4(run.w, c.T, c.k, run.offs, run.ws)
    assert M.nvfp4_get_device_error() == 6            # NVFP4_ERR_NONFINITE

    a2c = run.view("a2_codes", rc * I // 2, torch.uint8).cpu().numpy().reshape(rc, I // 2)
    a2s = M.sf_to_rows(run.view("a2_sf", rc * I // 16, torch.uint8).cpu().numpy(), rc, I)
    a2g = run.view("a2_g", rc, torch.float32).cpu().numpy()
    good = np.array([i for i in range(n) if i not in bad])
    hc, hs, hg = Q.quantize_rows(f[good])
    rows = run.real[good]
    assert np.array_equal(a2c[rows], Q.pack_nibbles(hc))
    assert np.array_equal(a2s[rows], hs)
    assert np.array_equal(a2g[rows].view(np.uint32), hg.view(np.uint32))
    for row in bad:
        r = run.real[row]
        assert not a2c[r].any() and not a2s[r].any() and a2g[r] == 0
    pads = np.nonzero(run.pair[:run.off_np[-1]] < 0)[0]
    assert len(pads) and not a2s[pads].any() and not a2g[pads].any()


def test_combine_stage(run):
    """The combine reads token t's slot s from the routed row the route sort recorded for
    (t, s); a seeded y is placed at those rows (every other row holds NaN, which must not
    leak into the output)."""
    c = run.cfg
    rc = run.lay.rows_cap
    rng = np.random.default_rng(c.T + 1)
    y = S.f32_to_bf16_bits(rng.standard_normal((c.T, c.k, c.H)).astype(np.float32)
                           * np.exp2(rng.uniform(-20, 20, (c.T, c.k, 1))).astype(np.float32))
    pair_row = run.view("pair_row", c.T * c.k, torch.int32).cpu().numpy()
    assert np.array_equal(pair_row[run.pair[run.real]], run.real)      # the inverse of the row map
    full = np.full((rc, c.H), 0x7FC0, np.uint16)
    full[pair_row] = y.reshape(c.T * c.k, c.H)
    run.view("y", rc * c.H, torch.int16).copy_(torch.from_numpy(full.view(np.int16).ravel()).cuda())
    out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
    M.moe_combine_bf16(run.w, c.T, c.k, out, run.ws)
    assert np.array_equal(torch_to_bf16_bits(out), OM.combine_slots(y))
