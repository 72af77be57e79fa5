"""Stage-by-stage parity at the large shapes the throughput workloads run, on the routed rows
of a sample of experts (the heaviest ones, the lightest non-empty one and a few others):

* ``large_t1024``: the large layer's shape (hidden 4096, expert intermediate 1536, 128 experts,
  top-8, Zipf-skewed routing, 1% x20 outlier channels, weights N(0, 0.015)) with 1024 tokens:
  FC1 walks K = 4096 in 16 stages over 12 n-tiles, FC2 K = 1536;
* ``qwen3_30b_a3b_skew``: the full 16384-token skewed workload of the 2048/768/128/top-8 layer.

Each stage is checked against the oracle at the tolerances of the method ("miniTE diagnoses
and narrows the cross-engine execution gap of NVFP4 RL", sections "How it differs" and "How
to use it"; "Finishing RL training faster...", section 4.4): the routed rows' codes, scales
and outer scales bit-exact; FC1 given those rows pre-cast within relative L2 1e-5 of the exact
FP64 values and within 1 BF16 ulp after the cast; SwiGLU x prob bit-exact where gate and up
agree and within the propagated bound elsewhere; the FC2 maxima equal max|h|; the
requantisation of the GPU's h bit-exact; FC2 given those codes within 1e-5 / 1 ulp; the
combine bit-exact on the GPU's own y; and the whole chain from X, per (token, slot) row of
the sampled experts, within relative L2 1e-2 with FC2 code flips <= 0.1%."""

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import formats as F
from oracle import moe as OM
from oracle import quant as Q
from _helpers import (FC2_CODE_FLIP_RATE, GEMM_BF16_ULP, GEMM_REL_L2, LAYER_REL_L2, bf16_to_torch,
                      bf16_ulp_distance, h_bound, rel_l2, torch_to_bf16_bits)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CASES = [
    S.LayerConfig("large_t1024", H=4096, I=1536, E=128, k=8, T=1024, routing="zipf", outlier_frac=0.01,
                  w_std=0.015),
    S.CONFIGS["qwen3_30b_a3b_skew"],
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def _rows(ws, off, n_rows, row_bytes, idx):
    """Rows idx (numpy int64, on the host) of a [n_rows][row_bytes] byte matrix in the workspace."""
    v = ws[off:off + n_rows * row_bytes].view(n_rows, row_bytes)
    return v[torch.from_numpy(idx).cuda()].cpu().numpy()


def _sf_rows(ws, off, n_rows, cols, idx):
    """Block scales [len(idx), cols/16] of rows idx from the library's scale-factor layout."""
    sf = ws[off:off + M.nvfp4_sf_bytes(n_rows, cols)]
    r = np.asarray(idx, np.int64)[:, None]
    b = np.arange(cols // 16, dtype=np.int64)[None, :]
    bidx = ((r >> 7) * (cols >> 6) + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)
    return sf[torch.from_numpy(bidx.ravel()).cuda()].cpu().numpy().reshape(bidx.shape)


class Big:
    def __init__(self, cfg):
        self.cfg = c = cfg
        self.L = L = S.make_layer(cfg)
        w1, w2 = bf16_to_torch(L["w1"]), bf16_to_torch(L["w2"])
        self.w = M.quantize_moe_weights(w1, w2)
        del w1, w2
        self.wq = OM.quantize_weights(L["w1"], L["w2"])
        self.ws = M.alloc_workspace(c.T, c.H, c.I, c.E, c.k)
        self.lay = lay = M.moe_workspace_layout_query(c.T, c.H, c.I, c.E, c.k)
        self.offs = torch.empty(c.E + 1, dtype=torch.int32, device="cuda")
        M.moe_route_sort_amax(bf16_to_torch(L["x"]), torch.from_numpy(L["topk_ids"]).cuda(),
                              torch.from_numpy(L["topk_w"]).cuda(), c.E, self.offs, self.ws)
        rc = lay.rows_cap
        self.fc1_dbg = torch.zeros((rc, 2 * c.I), dtype=torch.float32, device="cuda")
        self.fc2_dbg = torch.zeros((rc, c.H), dtype=torch.float32, device="cuda")
        M.moe_fc1_swiglu_nvfp4(self.w, c.T, c.k, self.offs, self.ws, debug=self.fc1_dbg)
        M.moe_requant_nvfp4(self.w, c.T, c.k, self.offs, self.ws)
        M.moe_fc2_nvfp4(self.w, c.T, c.k, self.offs, self.ws, debug=self.fc2_dbg)
        self.out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
        M.moe_combine_bf16(self.w, c.T, c.k, self.out, self.ws)
        assert M.nvfp4_get_device_error() == 0
        self.off_np = self.offs.cpu().numpy()
        pair = self.ws[lay.row_pair:lay.row_pair + 4 * rc].view(torch.int32).cpu().numpy()
        pair[self.off_np[-1]:] = -1
        self.pair = pair
        counts = np.bincount(L["topk_ids"].ravel(), minlength=c.E)
        order = np.argsort(-counts, kind="stable")
        nonempty = order[counts[order] > 0]
        rng = np.random.default_rng(c.T)
        pick = list(nonempty[:3]) + [nonempty[-1]] + list(rng.choice(nonempty[3:-1], 4, replace=False))
        self.experts = sorted(set(int(e) for e in pick))
        assert len(self.experts) >= 8 and int(order[0]) in self.experts

    def expert_rows(self, e):
        """Routed rows of expert e (pad rows excluded), in row order, and their (token, slot)."""
        r = np.arange(self.off_np[e], self.off_np[e + 1])
        r = r[self.pair[r] >= 0]
        p = self.pair[r]
        return r, p // self.cfg.k, p % self.cfg.k


@pytest.fixture(scope="module", params=CASES, ids=lambda c: c.name)
def big(request):
    b = Big(request.param)
    yield b
    del b
    torch.cuda.empty_cache()


def test_route_rows_bit_exact(big):
    c, lay = big.cfg, big.lay
    xq = Q.quantize_rows(F.bf16_bits_to_f32(big.L["x"]))
    rc = lay.rows_cap
    for e in big.experts:
        r, t, _ = big.expert_rows(e)
        assert len(r) == np.count_nonzero(big.L["topk_ids"] == e)
        codes = _rows(big.ws, lay.a_codes, rc, c.H // 2, r)
        assert np.array_equal(codes, Q.pack_nibbles(xq[0][t]))
        assert np.array_equal(_sf_rows(big.ws, lay.a_sf, rc, c.H, r), xq[1][t])
        g = big.ws[lay.a_g:lay.a_g + 4 * rc].view(torch.float32).cpu().numpy()[r]
        assert np.array_equal(g.view(np.uint32), xq[2][t].view(np.uint32))


def test_fc1_and_swiglu(big):
    c, lay = big.cfg, big.lay
    rc = lay.rows_cap
    xq = Q.quantize_rows(F.bf16_bits_to_f32(big.L["x"]))
    f = F.bf16_bits_to_f32
    for e in big.experts:
        r, t, s = big.expert_rows(e)
        v_gpu = big.fc1_dbg[torch.from_numpy(r).cuda()].cpu().numpy()
        (c1, s1, g1), _ = big.wq.expert(e)
        v_ref = OM.epilogue_f64(OM.qgemm_f64(xq[0][t], xq[1][t], c1, s1), xq[2][t], g1)
        assert rel_l2(v_gpu, v_ref) <= GEMM_REL_L2, e
        gu_gpu, gu_ref = F.round_to_bf16_bits(v_gpu), F.round_to_bf16_bits(v_ref)
        assert bf16_ulp_distance(gu_gpu, gu_ref).max() <= GEMM_BF16_ULP, e
        h_gpu = _rows(big.ws, lay.h, rc, 2 * c.I, r).view(np.uint16)
        p = big.L["topk_w"][t, s]
        h_ref = OM.swiglu_prob(gu_ref[:, :c.I], gu_ref[:, c.I:], p)
        same = (gu_gpu[:, :c.I] == gu_ref[:, :c.I]) & (gu_gpu[:, c.I:] == gu_ref[:, c.I:])
        assert np.array_equal(h_gpu[same], h_ref[same]), e
        d = ~same
        pr = np.broadcast_to(p[:, None], same.shape)
        bound = h_bound(f(gu_gpu[:, :c.I])[d], f(gu_gpu[:, c.I:])[d], f(gu_ref[:, :c.I])[d], f(gu_ref[:, c.I:])[d],
                        pr[d], f(h_gpu)[d], f(h_ref)[d])
        assert (np.abs(f(h_gpu)[d].astype(np.float64) - f(h_ref)[d]) <= bound).all(), e
        amax2 = big.ws[lay.amax2:lay.amax2 + 4 * rc].view(torch.int32).cpu().numpy().view(np.uint32)[r]
        assert np.array_equal(amax2, np.abs(f(h_gpu)).max(axis=1).view(np.uint32)), e


def test_requant_and_fc2(big):
    c, lay = big.cfg, big.lay
    rc = lay.rows_cap
    y = big.ws[lay.y:lay.y + 2 * rc * c.H].view(torch.int16).view(rc, c.H)      # per routed row
    for e in big.experts:
        r, t, s = big.expert_rows(e)
        h_gpu = F.bf16_bits_to_f32(_rows(big.ws, lay.h, rc, 2 * c.I, r).view(np.uint16))
        hc, hs, hg = Q.quantize_rows(h_gpu, amax=np.abs(h_gpu).max(axis=1))
        assert np.array_equal(_rows(big.ws, lay.a2_codes, rc, c.I // 2, r), Q.pack_nibbles(hc)), e
        assert np.array_equal(_sf_rows(big.ws, lay.a2_sf, rc, c.I, r), hs), e
        g2 = big.ws[lay.a2_g:lay.a2_g + 4 * rc].view(torch.float32).cpu().numpy()[r]
        assert np.array_equal(g2.view(np.uint32), hg.view(np.uint32)), e
        v_gpu = big.fc2_dbg[torch.from_numpy(r).cuda()].cpu().numpy()
        _, (c2, s2, gw2) = big.wq.expert(e)
        v_ref = OM.epilogue_f64(OM.qgemm_f64(hc, hs, c2, s2), hg, gw2)
        assert rel_l2(v_gpu, v_ref) <= GEMM_REL_L2, e
        y_rows = y[torch.from_numpy(r).cuda()].cpu().numpy().view(np.uint16)
        assert np.array_equal(y_rows, F.round_to_bf16_bits(v_gpu)), e
        assert bf16_ulp_distance(y_rows, F.round_to_bf16_bits(v_ref)).max() <= GEMM_BF16_ULP, e


def test_combine_on_gpu_y(big):
    c, lay = big.cfg, big.lay
    toks = np.sort(np.random.default_rng(1).choice(c.T, 64, replace=False))
    rc = lay.rows_cap
    y = big.ws[lay.y:lay.y + 2 * rc * c.H].view(torch.int16).view(rc, c.H)
    pair_row = big.ws[lay.pair_row:lay.pair_row + 4 * c.T * c.k].view(torch.int32).view(c.T, c.k)
    rows_t = pair_row[torch.from_numpy(toks).cuda()]
    y_t = y[rows_t.reshape(-1)].view(len(toks), c.k, c.H).cpu().numpy().view(np.uint16)
    got = torch_to_bf16_bits(big.out)[toks]
    assert np.array_equal(got, OM.combine_slots(y_t))


def test_chain_from_x(big):
    """The oracle's whole chain (its own FC1, SwiGLU x prob, requantisation and FC2) on the
    sampled experts' (token, slot) rows against the GPU's per-slot outputs."""
    c, lay = big.cfg, big.lay
    rc = lay.rows_cap
    y = big.ws[lay.y:lay.y + 2 * rc * c.H].view(torch.int16).view(rc, c.H)
    flips = n = 0
    for e in big.experts:
        r, t, s = big.expert_rows(e)
        ids = np.full((len(t), 1), e, np.int32)
        _, inter = OM.moe_forward(big.L["x"][t], ids, big.L["topk_w"][t, s][:, None], big.wq, keep=True)
        y_rows = y[torch.from_numpy(r).cuda()].cpu().numpy().view(np.uint16)
        assert rel_l2(F.bf16_bits_to_f32(y_rows), F.bf16_bits_to_f32(inter["y"][:, 0])) <= LAYER_REL_L2, e
        gpu_codes = Q.unpack_nibbles(_rows(big.ws, lay.a2_codes, rc, c.I // 2, r))
        flips += int((gpu_codes != inter["hq"][0]).sum())
        n += gpu_codes.size
    assert flips / n <= FC2_CODE_FLIP_RATE, flips / n
