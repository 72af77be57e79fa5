"""GPU parity of moe_route_sort_amax against the oracle: padded expert offsets,
the stable (token, slot) order inside each expert, pad rows, and the quantised
rows (codes, scales, g^x) bit-exact; index work compared exactly."""

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import formats as F
from oracle import moe as OM
from oracle import quant as Q
from _helpers import bf16_to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def ws_view(ws, off, n, dtype):
    nbytes = n * torch.empty(0, dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def run_route(x_bits, ids, probs, E, I=128):
    T, H = x_bits.shape
    k = ids.shape[1]
    ws = M.alloc_workspace(T, H, I, E, k)
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    M.moe_route_sort_amax(bf16_to_torch(x_bits), torch.from_numpy(ids).cuda(),
                          torch.from_numpy(probs).cuda(), E, offs, ws)
    assert M.nvfp4_get_device_error() == 0
    L = M.moe_workspace_layout_query(T, H, I, E, k)
    rc = L.rows_cap
    out = dict(
        L=L, offs=offs.cpu().numpy(),
        codes=ws_view(ws, L.a_codes, rc * H // 2, torch.uint8).cpu().numpy().reshape(rc, H // 2),
        sf=ws_view(ws, L.a_sf, rc * H // 16, torch.uint8).cpu().numpy(),
        g=ws_view(ws, L.a_g, rc, torch.float32).cpu().numpy(),
        pair=ws_view(ws, L.row_pair, rc, torch.int32).cpu().numpy(),
        prob=ws_view(ws, L.row_prob, rc, torch.float32).cpu().numpy(),
        amax2=ws_view(ws, L.amax2, rc, torch.int32).cpu().numpy(),
        pair_row=ws_view(ws, L.pair_row, T * k, torch.int32).cpu().numpy(),
    )
    return out


def check_route(x_bits, ids, probs, E):
    T, H = x_bits.shape
    k = ids.shape[1]
    r = run_route(x_bits, ids, probs, E)
    counts, uoff, order = OM.route_sort(ids, E)
    padded = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    assert np.array_equal(r["offs"], padded), "expert offsets"
    total = padded[-1]
    assert total <= r["L"].rows_cap
    xc, xs, xg = Q.quantize_rows(F.bf16_bits_to_f32(x_bits))
    xp = Q.pack_nibbles(xc)
    sf_rows = M.sf_to_rows(r["sf"], r["L"].rows_cap, H)
    for e in range(E):
        rows = np.arange(padded[e], padded[e] + counts[e])
        pads = np.arange(padded[e] + counts[e], padded[e + 1])
        want_pairs = order[uoff[e]:uoff[e + 1]]
        assert np.array_equal(r["pair"][rows], want_pairs), f"pair order of expert {e}"
        toks, slots = want_pairs // k, want_pairs % k
        assert np.array_equal(r["codes"][rows], xp[toks]), f"codes of expert {e}"
        assert np.array_equal(sf_rows[rows], xs[toks]), f"scales of expert {e}"
        assert np.array_equal(r["g"][rows].view(np.uint32), xg[toks].view(np.uint32))
        assert np.array_equal(r["prob"][rows], probs[toks, slots])
        assert not r["amax2"][rows].any()
        assert np.all(r["pair"][pads] == -1) and not r["g"][pads].any() and not r["prob"][pads].any()
        assert not sf_rows[pads].any() and not r["amax2"][pads].any()
        # each (token, slot) knows its row: the inverse of the row map
        assert np.array_equal(r["pair_row"][want_pairs], rows), f"pair rows of expert {e}"


@pytest.mark.parametrize("name,T,H,E,k,routing", [
    ("tiny", 64, 256, 8, 2, "uniform"),
    ("ragged", 1000, 2048, 128, 8, "uniform"),
    ("one_token", 1, 2048, 128, 8, "uniform"),
    ("skew", 1500, 2048, 128, 8, "zipf"),
    ("wide", 513, 4096, 16, 4, "zipf"),
    ("single_expert", 300, 256, 1, 1, "uniform"),
])
def test_route_sort_quant_bit_exact(name, T, H, E, k, routing):
    cfg = S.LayerConfig(name, H=H, I=128, E=E, k=k, T=T, routing=routing,
                        outlier_frac=0.01 if routing == "zipf" else 0.0)
    x = S.make_x(cfg)
    ids, probs = S.make_routing(cfg)
    check_route(x, ids, probs, E)


def test_route_qwen3_30b_a3b_full_size():
    cfg = S.CONFIGS["qwen3_30b_a3b"]
    x = S.make_x(cfg)
    ids, probs = S.make_routing(cfg)
    check_route(x, ids, probs, cfg.E)


def test_route_empty_batch():
    E = 8
    ws = M.alloc_workspace(0, 256, 128, E, 2)
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    M.moe_route_sort_amax(x, ids, w, E, offs, ws)
    assert not offs.cpu().numpy().any()


def test_bad_expert_id_flagged():
    cfg = S.LayerConfig("bad", H=256, I=128, E=8, k=2, T=40)
    x = S.make_x(cfg)
    ids, probs = S.make_routing(cfg)
    ids[7, 1] = 8                     # out of range: the kernel skips the pair and records the error
    ws = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    offs = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    assert M.nvfp4_get_device_error() == 0
    M.moe_route_sort_amax(bf16_to_torch(x), torch.from_numpy(ids).cuda(), torch.from_numpy(probs).cuda(),
                          cfg.E, offs, ws)
    assert M.nvfp4_get_device_error() == 5
    assert offs.cpu().numpy()[-1] <= M.moe_workspace_layout_query(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k).rows_cap
