"""moe_route_sort_amax_noalloc against moe_route_sort_amax.

Some callers cannot hand the library scratch memory: their device memory is
planned once at start-up (a serving engine that assigns every byte up front,
an embedded runtime with no allocator), or their hot path must not call
cudaMalloc because it can synchronise the device.  For them the route sort has
a variant whose scratch sits in a fixed array inside the library; the caller
passes only inputs and the routed-row outputs.  Here both entry points are
called through the C ABI on the same inputs, two calls in a row on different
shapes (so the second call runs on the array the first one left behind), and
every output must be bit-identical, the tolerance of the route-sort tests.
This file is collected last on purpose."""

import ctypes

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


def _outputs(buf, offs, lay, H):
    """Expert offsets, every routed-row output below expert_offsets[E] and the row of every
    (token, slot)."""
    o = offs.cpu().numpy()
    n = int(o[-1])
    b = buf.cpu().numpy()

    def rows(off, width):
        return b[off:off + n * width]

    pair = rows(lay.row_pair, 4).view(np.int32)
    # codes of pad rows are unspecified (their scales are zero); compare real rows
    codes = rows(lay.a_codes, H // 2).reshape(n, H // 2)[pair >= 0]
    return {
        "offsets": o,
        "codes": codes,
        "g": rows(lay.a_g, 4),
        "pair": rows(lay.row_pair, 4),
        "prob": rows(lay.row_prob, 4),
        "amax2": rows(lay.amax2, 4),
        "sf": b[lay.a_sf:lay.a_sf + n * H // 16],
        "pair_row": b[lay.pair_row:lay.pair_row + 4 * lay.T * lay.k],
    }


def _one_shape(cfg, seed_stream):
    x = bf16_to_torch(S.make_x(cfg, stream=seed_stream))
    ids_np, w_np = S.make_routing(cfg, stream=seed_stream)
    ids, w = torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda()
    lay = M.moe_workspace_layout_query(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    lib = M.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ws = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    offs_a = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    st = lib.moe_route_sort_amax(ctypes.c_void_p(x.data_ptr()), cfg.T, cfg.H, cfg.E, cfg.k,
                                 ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                 ctypes.c_void_p(offs_a.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                 ws.numel(), stream)
    assert st == 0

    # the variant gets only the routed-row outputs, filled with junk beforehand
    out = torch.full((lay.chunk_count,), 0xA5, dtype=torch.uint8, device="cuda")
    offs_b = torch.full((cfg.E + 1,), -3, dtype=torch.int32, device="cuda")
    st = lib.moe_route_sort_amax_noalloc(ctypes.c_void_p(x.data_ptr()), cfg.T, cfg.H, cfg.E, cfg.k,
                                         ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                         ctypes.c_void_p(offs_b.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                         out.numel(), stream)
    assert st == 0
    assert M.nvfp4_get_device_error() == 0
    a = _outputs(ws, offs_a, lay, cfg.H)
    b = _outputs(out, offs_b, lay, cfg.H)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_noalloc_matches_route_sort_two_calls_in_a_row():
    _one_shape(S.LayerConfig("first", H=2048, I=768, E=128, k=8, T=3000, routing="zipf", outlier_frac=0.01), 1)
    _one_shape(S.LayerConfig("second", H=1024, I=384, E=16, k=4, T=777), 2)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = M.lib()
    p = ctypes.c_void_p(1 << 20)
    # 8*E*ceil(T/256) + 4*T*k + 4*E > 2 MiB: rejected on the host, nothing launched
    assert lib.moe_route_sort_amax_noalloc(p, 60000, 2048, 128, 8, p, p, p, p, 1 << 40, None) == 2
