"""GPU parity of nvfp4_quantize_rows against the oracle: codes, block scales and
outer scales bit-exact, on seeded synthetic rows spanning several 128-row tiles
with a ragged tail, wide dynamic range, outliers and degenerate rows."""

import os

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import formats as F
from oracle import quant as Q
from _helpers import bf16_to_torch

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def gpu_quant(bits, ld=None):
    rows, cols = bits.shape
    if ld is None:
        x = bf16_to_torch(bits)
    else:
        full = np.zeros((rows, ld), np.uint16)
        full[:, :cols] = bits
        x = bf16_to_torch(full)[:, :cols]
    codes, sf, g = M.nvfp4_quantize_rows(x)
    assert M.nvfp4_get_device_error() == 0
    return codes.cpu().numpy(), sf.cpu().numpy(), g.cpu().numpy()


def oracle_quant(bits):
    c, s, g = Q.quantize_rows(F.bf16_bits_to_f32(bits))
    return Q.pack_nibbles(c), s, g


def synth_rows(rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x *= np.exp2(rng.uniform(-30, 30, (rows, 1))).astype(np.float32)      # row scales over 2^+-30
    ch = rng.choice(cols, max(1, cols // 100), replace=False)
    x[:, ch] *= 20                                                          # outlier channels
    if rows > 3:
        x[1] = 0.0                                                          # all-zero row
        x[2, :] = -0.0                                                      # negative zeros
        x[3, ::7] = 0.0
    if rows > 5:
        x[4] = 1e-38 * rng.standard_normal(cols)                            # BF16 subnormal range
        x[5, :16] = 0.0                                                     # a zero block
        x[5, 16:32] *= 1e-9                                                 # a block whose scale underflows
    return S.f32_to_bf16_bits(x)


def check_equal(bits, got):
    rows, cols = bits.shape
    gc, gs, gg = got
    oc, os_, og = oracle_quant(bits)
    assert np.array_equal(gc[:rows], oc), "codes differ"
    assert np.array_equal(M.sf_to_rows(gs, rows, cols), os_), "block scales differ"
    assert np.array_equal(gg.view(np.uint32), og.view(np.uint32)), "outer scales differ"
    rp = M.nvfp4_rows_padded(rows)
    assert not gc[rows:rp].any(), "pad rows must have zero codes"
    pad_idx = M.sf_byte_index(rp, cols)[rows:]
    assert not gs[pad_idx].any(), "pad rows must have zero scales"


@pytest.mark.parametrize("rows,cols", [(1, 64), (6, 128), (127, 256), (128, 2048), (300, 768),
                                       (130, 4096), (9, 8192), (257, 1536)])
def test_quantize_rows_bit_exact(rows, cols):
    bits = synth_rows(rows, cols, seed=rows * 131 + cols)
    check_equal(bits, gpu_quant(bits))


def test_quantize_rows_strided():
    bits = synth_rows(200, 512, seed=5)
    check_equal(bits, gpu_quant(bits, ld=640))


def test_golden_rows_on_gpu():
    rows = []
    for line in open(os.path.join(GOLDEN, "quant_rows.txt")):
        line = line.split("#")[0].strip()
        if line:
            rows.append([float(v) for v in line.split("|")[1].split()])
    x = np.zeros((len(rows), 64), np.float32)
    x[:, :32] = np.array(rows, np.float32)         # 32 more zero columns change nothing
    bits = S.f32_to_bf16_bits(x)
    check_equal(bits, gpu_quant(bits))


def test_weight_shapes_bit_exact():
    cfg = S.CONFIGS["qwen3_30b_a3b"]
    w1, w2 = S.make_weights(cfg, experts=2)
    for w in (w1.reshape(-1, cfg.H), w2.reshape(-1, cfg.I)):
        check_equal(w, gpu_quant(w))


def test_nonfinite_rows_flagged():
    bits = synth_rows(8, 128, seed=9)
    bits[3, 5] = 0x7F80                 # +inf
    x = bf16_to_torch(bits)
    assert M.nvfp4_get_device_error() == 0
    M.nvfp4_quantize_rows(x)
    assert M.nvfp4_get_device_error() == 6          # NVFP4_ERR_NONFINITE
    assert M.nvfp4_get_device_error() == 0          # cleared by the read
