"""Pins for the oracle's two-level NVFP4 row quantiser: hand-derived rows,
the per-element error bound, power-of-two scaling invariance and a scalar
restatement on small rows.  CPU only."""

import os
import struct

import numpy as np

from oracle import formats as F
from oracle import quant as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows():
    with open(os.path.join(GOLDEN, "quant_rows.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            name, xs, g, sc, codes = [p.strip() for p in line.split("|")]
            yield (name, np.array([float(v) for v in xs.split()], np.float32),
                   int(g, 16), [int(v, 16) for v in sc.split()], [int(v, 16) for v in codes.split()])


def test_golden_rows():
    n = 0
    for name, x, g_bits, scales, codes in _golden_rows():
        # inputs are BF16 values
        assert np.array_equal(F.bf16_bits_to_f32(F.round_to_bf16_bits(x)), x), name
        c, s, g = Q.quantize_rows(x[None, :])
        assert int(g.view(np.uint32)[0]) == g_bits, (name, hex(int(g.view(np.uint32)[0])))
        assert list(s[0]) == scales, (name, list(s[0]))
        assert list(c[0]) == codes, (name, list(c[0]))
        n += 1
    assert n == 6


def test_amax_maps_to_code6_scale448():
    # the hand test of the contract: amax = 6*448*g  ->  magnitude 6 (nibble 7), scale 448 (0x7E)
    for g_exp in (-12, -10, -3, 0, 4):
        amax = np.float32(2688.0 * 2.0 ** g_exp)
        rng = np.random.default_rng(g_exp + 20)
        x = (rng.uniform(-1, 1, 64) * amax * 0.9).astype(np.float32)
        x = F.bf16_bits_to_f32(F.round_to_bf16_bits(x))
        x[5] = -amax
        c, s, g = Q.quantize_rows(x[None, :])
        assert g[0] == np.float32(2.0 ** g_exp)
        assert s[0, 0] == 0x7E and c[0, 5] == 0xF


def test_grid_points_roundtrip():
    # every E2M1 magnitude times g*s dequantises back exactly, for several block scales
    g = np.float32(2.0 ** -10)
    for sc in (0x7E, 0x38, 0x44, 0x10, 0x01 + 0x20):
        s_val = F.E4M3_VALUES[sc]
        row = np.zeros(32, np.float32)
        row[0] = 2688.0 * float(g)                           # fixes g (block 0 scale 448)
        vals = np.array([6, 4, 3, 2, 1.5, 1, 0.5, 0, -0.5, -1, -1.5, -2, -3, -4, -6, 6.0])
        row[16:] = (vals * s_val * float(g)).astype(np.float32)
        c, s, gg = Q.quantize_rows(row[None, :])
        assert gg[0] == g and s[0, 1] == sc
        deq = Q.dequantize_rows(c, s, gg)[0, 16:]
        assert np.array_equal(deq, row[16:].astype(np.float64))


def test_zero_and_repeated_rows():
    c, s, g = Q.quantize_rows(np.zeros((3, 48), np.float32))
    assert not c.any() and not s.any() and not g.any()
    for v in (1.0, -7.5, 0.001, 300.0):
        c, s, g = Q.quantize_rows(np.full((1, 32), v, np.float32))
        assert np.all(s == 0x7E)
        assert np.all(c == (0xF if v < 0 else 0x7))


def _bf16_rows(rng, rows, cols, scale=1.0, outliers=False):
    x = rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(scale)
    if outliers:
        x[:, rng.choice(cols, max(1, cols // 100), replace=False)] *= 20
    return F.bf16_bits_to_f32(F.round_to_bf16_bits(x))


def test_error_bound():
    rng = np.random.default_rng(7)
    x = _bf16_rows(rng, 64, 256, outliers=True)
    c, s, g = Q.quantize_rows(x)
    deq = Q.dequantize_rows(c, s, g)
    sg = (F.e4m3_decode(s) * g.astype(np.float64)[:, None]).repeat(16, axis=1)
    y = x / sg                                   # exact-ish quotient in FP64
    mag = np.abs(F.e2m1_decode(c))
    gaps = np.diff(F.E2M1_VALUES)
    # half the gap to the neighbour on y's side
    idx = np.searchsorted(F.E2M1_VALUES, mag)
    half = np.where(np.abs(y) >= mag, np.append(gaps, 0)[idx], np.insert(gaps, 0, 0)[idx]) / 2
    err = np.abs(x - deq) / sg
    sat = np.abs(y) > 6
    assert np.all(err[~sat] <= half[~sat] * (1 + 1e-6) + 1e-6)
    # saturation only happens by at most the scale's rounding
    assert np.all(np.abs(y[sat]) <= 6 * (1 + 2.0 ** -3))


def test_power_of_two_scaling_invariance():
    rng = np.random.default_rng(8)
    x = _bf16_rows(rng, 16, 128)
    c0, s0, g0 = Q.quantize_rows(x)
    for n in (-20, -3, 1, 7, 30):
        c, s, g = Q.quantize_rows(x * np.float32(2.0 ** n))
        assert np.array_equal(c, c0) and np.array_equal(s, s0)
        assert np.array_equal(g, (g0 * np.float32(2.0 ** n)).astype(np.float32))


def test_row_independence():
    rng = np.random.default_rng(9)
    x = _bf16_rows(rng, 10, 64)
    c, s, g = Q.quantize_rows(x)
    perm = rng.permutation(10)
    c2, s2, g2 = Q.quantize_rows(x[perm])
    assert np.array_equal(c2, c[perm]) and np.array_equal(s2, s[perm]) and np.array_equal(g2, g[perm])


def _f32(v):
    return struct.unpack("f", struct.pack("f", v))[0]


def test_scalar_restatement_small_rows():
    # element-by-element restatement with Python floats rounded through struct
    rng = np.random.default_rng(10)
    x = _bf16_rows(rng, 6, 32, scale=0.3)
    c, s, g = Q.quantize_rows(x)
    grid = list(F.E2M1_VALUES)
    for r in range(x.shape[0]):
        row = [float(v) for v in x[r]]
        amax = max(abs(v) for v in row)
        gr = _f32(amax / 2688.0)
        assert gr == float(g[r])
        for b in range(2):
            blk = row[16 * b:16 * b + 16]
            rr = _f32(max(abs(v) for v in blk) / _f32(gr * 6.0))
            sv = float(F.E4M3_VALUES[int(s[r, b])])
            # the chosen scale is a nearest E4M3 value to rr
            dists = [abs(rr - e) for e in F.E4M3_VALUES]
            assert abs(rr - sv) == min(dists)
            d2 = _f32(gr * sv)
            for j, v in enumerate(blk):
                y = _f32(v / d2)
                m = int(c[r, 16 * b + j]) & 7
                dm = [abs(abs(y) - q) for q in grid]
                assert abs(abs(y) - grid[m]) == min(dm) or abs(y) > 6
                assert (int(c[r, 16 * b + j]) >> 3) == (1 if np.signbit(np.float32(v)) else 0)


def test_pack_unpack():
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    p = Q.pack_nibbles(codes)
    assert p.shape == (5, 32)
    assert p[0, 0] == (codes[0, 0] | (codes[0, 1] << 4))
    assert np.array_equal(Q.unpack_nibbles(p), codes)


def test_supplied_amax_must_match():
    x = np.ones((1, 16), np.float32)
    try:
        Q.quantize_rows(x, amax=np.array([2.0], np.float32))
    except ValueError:
        return
    raise AssertionError("mismatched amax accepted")
