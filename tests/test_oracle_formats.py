"""Pins for the oracle's number formats (BF16, E2M1, E4M3) against hand values,
exhaustive brute force and torch's independent casts.  CPU only."""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                yield line.split()


def _argmin_even(a, grid):
    """Brute force: nearest grid value by exhaustive distance, ties -> even index."""
    best = None
    for i, v in enumerate(grid):
        d = abs(Fraction(float(a)) - Fraction(float(v)))
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def test_e2m1_golden():
    for val, nib in _rows("e2m1_rne.txt"):
        got = int(F.e2m1_encode(np.float32(float(val))))
        assert got == int(nib), (val, got, nib)


def test_e4m3_golden():
    for val, code in _rows("e4m3_rne.txt"):
        got = int(F.e4m3_encode(np.float32(float(val))))
        assert got == int(code, 16), (val, hex(got), code)


def test_e2m1_bruteforce_dense():
    # every binary32 in [0, 8) on a fine stride plus the neighbours of every midpoint
    base = np.arange(0, 8, 1.0 / 4096, dtype=np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], dtype=np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(9))])
    ys = np.concatenate([base[::7], near])
    got = F.e2m1_encode(ys)
    for y, g in zip(ys, got):
        want = _argmin_even(y, F.E2M1_VALUES) if y <= 6 else 7
        assert g == want, (float(y), int(g), want)


def test_e2m1_roundtrip_and_sign():
    for nib in range(16):
        v = F.e2m1_decode(np.uint8(nib))
        enc = int(F.e2m1_encode(np.float32(v)))
        if nib == 8:                       # -0 decodes to -0.0 and re-encodes to 8
            assert enc == 8
        else:
            assert enc == nib


def test_e4m3_grid_properties():
    v = F.E4M3_VALUES
    assert len(v) == 127 and v[0] == 0 and v[1] == 2.0 ** -9 and v[0x7E] == 448.0
    assert np.all(np.diff(v) > 0)
    # every grid value round-trips
    assert np.array_equal(F.e4m3_encode(v.astype(np.float32)), np.arange(127, dtype=np.uint8))


def test_e4m3_bruteforce_vs_argmin():
    rng = np.random.default_rng(1)
    r = np.concatenate([
        rng.uniform(0, 500, 300).astype(np.float32),
        np.exp2(rng.uniform(-14, 9, 300)).astype(np.float32),
        ((F.E4M3_VALUES[:-1] + F.E4M3_VALUES[1:]) / 2).astype(np.float32),   # all midpoints
    ])
    got = F.e4m3_encode(r)
    for x, g in zip(r, got):
        want = _argmin_even(x, F.E4M3_VALUES) if x <= 448 else 0x7E
        assert g == want, (float(x), int(g), want)


def test_e4m3_vs_torch_float8():
    # torch's float8_e4m3fn cast is an independent RNE implementation; compare
    # inside the finite range where both agree on the definition.
    rng = np.random.default_rng(2)
    r = np.concatenate([
        np.exp2(rng.uniform(-12, 8.8, 20000)).astype(np.float32),
        ((F.E4M3_VALUES[:-1] + F.E4M3_VALUES[1:]) / 2).astype(np.float32),
    ])
    r = r[r <= 448]
    t = torch.from_numpy(r).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(r), t)


def test_bf16_from_f32_vs_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(50000).astype(np.float32) * np.float32(3.0),
        np.exp2(rng.uniform(-140, 120, 5000)).astype(np.float32),
        np.array([0.0, -0.0, 1.0, 65504.0, 3.0e38, -3.0e38, 1e-45], np.float32),
    ])
    t = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.round_to_bf16_bits(x), t)


def test_bf16_from_f64_single_rounding():
    # BF16 values near x: enumerate by exponent and compare exactly as rationals.
    rng = np.random.default_rng(4)
    xs = list(rng.standard_normal(300) * 10.0) + [1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40,
                                                  1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)]
    allvals = F.bf16_bits_to_f32(np.arange(0, 0x7F80, dtype=np.uint16)).astype(np.float64)
    for x in xs:
        a = abs(x)
        i = int(np.searchsorted(allvals, a))
        lo, hi = max(i - 1, 0), min(i, len(allvals) - 1)
        cands = [(abs(Fraction(a) - Fraction(float(allvals[j]))), j % 2, j) for j in {lo, hi}]
        cands.sort()
        d0 = cands[0][0]
        best = [c for c in cands if c[0] == d0]
        j = [c[2] for c in best if c[1] == 0][0] if len(best) > 1 else best[0][2]
        want = j | (0x8000 if x < 0 else 0)
        assert int(F.round_to_bf16_bits(np.float64(x))) == want, x
    assert int(F.round_to_bf16_bits(np.float64(1 + 2.0 ** -8))) == 0x3F80      # tie -> even
    assert int(F.round_to_bf16_bits(np.float64(1 + 2.0 ** -8 + 2.0 ** -40))) == 0x3F81


def test_bf16_bits_to_f32_exact():
    bits = np.arange(0, 0x7F80, 97, dtype=np.uint16)
    f = F.bf16_bits_to_f32(bits)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(f, t)


@pytest.mark.parametrize("bad", [-1.0, float("nan")])
def test_e4m3_rejects_negative_or_nan(bad):
    with pytest.raises(ValueError):
        F.e4m3_encode(np.float32(bad))
