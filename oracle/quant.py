"""Two-level NVFP4 row quantiser (E2M1 codes, E4M3 block scales, FP32 outer scale).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: page "miniTE diagnoses and narrows the cross-engine execution gap of
NVFP4 RL" (onedev.kr/papers/1404), section "How it differs": each row (a
token's activation row, or a weight row along the reduction dimension) gets an
FP32 outer scale g = max|row| / (6*448), blocks of 16 elements get an E4M3
scale, elements get E2M1 codes; rounding is round-to-nearest-even; no Hadamard
transform, no stochastic rounding.

The page gives the outer scale but not how the block scale is derived from it
nor the FP32 operation order.  Readings taken:

1. block scale  s_b = e4m3( bmax / (g * 6) )  with bmax = max|x| over the block:
   the largest code magnitude 6 times s_b times g reaches bmax, and since
   bmax <= amax = 2688*g, s_b <= 448 always;
2. element code q = e2m1( x / (g * s_b) );
3. both divisions are done in the two-step form written above, in IEEE
   binary32: first the product d = g*c (rounded), then x/d (rounded);
4. g == 0 (an all-zero row) gives all-zero codes and scales; a block whose
   divisor g*s_b is 0 (its scale rounded to 0, or the product underflowed)
   gets all-zero codes (nibble 0);
5. otherwise the sign bit of each code is copied from x (so tiny negatives
   become nibble 8, "-0");
6. packing: element 2j is the low nibble of byte j.

Parity: pinned (tests/test_oracle_quant.py) by hand values (E2M1 grid points
round-trip; a row with amax = 2688*g maps to magnitude 6 with block scale
448), by the per-element error bound, by exact power-of-two scaling
invariance and by a scalar pure-Python restatement on small rows.
"""

import numpy as np

from .formats import e2m1_encode, e4m3_encode, e4m3_decode, e2m1_decode

BLOCK = 16
# 6 * 448: the largest E2M1 magnitude times the largest E4M3 scale.
OUTER_DIVISOR = np.float32(2688.0)


def quantize_rows(x, amax=None):
    """Quantise each row of ``x`` ([rows, C] binary32 values, C % 16 == 0).

    ``amax`` optionally supplies max|row| (it must equal it; the FC2 input
    takes it from the activation's producer, which computed the same maximum).

    Returns (codes, scales, g):
      codes  uint8 [rows, C]      one E2M1 nibble per element (unpacked)
      scales uint8 [rows, C//16]  E4M3 code per 16-element block
      g      float32 [rows]       outer scale
    """
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % BLOCK:
        raise ValueError("quantize_rows: need [rows, C] with C a multiple of 16")
    if not np.all(np.isfinite(x)):
        raise ValueError("quantize_rows: non-finite input")
    rows, cols = x.shape
    nblk = cols // BLOCK
    ax = np.abs(x)
    row_max = ax.max(axis=1) if cols else np.zeros(rows, np.float32)
    if amax is None:
        amax = row_max
    else:
        amax = np.asarray(amax, dtype=np.float32)
        if not np.array_equal(amax, row_max):
            raise ValueError("quantize_rows: supplied amax differs from max|row|")

    g = (amax / OUTER_DIVISOR).astype(np.float32)                 # FP32 divide

    xb = x.reshape(rows, nblk, BLOCK)
    bmax = np.abs(xb).max(axis=2)                                  # [rows, nblk]
    d1 = (g * np.float32(6.0)).astype(np.float32)                  # g*6, rounded
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d1[:, None] > 0, bmax / d1[:, None], np.float32(0)).astype(np.float32)
    scales = e4m3_encode(r)
    s_val = e4m3_decode(scales).astype(np.float32)                 # exact
    d2 = (g[:, None] * s_val).astype(np.float32)                   # g*s_b, rounded
    live = d2 > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(live[:, :, None], xb / np.where(live, d2, 1)[:, :, None],
                     np.float32(0)).astype(np.float32)
    codes = e2m1_encode(y)
    codes = np.where(live[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    zero_row = g == 0
    scales = np.where(zero_row[:, None], np.uint8(0), scales).astype(np.uint8)
    return codes.reshape(rows, cols), scales, g


def dequantize_rows(codes, scales, g=None):
    """Float64 value q * s_b (* g if given) of each element; exact."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    q = e2m1_decode(codes).reshape(rows, cols // BLOCK, BLOCK)
    s = e4m3_decode(scales)[:, :, None]
    v = (q * s).reshape(rows, cols)
    if g is not None:
        v = v * np.asarray(g, dtype=np.float64)[:, None]
    return v


def pack_nibbles(codes):
    """[rows, C] nibbles -> [rows, C/2] bytes; element 2j is the low nibble of byte j."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = codes[:, 0::2] & 0xF
    hi = codes[:, 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    """Inverse of pack_nibbles."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    out = np.empty((rows, 2 * half), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out
