"""Number formats of the NVFP4 recipe: BF16, E2M1 and (unsigned) E4M3.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: page "miniTE diagnoses and narrows the cross-engine execution gap of
NVFP4 RL" (onedev.kr/papers/1404), section "How it differs": E2M1 element
codes, E4M3 block scales, round-to-nearest-even, no stochastic rounding.  The
formats themselves are the standard OCP / NVIDIA ones:

* E2M1: sign bit (bit 3) and magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} for
  nibbles 0..7.  No infinity, no NaN.
* E4M3 (used unsigned for scales): exponent bias 7, 3 mantissa bits,
  subnormals m * 2^-9, largest finite 448 = 0x7E.
* BF16: the upper half of an IEEE binary32.

Every encoder here rounds to the nearest representable value and breaks an
exact tie towards the even code, which for these formats is the code whose
mantissa LSB is 0.  Values beyond the largest magnitude saturate to it.

Parity: pinned (tests/test_oracle_formats.py) by exhaustive brute force over
the grids, by the hand values of the contract, and against torch's own
float8_e4m3fn / bfloat16 casts where those apply.
"""

import numpy as np

# Nibble i (i = 0..7) is the magnitude E2M1_VALUES[i]; bit 3 is the sign.
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _e4m3_values():
    """All 127 finite non-negative E4M3 values, indexed by their code 0x00..0x7E."""
    vals = np.empty(127, dtype=np.float64)
    for code in range(127):
        exp_field = code >> 3
        man_field = code & 7
        if exp_field == 0:
            vals[code] = man_field * 2.0 ** -9          # subnormal: 0.mmm * 2^(1-7)
        else:
            vals[code] = (8 + man_field) * 2.0 ** (exp_field - 10)  # 1.mmm * 2^(e-7)
    return vals


E4M3_VALUES = _e4m3_values()
E4M3_MAX = 448.0


def _round_to_grid_even(a, grid):
    """Index of the grid value nearest to each a >= 0; exact ties go to the even index.

    ``grid`` is ascending and the index is the code, so "even index" is
    "even code".  a >= grid[-1] saturates to the last index.  All comparisons
    are exact in float64 (a is a binary32 value, the grid and its midpoints are
    short dyadic numbers).
    """
    a = np.asarray(a, dtype=np.float64)
    n = len(grid)
    hi = np.searchsorted(grid, a, side="right")          # grid[hi-1] <= a < grid[hi]
    hi = np.clip(hi, 1, n - 1)
    lo = hi - 1
    mid = (grid[lo] + grid[hi]) * 0.5
    idx = np.where(a > mid, hi, lo)
    tie = a == mid
    idx = np.where(tie, np.where(lo % 2 == 0, lo, hi), idx)
    idx = np.where(a >= grid[-1], n - 1, idx)
    return idx.astype(np.uint8)


def e2m1_encode(y):
    """E2M1 nibble of each binary32 value y: |y| rounded RNE and saturated, sign in bit 3.

    The sign bit is copied from y, so -0.0 and small negatives give nibble 8.
    """
    y = np.asarray(y, dtype=np.float32)
    mag = _round_to_grid_even(np.abs(y), E2M1_VALUES)
    sign = np.signbit(y).astype(np.uint8)
    return (mag | (sign << 3)).astype(np.uint8)


def e2m1_decode(nib):
    """Value of each E2M1 nibble (float64, exact)."""
    nib = np.asarray(nib, dtype=np.uint8)
    mag = E2M1_VALUES[nib & 7]
    return np.where(nib & 8, -mag, mag)


def e4m3_encode(r):
    """Unsigned E4M3 code of each r >= 0 (binary32): RNE, saturating at 448, never NaN."""
    r = np.asarray(r, dtype=np.float32)
    if np.any(r < 0) or np.any(np.isnan(r)):
        raise ValueError("e4m3_encode: scales are non-negative and finite")
    return _round_to_grid_even(r, E4M3_VALUES)


def e4m3_decode(code):
    """Value of each unsigned E4M3 code 0..126 (float64, exact)."""
    code = np.asarray(code, dtype=np.uint8)
    if np.any(code > 126):
        raise ValueError("e4m3_decode: code outside the finite unsigned range")
    return E4M3_VALUES[code]


def bf16_bits_to_f32(bits):
    """BF16 bit patterns (uint16) -> their exact binary32 values."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def round_to_bf16_bits(x):
    """Round each value (float64 or float32, taken exactly) to BF16 once, RNE.

    BF16 keeps 8 significant bits; the spacing of values in [2^(e-1), 2^e) is
    2^(e-8), and below the smallest normal 2^-126 it is 2^-133.  Overflow gives
    +-inf, as an IEEE rounding does.  Returns uint16 bit patterns.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.any(np.isnan(x)):
        raise ValueError("round_to_bf16_bits: NaN input")
    sign = np.signbit(x)
    a = np.abs(x)
    _, e = np.frexp(a)                      # a = m * 2^e, 0.5 <= m < 1
    qexp = np.maximum(e - 8, -133)          # exponent of one unit in the last place
    r = np.round(np.ldexp(a, -qexp))        # numpy rounds half to even
    val = np.ldexp(r, qexp)                 # exact: at most 9 significant bits
    with np.errstate(over="ignore"):
        f32 = val.astype(np.float32)        # exact unless it overflows to inf
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    return bits | (sign.astype(np.uint16) << 15)
