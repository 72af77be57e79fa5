"""The SiLU table the FC1 epilogue compiles in, and the oracle's SiLU, at every BF16 input.

The library's table (nvfp4_moe_expert_gb300/silu_table.py) is computed exactly: 60
significant digits, then one rounding to the nearest binary32.  The oracle evaluates
a / (1 + exp(-a)) in FP64 and rounds once to FP32 (oracle.moe.silu_f32).  Both readings of
"SiLU rounded once" ("Finishing RL training faster: bitwise consistency, high performance,
agent-driven", section 4.4) must give the same bits at all 65,536 BF16 gate values, or the
FC1 epilogue and the oracle would disagree on h for the gates where they differ.  The exact
table is also a pin of the oracle's SiLU against the mathematics (not a restatement of it)."""

import math
from fractions import Fraction

import numpy as np
import pytest

from nvfp4_moe_expert_gb300 import silu_table as ST
from oracle import moe as OM


@pytest.fixture(scope="module")
def table():
    return np.array(ST.table(), dtype=np.uint32)


def test_table_equals_oracle_silu_everywhere(table):
    ref = OM.silu_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16)).view(np.uint32)
    nan_t = np.isnan(table.view(np.float32))
    nan_r = np.isnan(ref.view(np.float32))
    assert np.array_equal(nan_t, nan_r)
    assert nan_t.sum() == 255          # 254 BF16 NaN patterns and -inf
    bad = np.nonzero(table[~nan_t] != ref[~nan_t])[0]
    assert len(bad) == 0, [hex(int(i)) for i in np.nonzero(~nan_t)[0][bad][:10]]


def _f32(bits):
    return np.uint32(bits).view(np.float32)


def test_table_special_values(table):
    assert table[0x0000] == 0x00000000 and table[0x8000] == 0x80000000          # +-0
    assert table[0x7F80] == 0x7F800000                                          # +inf
    assert np.isnan(_f32(table[0xFF80]))                                        # -inf
    assert _f32(table[0x3F80]) == np.float32(1.0 / (1.0 + math.exp(-1.0)))      # silu(1)
    # far right: silu(a) rounds to a; far left: to -0
    assert table[0x4380] == 0x43800000          # a = 256
    assert table[0xC380] == 0x80000000          # a = -256
    # silu is odd-symmetric around a/2: silu(a) - silu(-a) = a
    for b in (0x3C00, 0x3E80, 0x4000, 0x40A0):
        a = float(_f32(b << 16))
        assert abs(float(_f32(table[b])) - float(_f32(table[b | 0x8000])) - a) <= 4 * abs(a) * 2.0 ** -24


def _rounded_exactly(v):
    """Nearest binary32 (ties to even) of a positive Fraction v in the normal range."""
    e = math.floor(math.log2(v.numerator) - math.log2(v.denominator))
    while Fraction(2) ** e > v:
        e -= 1
    while Fraction(2) ** (e + 1) <= v:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    n = math.floor(v / ulp)
    r = v / ulp - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2):
        n += 1
    return np.float32(float(n * ulp))


def test_rounding_against_rational_bounds(table):
    """For a sample of gates, the table entry is the binary32 value nearest to silu(a),
    checked with exact rational arithmetic on guaranteed bounds of e^-a (partial sums of
    its series with a remainder bound), independent of the generator's decimal code."""
    rng = np.random.default_rng(0)
    picks = rng.choice(np.arange(0x3C00, 0x4100), 40, replace=False)   # |a| in [2^-7, 8)
    picks = np.concatenate([picks, picks | 0x8000])
    for b in picks:
        a = Fraction(float(_f32(int(b) << 16)))
        x = -a
        # e^x = sum_{n<N} x^n/n! + R with |R| <= |x|^N/N! * e^|x| <= |x|^N/N! * 3^ceil|x|
        N = 60
        term, s = Fraction(1), Fraction(0)
        for n in range(N):
            s += term
            term = term * x / (n + 1)
        bound = abs(term) * Fraction(3) ** math.ceil(abs(x))
        lo_e, hi_e = s - bound, s + bound
        # silu(a) = a / (1 + e^-a) is monotone in e^-a; take both ends
        ends = [a / (1 + lo_e), a / (1 + hi_e)]
        got = np.float32(_f32(table[b]))
        want = {_rounded_exactly(abs(v)) for v in ends}
        assert len(want) == 1, "bounds straddle a rounding point; raise N"
        assert abs(got) == want.pop() and (got < 0) == (a < 0)
