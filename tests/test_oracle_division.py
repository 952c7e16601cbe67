"""Pins of the quantizer's division step (lpnh.cn DeepGEMM walkthrough §4.2
step 4: divide each element by the block's scale, then round to the nearest
E4M3 value, ties to even; §3.1: the scale is max_abs / 448 kept in FP32).

The reading is the IEEE binary32 quotient fl32(x / s). A quantizer that
multiplies by a rounded reciprocal, fl32(x * fl32(1 / s)), agrees with it on
almost every element but not on all: where x / s sits next to an E4M3 rounding
boundary the two land on different sides. These tests hold every quantizer of
the oracle (128x128, 1x128, and the requantized GEMM output, which runs them)
to the quotient:
* hand-derived cases (tests/golden/division_cases.json), re-derived here with
  exact rational arithmetic, each one shown to separate the two evaluations;
* a search over elements placed next to every E4M3 midpoint for random
  non-power-of-two scales, against numpy's IEEE float32 division followed by
  an encoder written in the tests, checked to contain separating elements.
"""
from fractions import Fraction

import numpy as np
import pytest

from conftest import load_golden
from test_oracle_e4m3 import quantum_encode

GOLD = load_golden("division_cases.json")


def _f32(hexbits):
    return np.array([int(hexbits, 16)], np.uint32).view(np.float32)[0]


def _e4m3_values():
    """Magnitudes of codes 0x00..0x7E from the OCP E4M3 layout, as exact fractions."""
    vals = []
    for c in range(0x7F):
        e, m = (c >> 3) & 0xF, c & 0x7
        vals.append(Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


_VALS = _e4m3_values()


def _exact_code(v):
    """E4M3 code of an FP32 value by exact comparison with the midpoints (ties to even, saturating)."""
    sign = 0x80 if np.signbit(v) else 0
    a = abs(Fraction(float(v)))
    if a >= 448:
        return sign | 0x7E
    lo = max(i for i in range(0x7F) if _VALS[i] <= a)
    mid = (_VALS[lo] + _VALS[lo + 1]) / 2
    code = lo if a < mid else lo + 1 if a > mid else (lo if lo % 2 == 0 else lo + 1)
    return sign | code


def _fl32(q):
    """Round an exact rational to the nearest FP32 value, ties to the even bit pattern.
    A first guess through float64 is at most one FP32 step off, so the answer is the
    guess or one of its two neighbours, whichever is exactly nearest."""
    f = np.float32(float(q))
    lo, hi = np.nextafter(f, np.float32(-np.inf)), np.nextafter(f, np.float32(np.inf))
    best = min((f, lo, hi), key=lambda c: (abs(Fraction(float(c)) - q), int(np.array(c).view(np.uint32)) & 1))
    return best


@pytest.mark.parametrize("case", GOLD["cases"], ids=lambda c: c["name"])
def test_fixture_is_consistent_and_separates_the_two_evaluations(case):
    amax, x, s = _f32(case["amax"]), _f32(case["x"]), _f32(case["scale"])
    assert s == np.float32(amax / np.float32(448.0))
    assert np.frexp(s)[0] != 0.5                                    # not a power of two
    quot = _fl32(Fraction(float(x)) / Fraction(float(s)))
    assert quot == _f32(case["quotient"]) == np.float32(x / s)
    recip = _fl32(1 / Fraction(float(s)))
    prod = _fl32(Fraction(float(x)) * Fraction(float(recip)))
    assert prod == _f32(case["reciprocal_product"])
    assert _exact_code(quot) == int(case["code"], 16)
    assert _exact_code(prod) == int(case["product_code"], 16)
    assert case["code"] != case["product_code"]


@pytest.mark.parametrize("case", GOLD["cases"], ids=lambda c: c["name"])
def test_quantizers_take_the_quotient(oracle_mod, case):
    amax, x = _f32(case["amax"]), _f32(case["x"])
    want = int(case["code"], 16)
    block = np.zeros((3, 200), np.float32)
    block[1, 7], block[1, 40] = amax, x
    q, s = oracle_mod.quantize(block, 0)
    assert s[0, 0] == _f32(case["scale"]) and q[1, 40] == want, case["derivation"]
    q1, s1 = oracle_mod.quantize_1x128(block, 0)
    assert s1[1, 0] == _f32(case["scale"]) and q1[1, 40] == want, case["derivation"]
    # The requantized GEMM output runs the same steps on the FP32 accumulator.
    for rows in (1, 128):
        qr, _ = oracle_mod.requantize_output(block.astype(np.float64), rows, 0)
        assert qr[1, 40] == want, (rows, case["derivation"])


def _near_midpoints(scales, rng):
    """For each scale s, one 128-element block row: the amax element 448 s' (s' chosen so
    that fl32(amax / 448) == s) and elements fl32(mid * s) +- 1 ulp for random E4M3
    midpoints mid."""
    mids = np.array([float((_VALS[i] + _VALS[i + 1]) / 2) for i in range(0x7E)])
    rows = []
    for s in scales:
        amax = np.float32(s * 448.0)
        sm = np.float32(amax / np.float32(448.0))
        pick = mids[rng.integers(0, len(mids), 127)]
        x0 = (pick * float(sm)).astype(np.float32)
        step = rng.integers(-1, 2, 127)
        x = np.where(step > 0, np.nextafter(x0, np.float32(np.inf)),
                     np.where(step < 0, np.nextafter(x0, np.float32(-np.inf)), x0)).astype(np.float32)
        x = np.minimum(x, amax) * np.where(rng.random(127) < 0.5, -1, 1).astype(np.float32)
        rows.append(np.concatenate([[amax], x]).astype(np.float32))
    return np.stack(rows)


def test_search_near_midpoints_matches_ieee_division(oracle_mod):
    rng = np.random.default_rng(41)
    scales = np.exp(rng.normal(-4.0, 3.0, 256)).astype(np.float32)
    x = _near_midpoints(scales, rng)                             # [256, 128]
    q1, s1 = oracle_mod.quantize_1x128(x, 0)
    want_s = (np.abs(x).max(axis=1) / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(s1[:, 0], want_s)
    quot = (x / want_s[:, None]).astype(np.float32)              # IEEE binary32 division
    want = quantum_encode(quot)
    assert np.array_equal(q1, want)
    # The same rows as 128x128 blocks: one block per row, each a full 128-row block of
    # that row repeated, so every block has the row's scale.
    blocks = np.repeat(x[:16], 128, axis=0)
    qb, sb = oracle_mod.quantize(blocks, 0)
    assert np.array_equal(sb[:, 0], want_s[:16])
    assert np.array_equal(qb[::128], want[:16])
    # The search is only a pin if it holds elements where the reciprocal product differs.
    recip = (np.float32(1.0) / want_s).astype(np.float32)
    prod = (x * recip[:, None]).astype(np.float32)
    assert np.count_nonzero(quantum_encode(prod) != want) >= 20
