"""Pins for the oracle's E4M3 decode table and its nearest-even encoder.

The oracle is checked against things it does not share code with:
* the OCP E4M3 closed form at named codes (1.0, 2.0, 448, 2^-6, 2^-9),
* PyTorch's CPU float8_e4m3fn conversion (a library routine, RNE),
* two encoders written here: a brute-force nearest search over all finite
  codes, and an exponent/quantum rounder built on numpy's round-half-even.
Sources: lpnh.cn DeepGEMM walkthrough §2.2 and §3.1 (E4M3, max 448) and §4.2
(round to nearest even).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def torch_decode():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def torch_encode(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def brute_encode(v, table):
    """Nearest finite code by exhaustive search; ties go to the even code."""
    v = np.asarray(v, np.float32)
    a = np.abs(v.astype(np.float64))
    mags = table[:0x7F]                     # codes 0x00..0x7E, magnitudes
    d = np.abs(a[:, None] - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates take the even code
    even = cand & ((np.arange(0x7F) % 2 == 0)[None, :])
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    pick = np.where(a >= 448.0, 0x7E, pick)
    sign = np.signbit(v).astype(np.uint8) << 7
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


def quantum_encode(v):
    """Round |v| on the E4M3 grid of its binade with round-half-even."""
    v = np.asarray(v, np.float32)
    a = np.abs(v.astype(np.float64))
    _, e = np.frexp(a)                      # a = m * 2^e, m in [0.5, 1)
    ex = np.maximum(e - 1, -6)              # binade exponent, subnormals share -6
    q = np.ldexp(1.0, ex - 3)               # spacing of 3 mantissa bits
    val = np.rint(a / q) * q                # numpy rint rounds half to even
    val = np.minimum(val, 448.0)
    code = np.zeros(a.shape, np.int64)
    sub = val < 2.0 ** -6
    code[sub] = np.rint(val[sub] / 2.0 ** -9).astype(np.int64)
    nz = ~sub
    _, e2 = np.frexp(val[nz])
    E = e2 - 1
    man = np.rint((val[nz] / np.ldexp(1.0, E) - 1.0) * 8).astype(np.int64)
    code[nz] = ((E + 7) << 3) | man
    sign = np.signbit(v).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def test_table_closed_form_points(oracle_mod):
    t = oracle_mod.e4m3_table()
    assert t[0x38] == 1.0 and t[0x40] == 2.0 and t[0x7E] == 448.0
    assert t[0x08] == 2.0 ** -6 and t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9
    assert t[0x00] == 0.0 and np.signbit(t[0x80]) and t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])


def test_table_structure(oracle_mod):
    t = oracle_mod.e4m3_table()
    finite = np.isfinite(t)
    assert finite.sum() == 254
    assert len(set(t[finite].tolist())) == 253          # +0 and -0 compare equal
    assert np.all(np.diff(t[:0x7F]) > 0)                # codes 0x00..0x7E increase
    for c in range(0x7F):
        assert t[c | 0x80] == -t[c]


def test_table_matches_torch(oracle_mod):
    t = oracle_mod.e4m3_table()
    ref = torch_decode()
    both = np.isfinite(ref)
    assert np.array_equal(np.isfinite(t), both)
    assert np.array_equal(t[both], ref[both])


def _midpoint_probes(table):
    mags = table[:0x7F]
    mids = 0.5 * (mags[:-1] + mags[1:])
    probes = [mags, mids, [448.0, 448.5, 455.0, 463.9, 464.0, 500.0, 1e6, 3e38]]
    v = np.concatenate([np.asarray(p, np.float64) for p in probes]).astype(np.float32)
    up = np.nextafter(v, np.float32(np.inf))
    dn = np.nextafter(v, np.float32(0))
    v = np.concatenate([v, up, dn, [0.0, 2.0 ** -149, 1e-30]]).astype(np.float32)
    return np.concatenate([v, -v])


def test_encoder_matches_bruteforce_at_midpoints(oracle_mod):
    t = oracle_mod.e4m3_table()
    v = _midpoint_probes(t)
    got = oracle_mod.e4m3_encode(v)
    assert np.array_equal(got, brute_encode(v, t))
    assert np.array_equal(got, quantum_encode(v))


def test_encoder_matches_torch_below_saturation(oracle_mod):
    t = oracle_mod.e4m3_table()
    rng = np.random.default_rng(11)
    v = np.concatenate([
        _midpoint_probes(t),
        rng.standard_normal(200000).astype(np.float32) * 50,
        (rng.uniform(-1, 1, 200000) * 2.0 ** rng.integers(-14, 9, 200000)).astype(np.float32),
    ]).astype(np.float32)
    v = v[np.abs(v) <= 464.0]               # torch turns larger values into NaN
    assert np.array_equal(oracle_mod.e4m3_encode(v), torch_encode(v))


def test_encoder_random_three_ways(oracle_mod):
    t = oracle_mod.e4m3_table()
    rng = np.random.default_rng(12)
    v = (rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 10, 20000)).astype(np.float32)
    got = oracle_mod.e4m3_encode(v)
    assert np.array_equal(got, quantum_encode(v))
    assert np.array_equal(got, brute_encode(v, t))


@pytest.mark.parametrize("value,code", [
    (1.0625, 0x38), (1.1875, 0x3A), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
    (432.0, 0x7E), (449.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE), (-1e-30, 0x80),
    (-0.0, 0x80), (0.0, 0x00), (240.0, 0x77), (-17.0, 0xD8),
])
def test_encoder_named_values(oracle_mod, value, code):
    assert int(oracle_mod.e4m3_encode([value])[0]) == code


def test_decode_encode_roundtrip(oracle_mod):
    t = oracle_mod.e4m3_table()
    codes = np.array([c for c in range(256) if np.isfinite(t[c])], np.uint8)
    back = oracle_mod.e4m3_encode(t[codes].astype(np.float32))
    assert np.array_equal(back, codes)


def test_pow2_ceil(oracle_mod):
    p = oracle_mod.pow2_ceil
    assert p(1.0) == 1.0 and p(1.0000001) == 2.0 and p(0.75) == 1.0
    assert p(10 / 448) == 2.0 ** -5 and p(2.0 ** -6) == 2.0 ** -6
    assert p(2.0 ** -140) == 2.0 ** -127                 # clamp to the UE8M0 floor
    assert p(1.5 * 2.0 ** -127) == 2.0 ** -126
    assert p(2.0 ** 100 * 1.01) == 2.0 ** 101
    rng = np.random.default_rng(3)
    for s in (rng.uniform(0.5, 2, 200) * 2.0 ** rng.integers(-120, 120, 200)).astype(np.float32):
        r = p(float(s))
        m, _ = np.frexp(r)
        assert m == 0.5 and r >= s and r / 2 < s
