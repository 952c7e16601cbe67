"""Pins of the oracle's requantized GEMM output (lpnh.cn DeepGEMM walkthrough
§2.2: the product is accumulated in FP32 and quantized on demand when written
back; §6: the scale computation fused into the kernel; §4.2: the quantization
steps; pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1: per-token scales).

Each property is checked against something other than the oracle itself:
* hand-derived codes and scales of a small exact GEMM (tests/golden);
* an exact integer matmul (numpy) in place of the oracle's GEMM;
* the E4M3 rounding bound of every dequantized value and the saturation of
  each block's largest element to +-448;
* the 128 x 128 variant on one row equals the per-row variant;
* the grouped variant equals dense calls per expert.
"""
import numpy as np
import pytest

import synthetic
from conftest import load_golden

GOLD = load_golden("requant_hand_cases.json")


def _sparse(spec, rows, cols):
    q = np.zeros((rows, cols), np.uint8)
    for r, k, code in spec:
        q[r, k] = int(code, 16)
    return q


def _gold_operands():
    op = GOLD["operands"]
    qa = _sparse(op["a"], op["M"], op["K"])
    qb = _sparse(op["b"], op["N"], op["K"])
    return qa, np.array(op["sa"], np.float32), qb, np.array(op["sb"], np.float32)


@pytest.mark.parametrize("case", GOLD["cases"], ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    qa, sa, qb, sb = _gold_operands()
    q, s, c, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, case["out_block_rows"], case["mode"])
    assert np.array_equal(c, np.array(GOLD["operands"]["C"], np.float64))
    want_s = np.array([[np.float32(3.0) / np.float32(448.0)] if v == "3/448" else v for v in case["scales"]],
                      np.float32)
    assert np.array_equal(s, want_s), (s, want_s)
    want_q = np.array([[int(h, 16) for h in row] for row in case["codes"]], np.uint8)
    assert np.array_equal(q, want_q), (q, want_q)


def _int_operands(m, n, k, seed):
    """Codes of -2, -1, 0, 1, 2 and unit scales: C is an integer matmul."""
    rng = np.random.default_rng(seed)
    code = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    va = rng.integers(-2, 3, (m, k))
    vb = rng.integers(-2, 3, (n, k))
    qa = np.vectorize(code.get)(va).astype(np.uint8)
    qb = np.vectorize(code.get)(vb).astype(np.uint8)
    sa = np.ones(((m + 127) // 128, k // 128), np.float32)
    sb = np.ones(((n + 127) // 128, k // 128), np.float32)
    return qa, sa, qb, sb, (va @ vb.T)


@pytest.mark.parametrize("block_rows", [1, 128])
@pytest.mark.parametrize("mode", [0, 1])
def test_integer_gemm_requant_matches_quantizing_the_integer_product(oracle_mod, block_rows, mode):
    qa, sa, qb, sb, exact = _int_operands(150, 300, 256, seed=7)
    q, s, c, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, block_rows, mode)
    assert np.array_equal(c, exact.astype(np.float64))
    x = exact.astype(np.float32)
    qr, sr = oracle_mod.quantize_1x128(x, mode) if block_rows == 1 else oracle_mod.quantize(x, mode)
    assert np.array_equal(q, qr) and np.array_equal(s, sr)


def _e4m3_half_step(x):
    """Half the spacing of E4M3 values around |x| (x in the representable range)."""
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 2.0 ** (e - 3) / 2


@pytest.mark.parametrize("block_rows", [1, 128])
@pytest.mark.parametrize("mode", [0, 1])
def test_dequantized_output_within_half_an_e4m3_step(oracle_mod, block_rows, mode):
    m, n, k = 260, 300, 384
    qa, sa = oracle_mod.quantize(synthetic.lognormal_rows((m, k), 11))
    qb, sb = oracle_mod.quantize(synthetic.lognormal_rows((n, k), 12))
    q, s, c, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, block_rows, mode)
    v = c.astype(np.float32).astype(np.float64)
    if block_rows == 1:
        d = oracle_mod.dequantize_1x128(q, s)
        srow = np.repeat(s.astype(np.float64), 128, axis=1)[:, :n]
    else:
        d = oracle_mod.dequantize(q, s)
        srow = np.repeat(np.repeat(s.astype(np.float64), 128, axis=0), 128, axis=1)[:m, :n]
    # |dec(q) s - v| <= s * half-step(v / s) (plus the FP32 division's rounding).
    bound = srow * _e4m3_half_step(v / srow) * (1 + 2.0 ** -20)
    assert np.all(np.abs(d - v) <= bound)
    # Each block's largest element maps to +-448 (FP32 scales) or into [224, 448] (powers of two).
    t = oracle_mod.e4m3_table()
    mag = np.abs(t[q])
    if block_rows == 1:
        for r in range(m):
            for j in range(s.shape[1]):
                seg = mag[r, 128 * j:128 * j + 128]
                assert seg.max() == 448.0 if mode == 0 else 224.0 <= seg.max() <= 448.0
    else:
        for i in range(s.shape[0]):
            for j in range(s.shape[1]):
                blk = mag[128 * i:128 * i + 128, 128 * j:128 * j + 128]
                assert blk.max() == 448.0 if mode == 0 else 224.0 <= blk.max() <= 448.0


@pytest.mark.parametrize("mode", [0, 1])
def test_single_row_block_equals_per_row(oracle_mod, mode):
    qa, sa = oracle_mod.quantize(synthetic.lognormal_rows((1, 256), 21))
    qb, sb = oracle_mod.quantize(synthetic.lognormal_rows((333, 256), 22))
    q1, s1, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, 1, mode)
    q2, s2, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, 128, mode)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_grouped_requant_equals_dense_per_expert(oracle_mod):
    k, n = 256, 200
    sizes = np.array([130, 0, 7])
    m_idx, _ = synthetic.moe_layout(sizes)
    a = synthetic.lognormal_rows((m_idx.size, k), 31)
    b = synthetic.lognormal_rows((3 * n, k), 32).reshape(3, n, k)
    qa, sa = oracle_mod.quantize_1x128(a)
    qs, ss = zip(*[oracle_mod.quantize(b[g]) for g in range(3)])
    qb, sb = np.stack(qs), np.stack(ss)
    q, s, _, _ = oracle_mod.grouped_gemm_requant(qa, sa, qb, sb, m_idx, 1, 0, a_1x128=True)
    for g in range(3):
        rows = np.flatnonzero(m_idx == g)
        if rows.size == 0:
            continue
        qd, sd, _, _ = oracle_mod.gemm_nt_requant(qa[rows], sa[rows], qb[g], sb[g], 1, 0, a_1x128=True)
        assert np.array_equal(q[rows], qd) and np.array_equal(s[rows], sd)
    pad = m_idx < 0
    assert np.all(q[pad] == 0) and np.all(s[pad] == 1.0)


@pytest.mark.parametrize("block_rows", [1, 128])
def test_parity_check_rejects_planted_errors(oracle_mod, block_rows):
    """The GPU tests' requantization check passes the oracle's own output and
    fails it once a code is moved two E4M3 steps or a scale is doubled."""
    from parity import assert_requant_within_bound
    m, n, k = 200, 300, 256
    qa, sa = oracle_mod.quantize(synthetic.lognormal_rows((m, k), 61))
    qb, sb = oracle_mod.quantize(synthetic.lognormal_rows((n, k), 62))
    q, s, c, e = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, block_rows, 0)
    assert_requant_within_bound(q, s, c, e, block_rows, False, "oracle", oracle_mod)
    i, j = np.unravel_index(np.argmax(np.abs(c[:, :128]) < np.abs(c[:, :128]).max() / 4), (m, 128))
    bad_q = q.copy()
    bad_q[i, j] = (int(q[i, j]) + 2) & 0xFF if (q[i, j] & 0x7F) < 0x7C else (int(q[i, j]) - 2)
    with pytest.raises(AssertionError):
        assert_requant_within_bound(bad_q, s, c, e, block_rows, False, "planted code", oracle_mod)
    bad_s = s.copy()
    bad_s[0, 0] *= 2
    with pytest.raises(AssertionError):
        assert_requant_within_bound(q, bad_s, c, e, block_rows, False, "planted scale", oracle_mod)
