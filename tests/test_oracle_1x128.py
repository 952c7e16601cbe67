"""Pins of the oracle's row-wise (1x128) quantizer and of its GEMMs with one A
scale per row and K block (lpnh.cn DeepGEMM walkthrough §2.3: the block shape
is a granularity trade-off, §4.2: the five quantization steps; pzsr.cn
"DeepGEMM: GPU上的高效BLAS内核库解析" §3.1: per-token activation scales beside
128x128 weight scales).

Each function is checked against something other than itself:
* the 1x128 quantizer against the (separately pinned) 128x128 quantizer run on
  one-row matrices, whose only block is exactly that row's 1x128 block, and
  against hand-derived codes;
* the per-row-scale GEMM against the 128x128-scale GEMM when every row of a
  128-row block carries the same scale, against exact integer matmuls with
  unit scales, and by the linearity of one row's scale;
* the grouped variant against per-expert dense calls.
"""
import numpy as np
import pytest

import synthetic


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(1, 128), (3, 300), (17, 1000), (5, 7)])
def test_1x128_equals_128x128_on_single_rows(oracle_mod, mode, shape):
    x = synthetic.lognormal_rows(shape, seed=shape[0] * 31 + shape[1])
    x[0, : min(5, shape[1])] = 0.0                      # zero prefix
    if shape[0] > 2:
        x[2, :] = 0.0                                   # an all-zero row
        x[1, 0] = -0.0
    q, s = oracle_mod.quantize_1x128(x, mode)
    nbc = -(-shape[1] // 128)
    assert q.shape == shape and s.shape == (shape[0], nbc)
    for r in range(shape[0]):
        q1, s1 = oracle_mod.quantize(x[r:r + 1], mode)
        assert np.array_equal(q1[0], q[r]), r
        assert np.array_equal(s1[0], s[r]), r


def test_1x128_hand_cases(oracle_mod):
    """Hand-derived (walkthrough §3.1: scale = max|x| / 448, §4.2: divide and
    round to E4M3, §5.4: an all-zero block gets scale 1)."""
    x = np.zeros((3, 256), np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 448.0, -224.0, 1.0      # block max 448 -> s = 1
    x[0, 128] = 896.0                                    # second block: s = 2, 896/2 = 448
    x[0, 129] = 3.0                                      # 3/2 = 1.5 = 0x3C
    x[1, 5] = -0.0                                       # all-zero row: s = 1, sign kept
    x[2, :128] = 2.0                                     # constant block: s = 2/448, x/s = 448
    q, s = oracle_mod.quantize_1x128(x)
    assert s[0, 0] == 1.0 and s[0, 1] == 2.0 and s[1, 0] == 1.0 and s[1, 1] == 1.0
    assert s[2, 0] == np.float32(2.0) / np.float32(448.0)
    assert (q[0, 0], q[0, 1], q[0, 2], q[0, 3]) == (0x7E, 0xF6, 0x38, 0x00)
    assert (q[0, 128], q[0, 129]) == (0x7E, 0x3C)
    assert q[1, 5] == 0x80 and q[1, 4] == 0x00
    assert np.all(q[2, :128] == 0x7E) and np.all(q[2, 128:] == 0x00)


def test_pow2_scales_are_powers_of_two(oracle_mod):
    x = synthetic.lognormal_rows((9, 640), seed=3)
    _, s = oracle_mod.quantize_1x128(x, 1)
    m, _ = np.frexp(s)
    assert np.all(m == 0.5) and np.all(s >= 2.0 ** -127)


def _operands(oracle_mod, m, n, k, seed):
    a = synthetic.lognormal_rows((m, k), seed)
    b = synthetic.lognormal_rows((n, k), seed + 1)
    qa, sa = oracle_mod.quantize_1x128(a)
    qb, sb = oracle_mod.quantize(b)
    return qa, sa, qb, sb


def test_rowwise_gemm_reduces_to_block_gemm(oracle_mod):
    """Every row of a 128-row block with the block's scale: the per-row GEMM
    must equal the 128x128-scale GEMM bit for bit."""
    m, n, k = 200, 150, 384
    qa, _, qb, sb = _operands(oracle_mod, m, n, k, 11)
    sblk = np.exp2(np.random.default_rng(1).integers(-4, 4, (2, 3))).astype(np.float32) * 0.75
    srow = np.repeat(sblk, 128, axis=0)[:m]
    c_blk, e_blk = oracle_mod.gemm_nt(qa, sblk, qb, sb)
    c_row, e_row = oracle_mod.gemm_nt(qa, srow, qb, sb, a_1x128=True)
    assert np.array_equal(c_blk, c_row) and np.array_equal(e_blk, e_row)


def test_rowwise_gemm_unit_scales_exact(oracle_mod):
    """Codes of -1, 0, 1, 2 and unit scales: an exact integer matmul."""
    rng = np.random.default_rng(5)
    m, n, k = 40, 24, 256
    va = rng.integers(-1, 3, (m, k))
    vb = rng.integers(-1, 2, (n, k))
    code = {-1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    qa = np.vectorize(code.get)(va).astype(np.uint8)
    qb = np.vectorize(code.get)(vb).astype(np.uint8)
    c, _ = oracle_mod.gemm_nt(qa, np.ones((m, 2), np.float32), qb, np.ones((1, 2), np.float32),
                              a_1x128=True)
    assert np.array_equal(c, (va @ vb.T).astype(np.float64))


def test_rowwise_gemm_row_scale_linearity(oracle_mod):
    """Doubling sa[i, kb] changes only row i, by exactly that block's share."""
    m, n, k = 7, 33, 256
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, 21)
    c0, _ = oracle_mod.gemm_nt(qa, sa, qb, sb, a_1x128=True)
    sa2 = sa.copy()
    sa2[3, 1] *= 2
    c1, _ = oracle_mod.gemm_nt(qa, sa2, qb, sb, a_1x128=True)
    other = np.ones(m, bool)
    other[3] = False
    assert np.array_equal(c0[other], c1[other])
    # Row 3 with K block 1 only (K block 0 codes zeroed): the change is exactly that term.
    qa_kb1 = qa.copy()
    qa_kb1[:, :128] = 0
    d, _ = oracle_mod.gemm_nt(qa_kb1, sa, qb, sb, a_1x128=True)
    np.testing.assert_allclose(c1[3] - c0[3], d[3], rtol=1e-12, atol=1e-300)


def test_rowwise_grouped_equals_dense_per_expert(oracle_mod):
    k, n = 256, 96
    sizes = np.array([130, 0, 5])
    m_idx, offs = synthetic.moe_layout(sizes)
    a = synthetic.lognormal_rows((m_idx.size, k), 31)
    b = synthetic.lognormal_rows((3 * n, k), 32).reshape(3, n, k)
    qa, sa = oracle_mod.quantize_1x128(a)
    qs, ss = zip(*[oracle_mod.quantize(b[g]) for g in range(3)])
    qb, sb = np.stack(qs), np.stack(ss)
    c, _ = oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, m_idx, a_1x128=True)
    for g in range(3):
        rows = np.flatnonzero(m_idx == g)
        if rows.size == 0:
            continue
        cd, _ = oracle_mod.gemm_nt(qa[rows], sa[rows], qb[g], sb[g], a_1x128=True)
        assert np.array_equal(c[rows], cd)
    assert np.all(c[m_idx < 0] == 0)
