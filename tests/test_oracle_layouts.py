"""Pins of the oracle's layouts (pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析"
§3.1: NT, TN, NN, TT from SM100 on) and of its K-grouped GEMM (§3.2: grouping
along K), each against something other than the oracle's own GEMM:
* integer operand values with power-of-two block scales: every layout equals
  an exact numpy integer matmul of the logical operands;
* the K-grouped GEMM equals numpy products per K range, and its groups add up
  to the whole-K product;
* swapping the roles of A and B transposes the result (C^T = B . A).
"""
import numpy as np
import pytest

CODE = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}


def _int_op(rng, rows, cols):
    v = rng.integers(-2, 3, (rows, cols))
    return v, np.vectorize(CODE.get)(v).astype(np.uint8)


def _pow2_scales(rng, shape):
    return np.exp2(rng.integers(-2, 3, shape)).astype(np.float64)


def _exact(va, vb, sa, sb):
    """sum_kb sa[m/128, kb] sb[n/128, kb] sum_k va[m, k] vb[n, k], exactly."""
    m, k = va.shape
    n = vb.shape[0]
    out = np.zeros((m, n))
    for kb in range(k // 128):
        p = va[:, 128 * kb:128 * kb + 128] @ vb[:, 128 * kb:128 * kb + 128].T
        out += np.repeat(sa[:, kb], 128)[:m, None] * np.repeat(sb[:, kb], 128)[None, :n] * p
    return out


@pytest.mark.parametrize("layout", ["NT", "TN", "NN", "TT"])
def test_layouts_equal_exact_integer_product(oracle_mod, layout):
    rng = np.random.default_rng(3)
    m, n, k = 150, 140, 384
    va, qa = _int_op(rng, m, k)     # logical A [M, K]
    vb, qb = _int_op(rng, n, k)     # logical B^T [N, K]
    sa = _pow2_scales(rng, (2, 3))
    sb = _pow2_scales(rng, (2, 3))
    a_st = qa.T.copy() if layout[0] == "T" else qa
    b_st = qb.T.copy() if layout[1] == "N" else qb
    c, _ = oracle_mod.gemm_layout(a_st, sa.astype(np.float32), b_st, sb.astype(np.float32), layout)
    assert np.array_equal(c, _exact(va, vb, sa, sb))


def test_swapping_operands_transposes(oracle_mod):
    rng = np.random.default_rng(4)
    va, qa = _int_op(rng, 130, 256)
    vb, qb = _int_op(rng, 200, 256)
    sa, sb = _pow2_scales(rng, (2, 2)).astype(np.float32), _pow2_scales(rng, (2, 2)).astype(np.float32)
    c1, _ = oracle_mod.gemm_layout(qa, sa, qb, sb, "NT")
    c2, _ = oracle_mod.gemm_layout(qb, sb, qa, sa, "NT")
    assert np.array_equal(c1, c2.T)


def test_k_grouped_equals_products_per_range(oracle_mod):
    rng = np.random.default_rng(5)
    m, n = 140, 200
    sizes = [256, 0, 128, 384]
    k_tot = sum(sizes)
    va, qa = _int_op(rng, m, k_tot)
    vb, qb = _int_op(rng, n, k_tot)
    sa = _pow2_scales(rng, (2, k_tot // 128))
    sb = _pow2_scales(rng, (2, k_tot // 128))
    c, _ = oracle_mod.k_grouped_gemm_tn(qa.T.copy(), sa.astype(np.float32), qb.T.copy(), sb.astype(np.float32),
                                        sizes)
    off = 0
    for g, kg in enumerate(sizes):
        want = _exact(va[:, off:off + kg], vb[:, off:off + kg], sa[:, off // 128:(off + kg) // 128],
                      sb[:, off // 128:(off + kg) // 128]) if kg else np.zeros((m, n))
        assert np.array_equal(c[g], want), g
        off += kg
    assert np.array_equal(c.sum(axis=0), _exact(va, vb, sa, sb))


def test_k_grouped_rejects_unaligned_sizes(oracle_mod):
    qa = np.zeros((256, 8), np.uint8)
    with pytest.raises(ValueError):
        oracle_mod.k_grouped_gemm_tn(qa, np.ones((1, 2), np.float32), qa, np.ones((1, 2), np.float32), [100, 156])
