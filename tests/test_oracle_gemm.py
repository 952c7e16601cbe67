"""Pins for the oracle's block-scaled NT GEMM (dense and M-grouped).

Sources: lpnh.cn DeepGEMM walkthrough §2.2 (per-block scales, the product
block carries scale_a * scale_b, FP32 accumulation), §4.3 (FP64 CPU reference),
§6 (unit scales plus exactly representable inputs isolate the kernel logic);
pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1 (NT layout) and §2.3/§3.2
(M-grouped GEMM for MoE experts).
Pins: hand-derived fixtures; exact integer-valued products against numpy's
int64 matmul; a naive dequantize-then-matmul in float64 (numpy BLAS, torch's
FP8 decode); one-hot B; linearity in one scale block; grouped == dense slices.
"""
import numpy as np
import pytest
import torch

from conftest import load_golden

import synthetic


def _decode(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double().numpy()


def _sparse(shape, entries):
    out = np.zeros(shape, np.uint8)
    for r, k, h in entries:
        out[r, k] = int(h, 16)
    return out


def _naive(qa, sa, qb, sb):
    """Dequantize every element (value * its block scale), then one float64 matmul."""
    def deq(q, s):
        e = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:q.shape[0], :q.shape[1]]
        return _decode(q) * e
    a, b = deq(qa, sa), deq(qb, sb)
    return a @ b.T, np.abs(a) @ np.abs(b).T


@pytest.mark.parametrize("case", load_golden("gemm_hand_cases.json")["cases"],
                         ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    m, n, k = case["M"], case["N"], case["K"]
    qa = _sparse((m, k), case["a"])
    qb = _sparse((n, k), case["b"])
    sa = np.array(case["sa"], np.float32)
    sb = np.array(case["sb"], np.float32)
    c, e = oracle_mod.gemm_nt(qa, sa, qb, sb)
    if "C" in case:
        want_c, want_e = np.array(case["C"]), np.array(case["E"])
    else:
        want_c, want_e = np.zeros((m, n)), np.zeros((m, n))
        for r, j, v in case["C_sparse"]:
            want_c[r, j] = v
        for r, j, v in case["E_sparse"]:
            want_e[r, j] = v
    assert np.array_equal(c, want_c), case["derivation"]
    assert np.array_equal(e, want_e)


def _codes_for_integers(rng, shape, lo, hi):
    """E4M3 codes of small integers in [lo, hi] (all exactly representable)."""
    vals = rng.integers(lo, hi + 1, shape)
    q = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(_decode(q), vals)
    return q, vals


def test_unit_scales_exact_integer_product(oracle_mod):
    rng = np.random.default_rng(31)
    m, n, k = 96, 200, 384
    qa, va = _codes_for_integers(rng, (m, k), -16, 16)
    qb, vb = _codes_for_integers(rng, (n, k), -16, 16)
    sa = np.ones((1, k // 128), np.float32)
    sb = np.ones((2, k // 128), np.float32)
    c, e = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert np.array_equal(c, (va.astype(np.int64) @ vb.T.astype(np.int64)).astype(np.float64))
    assert np.array_equal(e, (np.abs(va) @ np.abs(vb).T).astype(np.float64))


@pytest.mark.parametrize("m,n,k", [(64, 64, 128), (130, 257, 256), (1, 300, 512), (255, 17, 384)])
def test_matches_naive_dequantized_matmul(oracle_mod, m, n, k):
    a = synthetic.lognormal_rows((m, k), seed=32)
    b = synthetic.lognormal_rows((n, k), seed=33)
    qa, sa = oracle_mod.quantize(a, 0)
    qb, sb = oracle_mod.quantize(b, 0)
    c, e = oracle_mod.gemm_nt(qa, sa, qb, sb)
    c2, e2 = _naive(qa, sa, qb, sb)
    assert np.allclose(c, c2, rtol=0, atol=1e-12 * e2.max())
    assert np.allclose(e, e2, rtol=1e-12, atol=0)


def test_one_hot_b_reproduces_dequantized_a(oracle_mod):
    m, k = 150, 256
    a = synthetic.normal((m, k), seed=34)
    qa, sa = oracle_mod.quantize(a, 0)
    cols = np.array([0, 5, 127, 128, 200, 255])
    qb = np.zeros((cols.size, k), np.uint8)
    qb[np.arange(cols.size), cols] = 0x38                          # 1.0
    sb = np.ones((1, k // 128), np.float32)
    c, _ = oracle_mod.gemm_nt(qa, sa, qb, sb)
    deq = _decode(qa) * np.repeat(np.repeat(sa.astype(np.float64), 128, 0), 128, 1)[:m, :k]
    assert np.array_equal(c, deq[:, cols])


def test_linear_in_one_scale_block(oracle_mod):
    m, n, k = 200, 160, 384
    a = synthetic.lognormal_rows((m, k), seed=35)
    b = synthetic.lognormal_rows((n, k), seed=36)
    qa, sa = oracle_mod.quantize(a, 0)
    qb, sb = oracle_mod.quantize(b, 0)
    c0, _ = oracle_mod.gemm_nt(qa, sa, qb, sb)
    sa2 = sa.copy()
    sa2[1, 2] *= 2                                                 # rows 128.., K block 2
    c1, _ = oracle_mod.gemm_nt(qa, sa2, qb, sb)
    only = np.zeros_like(sa)
    only[1, 2] = sa[1, 2]
    contrib, _ = oracle_mod.gemm_nt(qa, only, qb, sb)
    assert np.allclose(c1 - c0, contrib, rtol=0, atol=1e-12 * np.abs(c0).max())
    assert np.array_equal(c1[:128], c0[:128])


def test_row_subset_equals_full(oracle_mod):
    a = synthetic.normal((300, 256), seed=37)
    b = synthetic.normal((90, 256), seed=38)
    qa, sa = oracle_mod.quantize(a, 0)
    qb, sb = oracle_mod.quantize(b, 0)
    full, efull = oracle_mod.gemm_nt(qa, sa, qb, sb)
    rows = np.array([299, 0, 128, 127, 17])
    part, epart = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows)
    assert np.array_equal(part, full[rows]) and np.array_equal(epart, efull[rows])


def test_error_against_unquantized_product_is_of_fp8_order(oracle_mod):
    """§4.3 of the walkthrough: ~1e-2 against FP64 is normal, 1e-1 is a bug."""
    m, n, k = 128, 256, 512
    a = synthetic.normal((m, k), seed=1000)
    b = synthetic.normal((n, k), seed=1001)
    qa, sa = oracle_mod.quantize(a, 0)
    qb, sb = oracle_mod.quantize(b, 0)
    c, _ = oracle_mod.gemm_nt(qa, sa, qb, sb)
    exact = a.astype(np.float64) @ b.astype(np.float64).T
    rel = np.linalg.norm(c - exact) / np.linalg.norm(exact)
    assert rel < 5e-2


def test_grouped_equals_dense_per_expert(oracle_mod):
    k, n, g = 256, 200, 3
    sizes = np.array([5, 130, 0])
    m_idx, offs = synthetic.moe_layout(sizes)
    a = synthetic.lognormal_rows((m_idx.size, k), seed=39)
    a[m_idx < 0] = 0
    b = synthetic.lognormal_rows((g * n, k), seed=40).reshape(g, n, k)
    qa, sa = oracle_mod.quantize(a, 0)
    qbs, sbs = zip(*[oracle_mod.quantize(b[i], 0) for i in range(g)])
    qb, sb = np.stack(qbs), np.stack(sbs)
    c, e = oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, m_idx)
    for gi in range(g):
        lo, hi = offs[gi], offs[gi] + sizes[gi]
        if hi == lo:
            continue
        cd, ed = oracle_mod.gemm_nt(qa, sa, qb[gi], sb[gi], rows=np.arange(lo, hi))
        assert np.array_equal(c[lo:hi], cd) and np.array_equal(e[lo:hi], ed)
    assert np.all(c[m_idx < 0] == 0) and np.all(e[m_idx < 0] == 0)


def test_grouped_rejects_bad_expert_id(oracle_mod):
    qa = np.zeros((128, 128), np.uint8)
    sa = np.ones((1, 1), np.float32)
    qb = np.zeros((2, 8, 128), np.uint8)
    sb = np.ones((2, 1, 1), np.float32)
    mi = np.zeros(128, np.int32)
    mi[3] = 2
    with pytest.raises(ValueError):
        oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, mi)


def _fp32_single_row(qa, sa, qb, sb, factor_first):
    """One row of A against B in FP32 arithmetic, summed in K order: either the
    K block's partial sum P_kb is formed first and then scaled, acc += s (sum a b),
    or each A value is scaled first, acc += (s a) b. Both are FP32 evaluations of
    the method's sum (walkthrough §2.2: the product block carries sa * sb)."""
    f32 = np.float32
    a = _decode(qa).astype(f32)[0]
    b = _decode(qb).astype(f32)
    n, k = b.shape
    acc = np.zeros(n, f32)
    for kb in range(k // 128):
        s = (sa[0, kb].astype(f32) * sb[np.arange(n) // 128, kb].astype(f32)).astype(f32)
        ks = slice(128 * kb, 128 * kb + 128)
        if factor_first:
            for kk in range(ks.start, ks.stop):
                acc = (acc + ((s * a[kk]).astype(f32) * b[:, kk]).astype(f32)).astype(f32)
        else:
            p = np.zeros(n, f32)
            for kk in range(ks.start, ks.stop):
                p = (p + (a[kk] * b[:, kk]).astype(f32)).astype(f32)
            acc = (acc + (s * p).astype(f32)).astype(f32)
    return acc.astype(np.float64)


@pytest.mark.parametrize("factor_first", [False, True])
def test_fp32_factor_order_within_parity_bound(oracle_mod, factor_first):
    """Whether the factor sa * sb multiplies the K block's FP32 partial sum or
    each A value before the FP32 sum, the result stays within the parity bound
    8e-3 |C| + 1e-4 sum|a~ b~| of the exact (float64) oracle result, with a
    margin: the bound the GPU kernels are held to covers either order."""
    n, k = 300, 2048
    qa, sa = oracle_mod.quantize(synthetic.lognormal_rows((1, k), 77), 0)
    qb, sb = oracle_mod.quantize(synthetic.lognormal_rows((n, k), 78), 0)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    got = _fp32_single_row(qa, sa, qb, sb, factor_first)
    bound = 8e-3 * np.abs(ref[0]) + 1e-4 * mag[0]
    assert np.all(np.abs(got - ref[0]) <= 0.1 * bound)
