"""Pins for the oracle's 128x128 block quantizer.

Sources: lpnh.cn DeepGEMM walkthrough §4.2 steps 1-5 (128x128 blocks,
scale = max_abs / 448 kept in FP32, divide, round to nearest even, scales in a
separate array), §5.4 (all-zero blocks), §4.1/§5.1 (tiny hand cases); pzsr.cn
"DeepGEMM: GPU上的高效BLAS内核库解析" §3.1 (power-of-two UE8M0 scales).
Pins: hand-derived fixtures, closed-form invariants (the amax element maps to
+-448, the error bound of one E4M3 rounding, scale factoring under 2^k), and
block independence (edge blocks and block indexing).
"""
import numpy as np
import pytest
import torch

from conftest import load_golden

import synthetic


def _dense_case(case):
    if "x" in case:
        x = np.array(case["x"], np.float32)
        codes = np.array([[int(c, 16) for c in row] for row in case["codes"]], np.uint8)
    else:
        x = np.zeros(case["sparse_shape"], np.float32)
        codes = np.zeros(case["sparse_shape"], np.uint8)
        for r, c, v in case["sparse_x"]:
            x[r, c] = v
        for r, c, h in case["sparse_codes"]:
            codes[r, c] = int(h, 16)
    return x, codes, np.array(case["scales"], np.float32)


@pytest.mark.parametrize("case", load_golden("quantize_hand_cases.json")["cases"],
                         ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    x, codes, scales = _dense_case(case)
    q, s = oracle_mod.quantize(x, case["mode"])
    assert np.array_equal(q, codes), case["derivation"]
    assert np.array_equal(s, scales)


def _decode(q):
    return torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()


def _expand(s, shape):
    return np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:shape[0], :shape[1]]


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (130, 200), (1, 7), (300, 129)])
@pytest.mark.parametrize("mode", [0, 1])
def test_block_amax_maps_to_448_and_scale_is_amax_over_448(oracle_mod, shape, mode):
    x = synthetic.lognormal_rows(shape, seed=21)
    q, s = oracle_mod.quantize(x, mode)
    rb, cb = s.shape
    assert (rb, cb) == (-(-shape[0] // 128), -(-shape[1] // 128))
    for bi in range(rb):
        for bj in range(cb):
            blk = x[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            fp32_scale = np.float32(amax / np.float32(448.0))
            i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            code = q[bi * 128 + i[0], bj * 128 + i[1]]
            if mode == 0:
                assert s[bi, bj] == fp32_scale
                assert code & 0x7F == 0x7E
            else:
                m, _ = np.frexp(s[bi, bj])
                assert m == 0.5 and s[bi, bj] >= fp32_scale and s[bi, bj] / 2 < fp32_scale
                assert 224.0 < _decode(np.array([code & 0x7F], np.uint8))[0] <= 448.0
            assert (code >> 7) == (blk[i] < 0)


@pytest.mark.parametrize("mode", [0, 1])
def test_error_bound_of_one_rounding(oracle_mod, mode):
    x = synthetic.lognormal_rows((256, 512), seed=22)
    q, s = oracle_mod.quantize(x, mode)
    se = _expand(s, x.shape)
    v = x.astype(np.float64) / se                   # exact quotient (close to fl32(x/s))
    err = np.abs(_decode(q) - v)
    _, e = np.frexp(np.abs(v))
    half_ulp = np.ldexp(1.0, np.maximum(e - 1, -6) - 4)   # half the E4M3 spacing
    tol = half_ulp + np.abs(v) * 2.0 ** -23                # plus the FP32 rounding of x / s
    assert np.all(err <= tol)


def test_zero_and_underflow_blocks(oracle_mod):
    x = np.zeros((256, 256), np.float32)
    x[0, 0] = -0.0
    x[130:132, 200] = 1e-44                          # amax / 448 underflows to 0 in FP32
    x[200, 10] = 3.0
    q, s = oracle_mod.quantize(x, 0)
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[1, 1] == 1.0
    assert s[1, 0] == np.float32(3.0) / np.float32(448.0)
    assert q[0, 0] == 0x80 and np.all(q[:128, 128:] == 0)
    assert q[130, 200] == 0x00 and q[200, 10] == 0x7E


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("k", [-20, -3, 5, 30])
def test_scale_factors_out_by_power_of_two(oracle_mod, mode, k):
    x = synthetic.normal((256, 256), seed=23)
    q0, s0 = oracle_mod.quantize(x, mode)
    q1, s1 = oracle_mod.quantize(np.ldexp(x, k).astype(np.float32), mode)
    assert np.array_equal(q0, q1)
    assert np.array_equal(s1, np.ldexp(s0, k).astype(np.float32))


@pytest.mark.parametrize("mode", [0, 1])
def test_blocks_are_independent_and_edges_use_valid_elements(oracle_mod, mode):
    x = synthetic.lognormal_rows((300, 270), seed=24)
    q, s = oracle_mod.quantize(x, mode)
    padded = np.zeros((384, 384), np.float32)
    padded[:300, :270] = x
    qp, sp = oracle_mod.quantize(padded, mode)
    assert np.array_equal(qp[:300, :270], q) and np.array_equal(sp, s)
    for bi, bj in [(0, 0), (1, 2), (2, 1), (2, 2)]:
        blk = x[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
        qb, sb = oracle_mod.quantize(blk, mode)
        assert sb.shape == (1, 1) and sb[0, 0] == s[bi, bj]
        assert np.array_equal(qb, q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128])


def test_rejects_non_finite(oracle_mod):
    x = np.ones((4, 4), np.float32)
    x[1, 1] = np.inf
    with pytest.raises(ValueError):
        oracle_mod.quantize(x, 0)


def test_quantization_error_order_of_the_pages(oracle_mod):
    """The walkthrough (§4.3) calls ~1e-2 relative error against an FP64
    reference normal for FP8; check the dequantized matrix is of that order."""
    x = synthetic.normal((512, 512), seed=25)
    q, s = oracle_mod.quantize(x, 0)
    deq = _decode(q) * _expand(s, x.shape)
    rel = np.linalg.norm(deq - x) / np.linalg.norm(x)
    assert 1e-3 < rel < 5e-2
