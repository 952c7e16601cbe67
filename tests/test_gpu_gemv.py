"""GPU parity of single-row GEMMs (M = 1, B stored K-major), which stream B
through the kernel of gemv.cu, against the oracle (lpnh.cn DeepGEMM
walkthrough §2.2, §3.2; pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1, §4.1).

* Exact cases: codes -2..2 with power-of-two scales keep every step exact, so
  the bf16 result equals the oracle's rounded to bf16, bit for bit, and equals
  the split-K kernel's (the kernel single rows take while an SM cap is set).
* General cases: |C_gpu - C_ref| <= 8e-3 |C_ref| + 1e-4 sum_k |a~ b~|, on the
  decode shapes 1 x 24576 x 1536 and 1 x 7168 x 16384 among others.
* Ragged N (not a multiple of the kernel's 4 or 8 rows per CTA), K not a
  multiple of 512 (partial warps) or of 4096 (partial last pass of the CTA),
  padded row strides."""
import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import assert_within_bound, device, to_dev

pytestmark = pytest.mark.gpu

CODES = np.array([0xC0, 0xB8, 0x00, 0x38, 0x40], np.uint8)  # -2, -1, 0, 1, 2


def _exact(n, k, seed):
    rng = np.random.default_rng(seed)
    qa = CODES[rng.integers(0, 5, (1, k))]
    qb = CODES[rng.integers(0, 5, (n, k))]
    sa = np.exp2(rng.integers(-2, 3, (1, k // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-2, 3, (-(-n // 128), k // 128))).astype(np.float32)
    return qa, sa, qb, sb


def _random(oracle_mod, n, k, seed, mode=0, a_1x128=False):
    quant_a = oracle_mod.quantize_1x128 if a_1x128 else oracle_mod.quantize
    qa, sa = quant_a(synthetic.lognormal_rows((1, k), seed), mode)
    qb, sb = oracle_mod.quantize(synthetic.lognormal_rows((n, k), seed + 1), mode)
    return qa, sa, qb, sb


def _in_wider(x, cols, dev):
    """x on the device inside a buffer of `cols` columns (row stride > width)."""
    buf = torch.zeros((x.shape[0], cols), dtype=torch.uint8, device=dev)
    buf[:, :x.shape[1]] = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return buf[:, :x.shape[1]]


def _gemm(a, sa, b, sb, n, layout="NT", mode=0, ldc=None, a_1x128=False):
    dev = device()
    ldc = ldc or -(-n // 8) * 8
    c = torch.full((1, ldc), float("nan"), dtype=torch.bfloat16, device=dev)[:, :n]
    if a_1x128:
        bq.dg_fp8_gemm_nt_1x128(c, a, b, sa, sb, mode)
    else:
        bq.dg_fp8_gemm(c, a, b, sa, sb, layout, mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return c


def _stored_a(qa, layout, dev):
    """A as the layout stores it: [1][K] (NT) or [K][1] inside 16-byte rows (TT)."""
    if layout == "NT":
        return to_dev(qa, dev)
    return _in_wider(qa.T, 16, dev)


def _bits(x):
    t = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.asarray(x, np.float32))
    return t.float().cpu().to(torch.bfloat16).view(torch.int16)


SHAPES = [(8, 128), (37, 384), (1000, 1536), (129, 4352), (300, 16384), (2112, 7168)]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("layout", ["NT", "TT"])
@pytest.mark.parametrize("nk", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_bit_identical(oracle_mod, nk, layout, mode):
    n, k = nk
    qa, sa, qb, sb = _exact(n, k, seed=n + k)
    dev = device()
    c = _gemm(_stored_a(qa, layout, dev), to_dev(sa, dev), to_dev(qb, dev), to_dev(sb, dev), n, layout, mode)
    a_st = qa if layout == "NT" else np.ascontiguousarray(qa.T)
    ref, _ = oracle_mod.gemm_layout(a_st, sa, qb, sb, layout)
    assert torch.equal(_bits(c), _bits(ref.astype(np.float32)))


def test_same_bits_as_split_k_kernel(oracle_mod):
    """Exact inputs: the streaming kernel and the split-K kernel (taken while an
    SM cap is set) give the same bits."""
    n, k = 2112, 7168
    qa, sa, qb, sb = _exact(n, k, seed=3)
    dev = device()
    args = (to_dev(qa, dev), to_dev(sa, dev), to_dev(qb, dev), to_dev(sb, dev), n)
    c_stream = _gemm(*args)
    try:
        bq.dg_set_num_sms(152)
        c_split = _gemm(*args)
    finally:
        bq.dg_set_num_sms(0)
    assert torch.equal(c_stream.view(torch.int16), c_split.view(torch.int16))


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("nk", [(24576, 1536), (7168, 16384), (2112, 7168), (1000, 640)],
                         ids=lambda s: "x".join(map(str, s)))
def test_random_within_bound(oracle_mod, nk, mode):
    n, k = nk
    qa, sa, qb, sb = _random(oracle_mod, n, k, seed=n % 97 + k, mode=mode)
    dev = device()
    c = _gemm(to_dev(qa, dev), to_dev(sa, dev), to_dev(qb, dev), to_dev(sb, dev), n, mode=mode)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_within_bound(c, ref, mag, f"1x{n}x{k} mode {mode}")


def test_row_wise_a_scales(oracle_mod):
    n, k = 4096, 7168
    qa, sa, qb, sb = _random(oracle_mod, n, k, seed=41, a_1x128=True)
    dev = device()
    c = _gemm(to_dev(qa, dev), to_dev(sa, dev), to_dev(qb, dev), to_dev(sb, dev), n, a_1x128=True)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, a_1x128=True)
    assert_within_bound(c, ref, mag, "1x128 A scales")


def test_padded_strides(oracle_mod):
    """B rows inside a wider buffer (ld_b = K + 128), C inside a wider row."""
    n, k = 777, 2048
    qa, sa, qb, sb = _exact(n, k, seed=7)
    dev = device()
    c = _gemm(to_dev(qa, dev), to_dev(sa, dev), _in_wider(qb, k + 128, dev), to_dev(sb, dev), n, ldc=1024)
    ref, _ = oracle_mod.gemm_layout(qa, sa, qb, sb, "NT")
    assert torch.equal(_bits(c), _bits(ref.astype(np.float32)))


def test_split_n_is_bit_identical(oracle_mod):
    """Rows of B are independent outputs: a split of N at a 128-row block edge
    reproduces the full result bit for bit."""
    n, k = 1000, 2048
    qa, sa, qb, sb = _random(oracle_mod, n, k, seed=13)
    dev = device()
    a, s_a = to_dev(qa, dev), to_dev(sa, dev)
    full = _gemm(a, s_a, to_dev(qb, dev), to_dev(sb, dev), n)
    left = _gemm(a, s_a, to_dev(qb[:512], dev), to_dev(sb[:4], dev), 512)
    right = _gemm(a, s_a, to_dev(qb[512:], dev), to_dev(sb[4:], dev), n - 512)
    assert torch.equal(torch.cat([left, right], 1).view(torch.int16), full.view(torch.int16))
