"""GPU parity of the row-wise (1x128) quantizer and of the GEMMs with one A
scale per row and K block, through the C ABI, against the oracle
(lpnh.cn DeepGEMM walkthrough §2.3, §4.2; pzsr.cn "DeepGEMM: GPU上的高效BLAS
内核库解析" §3.1: per-token activation scales beside 128x128 weight scales).

Codes and scales must match bit for bit; GEMM elements must satisfy
|C_gpu - C_ref| <= 8e-3 |C_ref| + 1e-4 sum_k |a~_ik b~_jk|."""
import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import assert_within_bound, device, host, sample_rows, to_dev

pytestmark = pytest.mark.gpu


def _gpu_quant(x, mode):
    q, s = bq.dg_quantize_fp8_1x128(x, mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return host(q), host(s)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(1, 128), (7, 300), (130, 1000), (257, 2048), (3, 5), (80000, 100), (30000, 300)])
def test_quantize_fp32_bit_exact(oracle_mod, mode, shape):
    x = synthetic.lognormal_rows(shape, seed=shape[0] * 13 + shape[1])
    x[0, : min(3, shape[1])] = 0.0
    if shape[0] > 2:
        x[1, :] = 0.0
        x[2, 0] = -0.0
    q, s = _gpu_quant(to_dev(x, device()), mode)
    qr, sr = oracle_mod.quantize_1x128(x, mode)
    assert np.array_equal(s, sr)
    assert np.array_equal(q, qr)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(5, 128), (64, 777), (300, 4096), (80000, 100), (30000, 300)])
def test_quantize_bf16_bit_exact(oracle_mod, mode, shape):
    """bfloat16 input: the oracle gets the exact FP32 values of the same bf16s."""
    x = torch.from_numpy(synthetic.lognormal_rows(shape, seed=shape[1] + 5)).to(torch.bfloat16)
    q, s = _gpu_quant(x.to(device()), mode)
    qr, sr = oracle_mod.quantize_1x128(x.float().numpy(), mode)
    assert np.array_equal(s, sr)
    assert np.array_equal(q, qr)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_unaligned_and_strided(oracle_mod, dtype):
    """A column slice starting one element in (scalar path) and a padded row stride."""
    full = torch.from_numpy(synthetic.normal((40, 520), seed=77)).to(dtype)
    xs = full[:, 1:301]
    q, s = _gpu_quant(full.to(device())[:, 1:301], 0)   # device view one element in, ld_x = 520
    qr, sr = oracle_mod.quantize_1x128(xs.float().numpy(), 0)
    assert np.array_equal(s, sr) and np.array_equal(q, qr)
    xd = full.to(device())[:, :384]            # ld_x = 520 > cols
    q2, s2 = _gpu_quant(xd, 1)
    qr2, sr2 = oracle_mod.quantize_1x128(full[:, :384].float().numpy(), 1)
    assert np.array_equal(s2, sr2) and np.array_equal(q2, qr2)


def test_quantize_16384x7168_sampled_rows(oracle_mod):
    """The benchmark activation size, 16384 x 7168 FP32, checked on sampled rows."""
    r, c = synthetic.QUANT_SHAPE
    x = synthetic.normal((r, c), seed=synthetic.seed_for(3, 99))
    q, s = _gpu_quant(to_dev(x, device()), 0)
    rows = sample_rows(r, 24, seed=3)
    qr, sr = oracle_mod.quantize_1x128(x[rows], 0)
    assert np.array_equal(s[rows], sr) and np.array_equal(q[rows], qr)


def _operands(oracle_mod, m, n, k, seed, mode=0):
    a = synthetic.lognormal_rows((m, k), seed)
    b = synthetic.lognormal_rows((n, k), seed + 500)
    qa, sa = oracle_mod.quantize_1x128(a, mode)
    qb, sb = oracle_mod.quantize(b, mode)
    return qa, sa, qb, sb


def _gemm(qa, sa, qb, sb, mode=0):
    dev = device()
    m, n = qa.shape[0], qb.shape[0]
    ldc = (n + 7) // 8 * 8                    # the C row stride must be a multiple of 8
    c = torch.full((m, ldc), float("nan"), dtype=torch.bfloat16, device=dev)[:, :n]
    bq.dg_fp8_gemm_nt_1x128(c, to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev), to_dev(sb, dev), mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return c


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("m,n,k", [
    (1, 256, 384), (16, 2112, 512), (100, 300, 640), (128, 1024, 1536),   # M <= 128: cluster split-K
    (129, 136, 384), (300, 130, 1152), (513, 257, 256), (1024, 2112, 2048),  # M > 128: CTA pairs
])
def test_gemm_rowwise(oracle_mod, mode, m, n, k):
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=m * 3 + n + k, mode=mode)
    c = _gemm(qa, sa, qb, sb, mode)
    rows = None if m <= 300 else sample_rows(m, 32, seed=m)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows, a_1x128=True)
    got = c if rows is None else c[torch.as_tensor(rows, device=c.device)]
    assert_within_bound(got, ref, mag, f"1x128 {m}x{n}x{k} mode {mode}")


def test_gemm_rowwise_one_sm_fallback(oracle_mod):
    """One SM allowed: the 1-SM kernel with per-row scales."""
    qa, sa, qb, sb = _operands(oracle_mod, 640, 768, 512, seed=91)
    try:
        bq.dg_set_num_sms(1)
        c = _gemm(qa, sa, qb, sb)
    finally:
        bq.dg_set_num_sms(0)
    rows = sample_rows(640, 24, seed=1)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows, a_1x128=True)
    assert_within_bound(c[torch.as_tensor(rows, device=c.device)], ref, mag, "1x128 one SM")


def test_gemm_rowwise_equals_block_gemm_when_rows_share_scales(oracle_mod):
    """Rows of each 128-row block given their block's scale: the per-row call
    must equal the 128x128-scale call bit for bit (same kernel arithmetic)."""
    m, n, k = 384, 512, 1024
    a = synthetic.lognormal_rows((m, k), 61)
    b = synthetic.lognormal_rows((n, k), 62)
    qa, sblk = oracle_mod.quantize(a)
    qb, sb = oracle_mod.quantize(b)
    srow = np.repeat(sblk, 128, axis=0)[:m]
    dev = device()
    c1 = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    c2 = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_gemm_nt(c1, to_dev(qa, dev), to_dev(qb, dev), to_dev(sblk, dev), to_dev(sb, dev))
    bq.dg_fp8_gemm_nt_1x128(c2, to_dev(qa, dev), to_dev(qb, dev), to_dev(srow, dev), to_dev(sb, dev))
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_llm_shape_rowwise(oracle_mod):
    """M = 4096, N = 7168, K = 2048 with row-wise activation scales."""
    m, n, k = synthetic.LLM_M, 7168, 2048
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=synthetic.seed_for(2, 40))
    c = _gemm(qa, sa, qb, sb)
    rows = sample_rows(m, 24, seed=5)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows, a_1x128=True)
    assert_within_bound(c[torch.as_tensor(rows, device=c.device)], ref, mag, "1x128 LLM")


def test_grouped_rowwise(oracle_mod):
    k, n, g = 512, 640, 3
    sizes = np.array([300, 5, 640])
    m_idx, _ = synthetic.moe_layout(sizes)
    m_idx = np.concatenate([m_idx, np.full(128, -1, np.int32)])
    a = synthetic.lognormal_rows((m_idx.size, k), 71)
    b = synthetic.lognormal_rows((g * n, k), 72).reshape(g, n, k)
    qa, sa = oracle_mod.quantize_1x128(a)
    qs, ss = zip(*[oracle_mod.quantize(b[i]) for i in range(g)])
    qb, sb = np.stack(qs), np.stack(ss)
    dev = device()
    c = torch.full((m_idx.size, n), float("nan"), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_grouped_gemm_contiguous_1x128(c, to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev),
                                            to_dev(sb, dev), to_dev(m_idx, dev))
    assert bq.dg_get_device_status() == bq.DG_OK
    ref, mag = oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, m_idx, a_1x128=True)
    assert_within_bound(c, ref, mag, "grouped 1x128")
    assert torch.count_nonzero(c[torch.as_tensor(m_idx < 0, device=c.device)]) == 0


def test_bf16_activations_end_to_end(oracle_mod):
    """bf16 activations -> GPU row-wise quantizer -> GEMM, against the oracle
    chain on the same bf16 values."""
    m, n, k = 200, 384, 1024
    x = torch.from_numpy(synthetic.lognormal_rows((m, k), 81)).to(torch.bfloat16)
    b = synthetic.lognormal_rows((n, k), 82)
    qb, sb = oracle_mod.quantize(b)
    dev = device()
    qa_d, sa_d = bq.dg_quantize_fp8_1x128(x.to(dev))
    c = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_gemm_nt_1x128(c, qa_d, to_dev(qb, dev), sa_d, to_dev(sb, dev))
    assert bq.dg_get_device_status() == bq.DG_OK
    qa, sa = oracle_mod.quantize_1x128(x.float().numpy())
    assert np.array_equal(host(qa_d), qa) and np.array_equal(host(sa_d), sa)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, a_1x128=True)
    assert_within_bound(c, ref, mag, "bf16 end to end")
