"""GPU parity of the M-grouped contiguous GEMM (MoE experts) against the CPU
oracle, through the C ABI (pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §2.3,
§3.2, §3.3: grouped GEMM along M, rows aligned to
get_mk_alignment_for_contiguous_layout()). Operands come from the oracle's
quantizer; padding rows (index -1) must come out as zeros."""
import ctypes

import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import assert_within_bound, device, rows_per_block, to_dev

pytestmark = pytest.mark.gpu


def _quantize_experts(oracle_mod, b, mode=0):
    qs, ss = zip(*[oracle_mod.quantize(b[g], mode) for g in range(b.shape[0])])
    return np.stack(qs), np.stack(ss)


def _run(qa, sa, qb, sb, m_idx, mode=0):
    dev = device()
    m_tot, n = qa.shape[0], qb.shape[1]
    c = torch.full((m_tot, n), float("nan"), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_grouped_gemm_contiguous(c, to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev),
                                      to_dev(sb, dev), to_dev(m_idx, dev), mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return c


def _rows_per_group(m_idx, per_group, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for g in np.unique(m_idx):
        idx = np.flatnonzero(m_idx == g)
        rows.append(idx[[0, -1]])
        rows.append(rng.choice(idx, size=min(per_group, idx.size), replace=False))
    return np.unique(np.concatenate(rows)).astype(np.int64)


def test_alignment_query():
    device()
    assert bq.dg_get_mk_alignment_for_contiguous_layout() == 128


@pytest.mark.parametrize("mode", [0, 1])
def test_small_groups_with_empty_expert_and_padding(oracle_mod, mode):
    k, n, g = 384, 200, 4
    sizes = np.array([5, 0, 130, 128])
    m_idx, offs = synthetic.moe_layout(sizes)
    m_idx = np.concatenate([m_idx, np.full(128, -1, np.int32)])   # one block of pure padding
    a = synthetic.lognormal_rows((m_idx.size, k), seed=201)
    b = synthetic.lognormal_rows((g * n, k), seed=202).reshape(g, n, k)
    qa, sa = oracle_mod.quantize(a, mode)
    qa[m_idx < 0] = 0x7F                       # NaN codes in padding rows must not leak
    qb, sb = _quantize_experts(oracle_mod, b, mode)
    c = _run(qa, sa, qb, sb, m_idx, mode)
    ref, mag = oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, m_idx)
    assert_within_bound(c, ref, mag, "small grouped")
    assert torch.count_nonzero(c[torch.as_tensor(m_idx < 0, device=c.device)]) == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_moe_8_experts_11008x4096(oracle_mod, mode):
    """8 experts, K = 4096 hidden, N = 11008 intermediate, 4096 tokens top-2,
    with FP32 and with power-of-two block scales."""
    mo = synthetic.MOE
    a, b, m_idx, sizes = synthetic.moe_inputs(seed=0, experts=mo["experts"], tokens=mo["tokens"],
                                               topk=mo["topk"], hidden=mo["hidden"],
                                               intermediate=mo["intermediate"])
    assert m_idx.size == 8960 and list(sizes) == [1033, 1551, 36, 6, 873, 2462, 1027, 1204]
    qa, sa = oracle_mod.quantize(a, mode)
    qb, sb = _quantize_experts(oracle_mod, b, mode)
    c = _run(qa, sa, qb, sb, m_idx, mode)
    # Every 128-row block (each expert's blocks, its partial last block) plus
    # each expert's first and last rows.
    rows = np.union1d(_rows_per_group(m_idx, 6, seed=1), rows_per_block(m_idx.size, 128, seed=2, valid=m_idx >= 0))
    ref, mag = oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, m_idx, rows=rows)
    assert_within_bound(c[torch.as_tensor(rows, device=c.device)], ref, mag, "MoE 8x11008x4096")
    assert torch.count_nonzero(c[torch.as_tensor(m_idx < 0, device=c.device)]) == 0


def test_grouped_few_sms(oracle_mod):
    """Grouped GEMM with many tiles per persistent CTA."""
    k, n, g = 512, 640, 3
    sizes = np.array([300, 5, 640])
    m_idx, _ = synthetic.moe_layout(sizes)
    a = synthetic.lognormal_rows((m_idx.size, k), seed=205)
    b = synthetic.lognormal_rows((g * n, k), seed=206).reshape(g, n, k)
    qa, sa = oracle_mod.quantize(a)
    qb, sb = _quantize_experts(oracle_mod, b)
    try:
        bq.dg_set_num_sms(2)
        c = _run(qa, sa, qb, sb, m_idx)
    finally:
        bq.dg_set_num_sms(0)
    ref, mag = oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, m_idx)
    assert_within_bound(c, ref, mag, "grouped, 2 SMs")


def test_grouped_matches_dense_bitwise(oracle_mod):
    """A grouped call with one expert per 128-row block equals the dense calls on
    each expert's rows, bit for bit."""
    k, n = 256, 384
    sizes = np.array([128, 256])
    m_idx, offs = synthetic.moe_layout(sizes)
    a = synthetic.normal((m_idx.size, k), seed=203)
    b = synthetic.normal((2 * n, k), seed=204).reshape(2, n, k)
    qa, sa = oracle_mod.quantize(a)
    qb, sb = _quantize_experts(oracle_mod, b)
    c = _run(qa, sa, qb, sb, m_idx)
    dev = device()
    for g in range(2):
        lo, hi = offs[g], offs[g + 1]
        cd = torch.empty((hi - lo, n), dtype=torch.bfloat16, device=dev)
        bq.dg_fp8_gemm_nt(cd, to_dev(qa[lo:hi], dev), to_dev(qb[g], dev),
                          to_dev(sa[lo // 128:hi // 128], dev), to_dev(sb[g], dev))
        assert torch.equal(cd.view(torch.int16), c[lo:hi].view(torch.int16))


@pytest.mark.parametrize("mode", [0, 1])
def test_expert_id_past_the_last_group_is_zeroed_and_reported(oracle_mod, mode):
    """A 128-row block whose expert id equals num_groups reads no B or sb of
    that id, comes out as zeros, and sets DG_ERR_BAD_GROUP. B and sb are
    allocated for one expert more than num_groups, so that even a read of the
    bad id would stay inside the allocations."""
    dev = device()
    k, n, g = 256, 256, 2
    m_idx = np.concatenate([np.full(128, 0, np.int32), np.full(128, g, np.int32),
                            np.full(100, 1, np.int32), np.full(28, -1, np.int32)])
    a = synthetic.lognormal_rows((m_idx.size, k), seed=211)
    b = synthetic.lognormal_rows(((g + 1) * n, k), seed=212).reshape(g + 1, n, k)
    qa, sa = oracle_mod.quantize(a, mode)
    qb, sb = _quantize_experts(oracle_mod, b, mode)
    c = torch.full((m_idx.size, n), float("nan"), dtype=torch.bfloat16, device=dev)
    # Every device buffer stays referenced until the kernel has run.
    qa_d, sa_d, qb_d, sb_d, mi_d = (to_dev(v, dev) for v in (qa, sa, qb, sb, m_idx))
    rc = bq.lib().dg_fp8_grouped_gemm_contiguous(
        ctypes.c_void_p(c.data_ptr()), n, ctypes.c_void_p(qa_d.data_ptr()), k,
        ctypes.c_void_p(sa_d.data_ptr()), ctypes.c_void_p(qb_d.data_ptr()),
        ctypes.c_void_p(sb_d.data_ptr()), g, ctypes.c_void_p(mi_d.data_ptr()),
        m_idx.size, n, k, mode, ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert rc == bq.DG_OK
    assert bq.dg_get_device_status() == bq.DG_ERR_BAD_GROUP
    assert bq.dg_get_device_status() == bq.DG_OK          # taken and cleared
    got = c.float().cpu().numpy()
    assert np.all(got[128:256] == 0.0)
    good = np.where(m_idx == g, -1, m_idx).astype(np.int32)
    ref, mag = oracle_mod.grouped_gemm_contiguous(qa, sa, qb[:g], sb[:g], good)
    assert_within_bound(c, ref, mag, "grouped with a bad expert id")
