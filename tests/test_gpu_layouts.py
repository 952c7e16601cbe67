"""GPU parity of the dense GEMM in the layouts NT, TN, NN, TT and of the
K-grouped TN GEMM (pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1: all four
layouts from SM100 on; §3.2: grouping along K), through the C ABI, against
the oracle.

* Exact cases: operand values -2..2 with power-of-two scales make the FP32
  accumulator exact, so the bf16 output must equal the oracle's result
  rounded to bf16, bit for bit, on every kernel path.
* General cases: |C_gpu - C_ref| <= 8e-3 |C_ref| + 1e-4 sum_k |a~ b~|."""
import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import assert_within_bound, device, sample_rows, to_dev

pytestmark = pytest.mark.gpu

CODES = np.array([0xC0, 0xB8, 0x00, 0x38, 0x40], np.uint8)  # -2, -1, 0, 1, 2


def _exact_logical(m, n, k, seed):
    rng = np.random.default_rng(seed)
    qa = CODES[rng.integers(0, 5, (m, k))]          # logical A [M, K]
    qb = CODES[rng.integers(0, 5, (n, k))]          # logical B^T [N, K]
    sa = np.exp2(rng.integers(-2, 3, (-(-m // 128), k // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-2, 3, (-(-n // 128), k // 128))).astype(np.float32)
    return qa, sa, qb, sb


def _stored(qa, qb, layout):
    a_st = np.ascontiguousarray(qa.T) if layout[0] == "T" else qa
    b_st = np.ascontiguousarray(qb.T) if layout[1] == "N" else qb
    return a_st, b_st


def _padded(x, dev):
    """x on the device with its row stride rounded up to 16 bytes (the TMA rule)."""
    rows, cols = x.shape
    buf = torch.zeros((rows, -(-cols // 16) * 16), dtype=torch.uint8, device=dev)
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return buf[:, :cols]


def _run(a_st, sa, b_st, sb, m, n, layout, mode):
    dev = device()
    c = torch.full((m, -(-n // 8) * 8), float("nan"), dtype=torch.bfloat16, device=dev)[:, :n]
    bq.dg_fp8_gemm(c, _padded(a_st, dev), _padded(b_st, dev), to_dev(sa, dev), to_dev(sb, dev), layout, mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return c


def _bf16_bits(x):
    t = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.asarray(x, np.float32))
    return t.cpu().to(torch.bfloat16).view(torch.int16)


# M > 128: CTA pairs (FP32 promotion with mode 0, block-scaled MMA with mode 1);
# M <= 128: cluster split-K.
SHAPES = [(256, 256, 512), (300, 200, 1024), (129, 136, 384), (513, 257, 768), (1, 384, 256), (100, 300, 640)]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("layout", ["NT", "TN", "NN", "TT"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_bit_identical(oracle_mod, shape, layout, mode):
    m, n, k = shape
    qa, sa, qb, sb = _exact_logical(m, n, k, seed=m + 3 * n + k)
    a_st, b_st = _stored(qa, qb, layout)
    c = _run(a_st, sa, b_st, sb, m, n, layout, mode)
    ref, _ = oracle_mod.gemm_layout(a_st, sa, b_st, sb, layout)
    got, want = _bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32))
    assert torch.equal(got, want), f"{int((got != want).sum())} outputs differ"


# Decode shapes whose plans cover the cluster reduction's K splits 2, 4, 5, 6 and 8
# (column shares of uneven width, pushed to their owners), a ragged last tile and
# odd row counts, plus a plan without a K split.
DECODE_SHAPES = [(16, 7168, 16384), (64, 7168, 16384), (128, 7168, 16384), (128, 2112, 7168), (16, 1536, 7168),
                 (5, 4000, 2048), (77, 2000, 4096), (16, 24576, 1536)]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_decode_splits(oracle_mod, shape, mode):
    m, n, k = shape
    qa, sa, qb, sb = _exact_logical(m, n, k, seed=7 * m + n + k)
    c = _run(qa, sa, qb, sb, m, n, "NT", mode)
    ref, _ = oracle_mod.gemm_layout(qa, sa, qb, sb, "NT")
    got, want = _bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32))
    assert torch.equal(got, want), f"{int((got != want).sum())} outputs differ"


@pytest.mark.parametrize("cap", [4, 10])
@pytest.mark.parametrize("shape", [(16, 7168, 4096), (77, 2000, 2048), (128, 4096, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_exact_decode_many_tiles_per_cluster(oracle_mod, shape, cap):
    """An SM cap leaves a few clusters for many tiles: every cluster's
    reduction buffers and barriers go through many phases (tile after tile)."""
    m, n, k = shape
    qa, sa, qb, sb = _exact_logical(m, n, k, seed=3 * m + cap)
    try:
        bq.dg_set_num_sms(cap)
        c = _run(qa, sa, qb, sb, m, n, "NT", 0)
    finally:
        bq.dg_set_num_sms(0)
    ref, _ = oracle_mod.gemm_layout(qa, sa, qb, sb, "NT")
    got, want = _bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32))
    assert torch.equal(got, want), f"{int((got != want).sum())} outputs differ"


@pytest.mark.parametrize("layout", ["TN", "NN", "TT"])
def test_exact_one_sm_fallback(oracle_mod, layout):
    """One SM allowed: the 1-SM kernel (256-column tiles) with MN-major operands."""
    m, n, k = 640, 700, 512
    qa, sa, qb, sb = _exact_logical(m, n, k, seed=11)
    a_st, b_st = _stored(qa, qb, layout)
    try:
        bq.dg_set_num_sms(1)
        c = _run(a_st, sa, b_st, sb, m, n, layout, 0)
    finally:
        bq.dg_set_num_sms(0)
    ref, _ = oracle_mod.gemm_layout(a_st, sa, b_st, sb, layout)
    assert torch.equal(_bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32)))


def _random_logical(oracle_mod, m, n, k, seed, mode):
    qa, sa = oracle_mod.quantize(synthetic.lognormal_rows((m, k), seed), mode)
    qb, sb = oracle_mod.quantize(synthetic.lognormal_rows((n, k), seed + 1), mode)
    return qa, sa, qb, sb


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("layout", ["TN", "NN", "TT"])
@pytest.mark.parametrize("shape", [(512, 640, 1024), (64, 1000, 768)], ids=lambda s: "x".join(map(str, s)))
def test_random_within_bound(oracle_mod, shape, layout, mode):
    m, n, k = shape
    qa, sa, qb, sb = _random_logical(oracle_mod, m, n, k, seed=m + n, mode=mode)
    a_st, b_st = _stored(qa, qb, layout)
    c = _run(a_st, sa, b_st, sb, m, n, layout, mode)
    ref, mag = oracle_mod.gemm_layout(a_st, sa, b_st, sb, layout)
    assert_within_bound(c, ref, mag, f"{layout} {m}x{n}x{k} mode {mode}")


def test_padded_strides(oracle_mod):
    """MN-major operands inside wider buffers: ld_a > M, ld_b > N."""
    m, n, k = 200, 150, 512
    qa, sa, qb, sb = _exact_logical(m, n, k, seed=21)
    dev = device()
    a_buf = torch.zeros((k, 256), dtype=torch.uint8, device=dev)
    a_buf[:, :m] = torch.from_numpy(qa.T.copy()).to(dev)
    b_buf = torch.zeros((k, 192), dtype=torch.uint8, device=dev)
    b_buf[:, :n] = torch.from_numpy(qb.T.copy()).to(dev)
    with pytest.raises(ValueError):  # a [K, 256] does not describe M = 200
        bq.dg_fp8_gemm(torch.empty((m, n), dtype=torch.bfloat16, device=dev), a_buf, b_buf[:, :n],
                       to_dev(sa, dev), to_dev(sb, dev), "TN")
    c = torch.empty((m, 152), dtype=torch.bfloat16, device=dev)[:, :n]
    bq.dg_fp8_gemm(c, a_buf[:, :m], b_buf[:, :n], to_dev(sa, dev), to_dev(sb, dev), "TN")
    assert bq.dg_get_device_status() == bq.DG_OK
    ref, _ = oracle_mod.gemm_layout(qa.T.copy(), sa, qb.T.copy(), sb, "TN")
    assert torch.equal(_bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32)))


def test_llm_shape_nn_sampled(oracle_mod):
    """M = 4096, N = 7168, K = 2048 with B stored [K][N], checked on sampled rows."""
    m, n, k = synthetic.LLM_M, 7168, 2048
    qa, sa, qb, sb = _random_logical(oracle_mod, m, n, k, seed=synthetic.seed_for(2, 80), mode=0)
    a_st, b_st = _stored(qa, qb, "NN")
    c = _run(a_st, sa, b_st, sb, m, n, "NN", 0)
    rows = sample_rows(m, 24, seed=7)
    ref, mag = oracle_mod.gemm_layout(a_st, sa, b_st, sb, "NN", rows=rows)
    assert_within_bound(c[torch.as_tensor(rows, device=c.device)], ref, mag, "NN LLM")


def _k_grouped(oracle_mod, m, n, sizes, exact, seed, mode=0):
    k_tot = sum(sizes)
    if exact:
        qa, sa, qb, sb = _exact_logical(m, n, k_tot, seed)
    else:
        qa, sa, qb, sb = _random_logical(oracle_mod, m, n, k_tot, seed, mode)
    a_st, b_st = np.ascontiguousarray(qa.T), np.ascontiguousarray(qb.T)   # [K_tot, M], [K_tot, N]
    dev = device()
    c = torch.full((len(sizes), m, n), float("nan"), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_k_grouped_gemm_tn(c, _padded(a_st, dev), _padded(b_st, dev), to_dev(sa, dev), to_dev(sb, dev), sizes,
                                mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return c, (a_st, sa, b_st, sb)


@pytest.mark.parametrize("mode", [0, 1])
def test_k_grouped_exact(oracle_mod, mode):
    sizes = [256, 0, 384, 128, 1024]
    c, (a_st, sa, b_st, sb) = _k_grouped(oracle_mod, 300, 200, sizes, exact=True, seed=31, mode=mode)
    ref, _ = oracle_mod.k_grouped_gemm_tn(a_st, sa, b_st, sb, sizes)
    assert torch.equal(_bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32)))


@pytest.mark.parametrize("mode", [0, 1])
def test_k_grouped_small_m_exact(oracle_mod, mode):
    sizes = [128, 512]
    c, (a_st, sa, b_st, sb) = _k_grouped(oracle_mod, 96, 640, sizes, exact=True, seed=33, mode=mode)
    ref, _ = oracle_mod.k_grouped_gemm_tn(a_st, sa, b_st, sb, sizes)
    assert torch.equal(_bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32)))


@pytest.mark.parametrize("mode", [0, 1])
def test_k_grouped_many_ranges_exact(oracle_mod, mode):
    """Twenty ranges of 0-384 rows (empty ones among them) in one launch: the
    units of consecutive ranges share the pairs, and a pair row (M = 384) and a
    column tile (N = 320) cross the matrix edges of every output. With
    power-of-two scales, ranges of one and three K blocks end on a half-filled
    two-block stage of the block-scaled kernel."""
    rng = np.random.default_rng(7)
    sizes = [int(v) * 128 for v in rng.integers(0, 4, 20)]
    sizes[0], sizes[-1] = 0, 256
    c, (a_st, sa, b_st, sb) = _k_grouped(oracle_mod, 384, 320, sizes, exact=True, seed=37, mode=mode)
    ref, _ = oracle_mod.k_grouped_gemm_tn(a_st, sa, b_st, sb, sizes)
    assert torch.equal(_bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32)))


@pytest.mark.parametrize("mode", [0, 1])
def test_k_grouped_padded_output_rows_untouched(oracle_mod, mode):
    """One launch writing C [G][M][ld_c] with ld_c > N: every value of the
    padding columns stays as it was (the 3-D output map clips at N and at M)."""
    sizes = [256, 0, 128, 384]
    m, n, ld = 300, 200, 232
    k_tot = sum(sizes)
    qa, sa, qb, sb = _exact_logical(m, n, k_tot, 43)
    a_st, b_st = np.ascontiguousarray(qa.T), np.ascontiguousarray(qb.T)
    dev = device()
    c_full = torch.full((len(sizes), m, ld), float("nan"), dtype=torch.bfloat16, device=dev)
    c = c_full[:, :, :n]
    bq.dg_fp8_k_grouped_gemm_tn(c, _padded(a_st, dev), _padded(b_st, dev), to_dev(sa, dev), to_dev(sb, dev), sizes,
                                mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    ref, _ = oracle_mod.k_grouped_gemm_tn(a_st, sa, b_st, sb, sizes)
    assert torch.equal(_bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32)))
    assert torch.isnan(c_full[:, :, n:].float()).all()


@pytest.mark.parametrize("mode", [0, 1])
def test_k_grouped_more_ranges_than_one_launch_holds_exact(oracle_mod, mode):
    """300 non-empty ranges: past the 256 a single launch carries, the ranges
    run one after another."""
    sizes = [128] * 300
    sizes[5] = 0
    c, (a_st, sa, b_st, sb) = _k_grouped(oracle_mod, 256, 128, sizes, exact=True, seed=39, mode=mode)
    ref, _ = oracle_mod.k_grouped_gemm_tn(a_st, sa, b_st, sb, sizes)
    assert torch.equal(_bf16_bits(c.float()), _bf16_bits(ref.astype(np.float32)))


@pytest.mark.parametrize("mode", [0, 1])
def test_k_grouped_moe_weight_gradient_sampled(oracle_mod, mode):
    """8 experts, token counts padded to 128 (the MoE layout's group sizes),
    M = 2048 hidden x N = 1408 intermediate: the shape of a weight gradient."""
    mo = synthetic.MOE
    sizes = synthetic.moe_group_sizes(mo["experts"], 2048, 2, 1)
    sizes = [int(-(-s // 128) * 128) for s in sizes]
    m, n = 2048, 1408
    c, (a_st, sa, b_st, sb) = _k_grouped(oracle_mod, m, n, sizes, exact=False, seed=35, mode=mode)
    rows = sample_rows(m, 16, seed=3)
    ref, mag = oracle_mod.k_grouped_gemm_tn(a_st, sa, b_st, sb, sizes, rows=rows)
    idx = torch.as_tensor(rows, device=c.device)
    for g in range(len(sizes)):
        assert_within_bound(c[g][idx], ref[g], mag[g], f"k-grouped group {g}")
