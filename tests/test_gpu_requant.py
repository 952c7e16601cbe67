"""GPU parity of the GEMMs whose epilogue requantizes the FP32 accumulators to
E4M3 codes plus block scales, through the C ABI, against the oracle
(lpnh.cn DeepGEMM walkthrough §2.2: quantize on demand at write-back; §6: fuse
the scale computation into the kernel; §4.2: the quantization steps).

* Exact cases: operand codes of -2..2 and power-of-two scales make every
  partial sum and every FP32 accumulation exact, so codes and scales must
  equal the oracle's bit for bit on every kernel path.
* General cases: the accumulator carries rounding error, so each code must be
  the E4M3 rounding of a value within the GEMM bound of the exact result and
  each scale within that bound of the exact block max / 448
  (parity.assert_requant_within_bound)."""
import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import assert_requant_within_bound, device, host, sample_rows, to_dev

pytestmark = pytest.mark.gpu


def _exact_operands(m, n, k, seed, a_rows=128, g=None):
    """Codes of -2, -1, 0, 1, 2 with power-of-two scales in [2^-2, 2^2]."""
    rng = np.random.default_rng(seed)
    codes = np.array([0xC0, 0xB8, 0x00, 0x38, 0x40], np.uint8)
    qa = codes[rng.integers(0, 5, (m, k))]
    nb = g if g is not None else 1
    qb = codes[rng.integers(0, 5, (nb, n, k))]
    sa = np.exp2(rng.integers(-2, 3, ((m if a_rows == 1 else -(-m // 128)), k // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-2, 3, (nb, -(-n // 128), k // 128))).astype(np.float32)
    if g is None:
        return qa, sa, qb[0], sb[0]
    return qa, sa, qb, sb


def _run_dense(qa, sa, qb, sb, in_mode, block_rows, out_mode):
    dev = device()
    cq, cs = bq.dg_fp8_gemm_nt_requant(to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev), to_dev(sb, dev),
                                       in_mode, block_rows, out_mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return host(cq), host(cs)


# (M, N, K): M > 128 runs on CTA pairs (FP32 promotion for in_mode 0, the
# block-scaled MMA for in_mode 1), M <= 128 on the split-K kernel.
EXACT_SHAPES = [(256, 256, 512), (300, 200, 1024), (129, 136, 384), (1, 384, 256), (100, 300, 640)]


@pytest.mark.parametrize("out_mode", [0, 1])
@pytest.mark.parametrize("block_rows", [1, 128])
@pytest.mark.parametrize("in_mode", [0, 1])
@pytest.mark.parametrize("shape", EXACT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_bit_identical(oracle_mod, shape, in_mode, block_rows, out_mode):
    m, n, k = shape
    qa, sa, qb, sb = _exact_operands(m, n, k, seed=m + 7 * n + k)
    q, s = _run_dense(qa, sa, qb, sb, in_mode, block_rows, out_mode)
    qr, sr, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, block_rows, out_mode)
    assert np.array_equal(s, sr), f"scales differ at {np.argwhere(s != sr)[:5].tolist()}"
    assert np.array_equal(q, qr), f"codes differ at {np.argwhere(q != qr)[:5].tolist()}"


# Decode shapes: the split-K kernel reduces over a cluster and exchanges the
# block maxima between its CTAs (split >= 2 for these K).
DECODE_SHAPES = [(1, 7168, 4096), (16, 2304, 8192), (128, 1152, 4096), (77, 500, 2048)]


@pytest.mark.parametrize("out_mode", [0, 1])
@pytest.mark.parametrize("block_rows", [1, 128])
@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_decode_cluster(oracle_mod, shape, block_rows, out_mode):
    m, n, k = shape
    qa, sa, qb, sb = _exact_operands(m, n, k, seed=m + n)
    q, s = _run_dense(qa, sa, qb, sb, 0, block_rows, out_mode)
    qr, sr, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, block_rows, out_mode)
    assert np.array_equal(s, sr), f"scales differ at {np.argwhere(s != sr)[:5].tolist()}"
    assert np.array_equal(q, qr), f"codes differ at {np.argwhere(q != qr)[:5].tolist()}"


@pytest.mark.parametrize("cap", [4, 10])
@pytest.mark.parametrize("shape", [(16, 7168, 4096), (77, 2000, 2048)], ids=lambda s: "x".join(map(str, s)))
def test_exact_decode_many_tiles_per_cluster(oracle_mod, shape, cap):
    """An SM cap leaves a few clusters for many tiles: every cluster's
    reduction buffers and barriers go through many phases (tile after tile)."""
    m, n, k = shape
    qa, sa, qb, sb = _exact_operands(m, n, k, seed=5 * m + cap)
    try:
        bq.dg_set_num_sms(cap)
        q, s = _run_dense(qa, sa, qb, sb, 0, 1, 0)
    finally:
        bq.dg_set_num_sms(0)
    qr, sr, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, 1, 0)
    assert np.array_equal(s, sr), f"scales differ at {np.argwhere(s != sr)[:5].tolist()}"
    assert np.array_equal(q, qr), f"codes differ at {np.argwhere(q != qr)[:5].tolist()}"


@pytest.mark.parametrize("block_rows", [1, 128])
def test_random_decode_cluster(oracle_mod, block_rows):
    m, n, k = 128, 7168, 16384
    qa, sa, qb, sb = _random_operands(oracle_mod, m, n, k, seed=91)
    q, s = _run_dense(qa, sa, qb, sb, 0, block_rows, 0)
    c, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_requant_within_bound(q, s, c, mag, block_rows, False, f"decode 128x7168x16384 rows {block_rows}",
                                oracle_mod)


@pytest.mark.parametrize("block_rows", [1, 128])
def test_exact_one_sm_fallback_wide_tiles(oracle_mod, block_rows):
    """One SM allowed: the 1-SM kernel with 256-column tiles (M > 256)."""
    qa, sa, qb, sb = _exact_operands(640, 700, 512, seed=5)
    try:
        bq.dg_set_num_sms(1)
        q, s = _run_dense(qa, sa, qb, sb, 0, block_rows, 0)
    finally:
        bq.dg_set_num_sms(0)
    qr, sr, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, block_rows, 0)
    assert np.array_equal(s, sr) and np.array_equal(q, qr)


@pytest.mark.parametrize("block_rows", [1, 128])
def test_exact_grouped(oracle_mod, block_rows):
    sizes = np.array([300, 0, 5, 256])
    m_idx, _ = synthetic.moe_layout(sizes)
    m_idx = np.concatenate([m_idx, np.full(128, -1, np.int32)])
    k, n, g = 512, 384, 4
    qa, sa, qb, sb = _exact_operands(m_idx.size, n, k, seed=17, g=g)
    dev = device()
    cq, cs = bq.dg_fp8_grouped_gemm_contiguous_requant(to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev),
                                                       to_dev(sb, dev), to_dev(m_idx, dev), 0, block_rows, 0)
    assert bq.dg_get_device_status() == bq.DG_OK
    qr, sr, _, _ = oracle_mod.grouped_gemm_requant(qa, sa, qb, sb, m_idx, block_rows, 0)
    assert np.array_equal(host(cs), sr) and np.array_equal(host(cq), qr)


def _random_operands(oracle_mod, m, n, k, seed, a_1x128=False, in_mode=0):
    a = synthetic.lognormal_rows((m, k), seed)
    b = synthetic.lognormal_rows((n, k), seed + 1)
    qa, sa = oracle_mod.quantize_1x128(a, in_mode) if a_1x128 else oracle_mod.quantize(a, in_mode)
    qb, sb = oracle_mod.quantize(b, in_mode)
    return qa, sa, qb, sb


@pytest.mark.parametrize("out_mode", [0, 1])
@pytest.mark.parametrize("block_rows", [1, 128])
@pytest.mark.parametrize("in_mode", [0, 1])
@pytest.mark.parametrize("shape", [(513, 257, 768), (64, 1000, 512), (256, 1024, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_random_within_bound(oracle_mod, shape, in_mode, block_rows, out_mode):
    m, n, k = shape
    qa, sa, qb, sb = _random_operands(oracle_mod, m, n, k, seed=m + n + k, in_mode=in_mode)
    q, s = _run_dense(qa, sa, qb, sb, in_mode, block_rows, out_mode)
    c, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_requant_within_bound(q, s, c, mag, block_rows, out_mode == 1,
                                f"{m}x{n}x{k} in {in_mode} rows {block_rows} out {out_mode}", oracle_mod)


@pytest.mark.parametrize("block_rows", [1, 128])
def test_rowwise_activation_scales(oracle_mod, block_rows):
    """sa [M, K/128] (per-row activation scales) in, requantized output out."""
    m, n, k = 300, 520, 1024
    qa, sa, qb, sb = _random_operands(oracle_mod, m, n, k, seed=3, a_1x128=True)
    q, s = _run_dense(qa, sa, qb, sb, 0, block_rows, 0)
    c, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, a_1x128=True)
    assert_requant_within_bound(q, s, c, mag, block_rows, False, "1x128 in", oracle_mod)


def test_llm_shape_sampled(oracle_mod):
    """M = 4096, N = 7168, K = 2048 with per-row output scales, checked on sampled rows."""
    m, n, k = synthetic.LLM_M, 7168, 2048
    qa, sa, qb, sb = _random_operands(oracle_mod, m, n, k, seed=synthetic.seed_for(2, 70))
    q, s = _run_dense(qa, sa, qb, sb, 0, 1, 0)
    rows = sample_rows(m, 24, seed=9)
    c, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows)
    assert_requant_within_bound(q[rows], s[rows], c, mag, 1, False, "LLM rows", oracle_mod)


def test_llm_shape_block_scales_sampled_blocks(oracle_mod):
    """M = 4096, N = 7168, K = 2048 with 128 x 128 output blocks: two whole block rows."""
    m, n, k = synthetic.LLM_M, 7168, 2048
    qa, sa, qb, sb = _random_operands(oracle_mod, m, n, k, seed=synthetic.seed_for(2, 71))
    q, s = _run_dense(qa, sa, qb, sb, 0, 128, 0)
    for mb in (0, 17):
        rows = np.arange(128 * mb, 128 * mb + 128)
        c, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows)
        assert_requant_within_bound(q[rows], s[mb:mb + 1], c, mag, 128, False, f"LLM block row {mb}", oracle_mod)


def test_grouped_random_within_bound(oracle_mod):
    sizes = np.array([200, 7, 0, 390])
    m_idx, _ = synthetic.moe_layout(sizes)
    k, n, g = 768, 640, 4
    a = synthetic.lognormal_rows((m_idx.size, k), 41)
    b = synthetic.lognormal_rows((g * n, k), 42).reshape(g, n, k)
    qa, sa = oracle_mod.quantize(a)
    qs, ss = zip(*[oracle_mod.quantize(b[i]) for i in range(g)])
    qb, sb = np.stack(qs), np.stack(ss)
    dev = device()
    cq, cs = bq.dg_fp8_grouped_gemm_contiguous_requant(to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev),
                                                       to_dev(sb, dev), to_dev(m_idx, dev))
    assert bq.dg_get_device_status() == bq.DG_OK
    c, mag = oracle_mod.grouped_gemm_contiguous(qa, sa, qb, sb, m_idx)
    q, s = host(cq), host(cs)
    assert_requant_within_bound(q, s, c, mag, 1, False, "grouped", oracle_mod)
    pad = m_idx < 0
    assert np.all(q[pad] == 0) and np.all(s[pad] == 1.0)


def test_chain_requantized_output_feeds_next_gemm(oracle_mod):
    """The per-row requantized output of one GEMM is a valid activation for
    the next (sa [M, K/128]): run both on the GPU and check the second against
    the oracle on the GPU's codes and scales."""
    m, n1, k = 256, 512, 768
    qa, sa, qb, sb = _random_operands(oracle_mod, m, n1, k, seed=51)
    dev = device()
    cq, cs = bq.dg_fp8_gemm_nt_requant(to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev), to_dev(sb, dev))
    w = synthetic.lognormal_rows((384, n1), 52)
    qw, sw = oracle_mod.quantize(w)
    c2 = torch.empty((m, 384), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_gemm_nt_1x128(c2, cq.contiguous(), to_dev(qw, dev), cs, to_dev(sw, dev))
    assert bq.dg_get_device_status() == bq.DG_OK
    from parity import assert_within_bound
    ref, mag = oracle_mod.gemm_nt(host(cq.contiguous()), host(cs), qw, sw, a_1x128=True)
    assert_within_bound(c2, ref, mag, "chained GEMM")


def test_output_padding_untouched():
    """Codes beyond column N of a padded row stride keep their old bytes."""
    m, n, k = 300, 200, 256
    rng = np.random.default_rng(1)
    qa = rng.integers(0, 0x70, (m, k)).astype(np.uint8)
    qb = rng.integers(0, 0x70, (n, k)).astype(np.uint8)
    sa = np.ones((3, 2), np.float32)
    sb = np.ones((2, 2), np.float32)
    dev = device()
    for block_rows in (1, 128):
        full = torch.full((m, 224), 0xA5, dtype=torch.uint8, device=dev)
        bq.dg_fp8_gemm_nt_requant(to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev), to_dev(sb, dev),
                                  out_block_rows=block_rows, cq=full[:, :n])
        assert bq.dg_get_device_status() == bq.DG_OK
        assert torch.all(full[:, n:] == 0xA5)


def test_k_zero_writes_zero_codes_and_unit_scales():
    dev = device()
    a = torch.zeros((5, 0), dtype=torch.uint8, device=dev)
    b = torch.zeros((130, 0), dtype=torch.uint8, device=dev)
    sa = torch.zeros((1, 0), dtype=torch.float32, device=dev)
    sb = torch.zeros((2, 0), dtype=torch.float32, device=dev)
    cq = torch.full((5, 144), 7, dtype=torch.uint8, device=dev)[:, :130]
    cs = torch.zeros((5, 2), dtype=torch.float32, device=dev)
    bq.dg_fp8_gemm_nt_requant(a, b, sa, sb, cq=cq, cs=cs)
    assert bq.dg_get_device_status() == bq.DG_OK
    assert torch.all(cq == 0) and torch.all(cs == 1.0)


def _stored_padded(x, dev):
    """x on the device with its row stride rounded up to 16 bytes (the TMA rule)."""
    rows, cols = x.shape
    buf = torch.zeros((rows, -(-cols // 16) * 16), dtype=torch.uint8, device=dev)
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return buf[:, :cols]


@pytest.mark.parametrize("in_mode", [0, 1])
@pytest.mark.parametrize("layout", ["TN", "NN", "TT"])
@pytest.mark.parametrize("shape", [(300, 200, 1024), (16, 2304, 8192), (100, 300, 640)],
                         ids=lambda s: "x".join(map(str, s)))
def test_exact_layouts(oracle_mod, shape, layout, in_mode):
    """Requantized output with MN-major operands: pair kernels (M > 128) and
    the split-K kernel (M <= 128), per-row output scales."""
    m, n, k = shape
    qa, sa, qb, sb = _exact_operands(m, n, k, seed=3 * m + n)
    dev = device()
    a_st = qa.T if layout[0] == "T" else qa
    b_st = qb.T if layout[1] == "N" else qb
    cq, cs = bq.dg_fp8_gemm_requant(_stored_padded(a_st, dev), _stored_padded(b_st, dev), to_dev(sa, dev),
                                    to_dev(sb, dev), m, n, layout, in_mode, 1, 0)
    assert bq.dg_get_device_status() == bq.DG_OK
    qr, sr, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, 1, 0)
    assert np.array_equal(host(cs), sr) and np.array_equal(host(cq), qr)


@pytest.mark.parametrize("layout", ["NT", "TT"])
def test_exact_layouts_rowwise_a_scales_block_output(oracle_mod, layout):
    """Per-row A scales in, 128 x 128 output blocks out, A stored either way
    (B stays [N][K]: NT and TT)."""
    m, n, k = 260, 384, 512
    qa, sa, qb, sb = _exact_operands(m, n, k, seed=77, a_rows=1)
    dev = device()
    a_st = qa.T if layout[0] == "T" else qa
    cq, cs = bq.dg_fp8_gemm_requant(_stored_padded(a_st, dev), to_dev(qb, dev), to_dev(sa, dev), to_dev(sb, dev),
                                    m, n, layout, 0, 128, 0, a_scale_rows=1)
    assert bq.dg_get_device_status() == bq.DG_OK
    qr, sr, _, _ = oracle_mod.gemm_nt_requant(qa, sa, qb, sb, 128, 0, a_1x128=True)
    assert np.array_equal(host(cs), sr) and np.array_equal(host(cq), qr)
