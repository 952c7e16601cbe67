"""GPU parity of the dense block-scaled NT GEMM against the CPU oracle, through
the C ABI. Inputs are quantized by the ORACLE and the same codes and scales go
to both sides; the bound per element is
|C_gpu - C_ref| <= 8e-3 |C_ref| + 1e-4 sum_k |a~_ik b~_jk|.
Sources: lpnh.cn DeepGEMM walkthrough §2.2, §3.2, §4.3, §5.4 row 2 (ragged
dimensions), §6 (unit scales and exact inputs); pzsr.cn page §3.1, §4.1."""
import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import assert_within_bound, device, host, rows_per_block, sample_rows, to_dev

pytestmark = pytest.mark.gpu


def _operands(oracle_mod, m, n, k, seed, mode=0, dist="normal"):
    gen = synthetic.normal if dist == "normal" else synthetic.lognormal_rows
    a = gen((m, k), seed)
    b = gen((n, k), seed + 500)
    qa, sa = oracle_mod.quantize(a, mode)
    qb, sb = oracle_mod.quantize(b, mode)
    return qa, sa, qb, sb


def _run(qa, sa, qb, sb, mode=0, ldc_pad=0):
    dev = device()
    m, n = qa.shape[0], qb.shape[0]
    ldc = n + ldc_pad
    ldc = (ldc + 7) // 8 * 8
    cbuf = torch.full((m, ldc), float("nan"), dtype=torch.bfloat16, device=dev)
    c = cbuf[:, :n]
    bq.dg_fp8_gemm_nt(c, to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev), to_dev(sb, dev), mode)
    assert bq.dg_get_device_status() == bq.DG_OK
    return c, cbuf


def _check(oracle_mod, qa, sa, qb, sb, rows=None, mode=0, what=""):
    c, cbuf = _run(qa, sa, qb, sb, mode)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows)
    got = c if rows is None else c[torch.as_tensor(rows, device=c.device)]
    return assert_within_bound(got, ref, mag, what)


def test_tiny_128x256x512(oracle_mod):
    m, n, k = synthetic.TINY
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, synthetic.seed_for(1))
    _check(oracle_mod, qa, sa, qb, sb, what="128x256x512")


@pytest.mark.parametrize("m,n,k", [
    (1, 16, 128), (1, 256, 128), (16, 2112, 512), (17, 24, 128), (64, 7168, 1024), (127, 300, 256),
    (129, 136, 384), (200, 1000, 640), (256, 256, 128), (513, 257, 256), (300, 130, 1152),
    (1024, 2112, 2048),
])
def test_edge_shapes(oracle_mod, m, n, k):
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=m * 7 + n + k, dist="lognormal")
    _check(oracle_mod, qa, sa, qb, sb, what=f"{m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [
    (129, 136, 384), (200, 1000, 640), (256, 256, 128), (513, 257, 256), (300, 130, 1152),
    (1024, 2112, 2048),
])
def test_edge_shapes_pow2_scales(oracle_mod, m, n, k):
    """Power-of-two (UE8M0) scales: for M > 128 the tensor core applies them
    (block-scaled MMA) instead of the FP32 promotion; ragged M and N, odd
    numbers of K blocks."""
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=m * 5 + n + k, mode=1, dist="lognormal")
    assert np.all(np.frexp(sa)[0] == 0.5) and np.all(np.frexp(sb)[0] == 0.5)
    _check(oracle_mod, qa, sa, qb, sb, mode=1, what=f"{m}x{n}x{k} pow2")


def test_output_padding_untouched(oracle_mod):
    qa, sa, qb, sb = _operands(oracle_mod, 130, 130, 256, seed=7)
    c, cbuf = _run(qa, sa, qb, sb, ldc_pad=30)
    assert torch.isnan(cbuf[:, 130:].float()).all()
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_within_bound(c, ref, mag, "ld_c > N")


@pytest.mark.parametrize("mode", [0, 1])
def test_unit_scales_exact(oracle_mod, mode):
    """Scales 1 and codes of -1, 0, 1: every sum is an integer of magnitude
    <= K/... that bf16 holds exactly, so the kernel must reproduce it exactly."""
    rng = np.random.default_rng(8)
    m, n, k = 256, 384, 256
    va = rng.integers(-1, 2, (m, k))
    vb = rng.integers(-1, 2, (n, k))
    code = {-1: 0xB8, 0: 0x00, 1: 0x38}
    qa = np.vectorize(code.get)(va).astype(np.uint8)
    qb = np.vectorize(code.get)(vb).astype(np.uint8)
    sa = np.ones((m // 128, k // 128), np.float32)
    sb = np.ones((n // 128, k // 128), np.float32)
    c, _ = _run(qa, sa, qb, sb, mode)
    exact = (va @ vb.T).astype(np.float64)
    assert np.abs(exact).max() <= 256
    assert np.array_equal(c.float().cpu().numpy().astype(np.float64), exact)


@pytest.mark.parametrize("nk", synthetic.LLM_NK)
def test_llm_projection_shapes(oracle_mod, nk):
    n, k = nk
    m = synthetic.LLM_M
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, synthetic.seed_for(2, synthetic.LLM_NK.index(nk)),
                               dist="lognormal")
    _check(oracle_mod, qa, sa, qb, sb, rows=rows_per_block(m, 128, seed=n), what=f"{m}x{n}x{k}")


@pytest.mark.parametrize("m", synthetic.SMALL_M)
@pytest.mark.parametrize("nk", synthetic.SMALL_NK)
def test_small_m_shapes(oracle_mod, m, nk):
    n, k = nk
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, synthetic.seed_for(3, m))
    rows = None if m <= 16 else sample_rows(m, 12, seed=m)
    _check(oracle_mod, qa, sa, qb, sb, rows=rows, what=f"{m}x{n}x{k}")


@pytest.mark.parametrize("m", [16, 64])
def test_decode_192_column_tiles_with_ragged_last_tile(oracle_mod, m):
    """N = 24512 with K = 1536: 128 tiles of 192 columns fill the SMs better
    than 96 of 256, and the last 192-column tile is cut at N; every column of
    the last tiles is checked, with ld_c > N so that no store may cross it."""
    n, k = 24512, 1536
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=1000 + m)
    c, cbuf = _run(qa, sa, qb, sb, ldc_pad=40)
    assert torch.isnan(cbuf[:, n:].float()).all()
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_within_bound(c, ref, mag, f"{m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [
    (64, 4096, 3072),    # 64 rows, B exactly 12 MiB: the 1-SM kernel, 32-column tiles (128 tiles)
    (96, 7000, 1536),    # ragged N past one wave of 32-column tiles: 64-column tiles, last one cut
    (128, 300, 640),     # ragged N inside one tile
    (63, 1024, 1024),    # 63 rows: the split-K cluster kernel
    (64, 8192, 2048),    # 16 MiB of B: the split-K cluster kernel
])
def test_small_problem_routing_edges(oracle_mod, m, n, k):
    """Small GEMMs on both sides of the switch between the 1-SM kernel and the
    split-K cluster kernel (64-128 rows, B up to 12 MiB), with ld_c > N so that
    no store may cross N."""
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=2000 + m + n)
    c, cbuf = _run(qa, sa, qb, sb, ldc_pad=24)
    assert torch.isnan(cbuf[:, n:].float()).all()
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_within_bound(c, ref, mag, f"{m}x{n}x{k}")


@pytest.mark.parametrize("size", synthetic.SQUARES)
@pytest.mark.parametrize("mode", [0, 1])
def test_square_shapes(oracle_mod, size, mode):
    qa, sa, qb, sb = _operands(oracle_mod, size, size, size, synthetic.seed_for(5, size), mode)
    if mode == 1:
        assert np.all(np.frexp(sa)[0] == 0.5) and np.all(np.frexp(sb)[0] == 0.5)
    # One row in every 128-row block: every CTA of every 256-row pair tile, and
    # the first and last rows of the final tile.
    _check(oracle_mod, qa, sa, qb, sb, rows=rows_per_block(size, 128, seed=size + mode), mode=mode,
           what=f"{size}^3 mode {mode}")


def test_split_n_and_m_are_bit_identical(oracle_mod):
    """Output tiles are independent (no split-K), so sub-GEMMs on row or column
    slices reproduce the full result bit for bit (the sharding of a
    multi-GPU run)."""
    m, n, k = 512, 1024, 1024
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=9, dist="lognormal")
    full, _ = _run(qa, sa, qb, sb)
    left, _ = _run(qa, sa, qb[:512], sb[:4])
    right, _ = _run(qa, sa, qb[512:], sb[4:])
    top, _ = _run(qa[:256], sa[:2], qb, sb)
    bottom, _ = _run(qa[256:], sa[2:], qb, sb)
    f = full.view(torch.int16)
    assert torch.equal(torch.cat([left, right], 1).view(torch.int16), f)
    assert torch.equal(torch.cat([top, bottom], 0).view(torch.int16), f)


def test_num_sms_cap_is_bit_identical(oracle_mod):
    qa, sa, qb, sb = _operands(oracle_mod, 640, 768, 512, seed=10)
    full, _ = _run(qa, sa, qb, sb)
    try:
        bq.dg_set_num_sms(7)
        capped, _ = _run(qa, sa, qb, sb)
    finally:
        bq.dg_set_num_sms(0)
    assert torch.equal(full.view(torch.int16), capped.view(torch.int16))


@pytest.mark.parametrize("cap", [2, 5])
@pytest.mark.parametrize("mnk", [(1024, 2048, 1024), (640, 1000, 384), (200, 3000, 640)])
def test_many_tiles_per_pair_pow2_scales(oracle_mod, cap, mnk):
    """Power-of-two scales on one or two CTA pairs: every accumulator, scale
    slot and stage barrier goes through many phases."""
    m, n, k = mnk
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=40 + cap, mode=1, dist="lognormal")
    full, _ = _run(qa, sa, qb, sb, mode=1)
    try:
        bq.dg_set_num_sms(cap)
        capped, _ = _run(qa, sa, qb, sb, mode=1)
    finally:
        bq.dg_set_num_sms(0)
    rows = sample_rows(m, 16, seed=cap)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows)
    assert_within_bound(capped[torch.as_tensor(rows, device=capped.device)], ref, mag, f"pow2 cap {cap}")
    assert torch.equal(full.view(torch.int16), capped.view(torch.int16))


@pytest.mark.parametrize("cap", [1, 2, 5])
@pytest.mark.parametrize("mnk", [(1024, 2048, 1024), (640, 1000, 384), (200, 3000, 640)])
def test_many_tiles_per_cta(oracle_mod, cap, mnk):
    """Few SMs -> each persistent CTA runs many tiles, so every pipeline buffer
    and barrier goes through many phases (catches phase-aliasing races)."""
    m, n, k = mnk
    qa, sa, qb, sb = _operands(oracle_mod, m, n, k, seed=12 + cap, dist="lognormal")
    full, _ = _run(qa, sa, qb, sb)
    try:
        bq.dg_set_num_sms(cap)
        capped, _ = _run(qa, sa, qb, sb)
    finally:
        bq.dg_set_num_sms(0)
    rows = sample_rows(m, 16, seed=cap)
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb, rows=rows)
    assert_within_bound(capped[torch.as_tensor(rows, device=capped.device)], ref, mag, f"cap {cap}")
    assert torch.equal(full.view(torch.int16), capped.view(torch.int16))


def test_empty_and_zero_k():
    dev = device()
    a = torch.zeros((0, 128), dtype=torch.uint8, device=dev)
    b = torch.zeros((16, 128), dtype=torch.uint8, device=dev)
    c = torch.empty((0, 16), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_gemm_nt(c, a, b, torch.ones((0, 1), device=dev), torch.ones((1, 1), device=dev))
    a0 = torch.zeros((8, 0), dtype=torch.uint8, device=dev)
    b0 = torch.zeros((16, 0), dtype=torch.uint8, device=dev)
    c0 = torch.full((8, 16), 3.0, dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_gemm_nt(c0, a0, b0, torch.ones((1, 0), device=dev), torch.ones((1, 0), device=dev))
    torch.cuda.synchronize()
    assert torch.count_nonzero(c0) == 0


def test_other_stream(oracle_mod):
    qa, sa, qb, sb = _operands(oracle_mod, 256, 512, 384, seed=11)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c, _ = _run(qa, sa, qb, sb)
    s.synchronize()
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_within_bound(c, ref, mag, "side stream")
