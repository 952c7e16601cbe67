"""GPU parity of the block quantizer: E4M3 codes and scales bit-exact against
the CPU oracle (lpnh.cn DeepGEMM walkthrough §4.2, §3.1, §5.4; pzsr.cn page
§3.1 for power-of-two scales), through the C ABI."""
import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import device, host, to_dev

pytestmark = pytest.mark.gpu


def _check(x_np, mode, oracle_mod, x_dev=None):
    dev = device()
    xd = to_dev(x_np, dev) if x_dev is None else x_dev
    q, s = bq.dg_quantize_fp8_block(xd, mode)
    torch.cuda.synchronize()
    rq, rs = oracle_mod.quantize(x_np, mode)
    gq, gs = host(q), host(s)
    assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32)), "scales differ"
    if not np.array_equal(gq, rq):
        bad = np.argwhere(gq != rq)[:5]
        raise AssertionError(f"{int((gq != rq).sum())} codes differ, e.g. " + ", ".join(
            f"{tuple(i)} x={x_np[tuple(i)]!r} gpu=0x{gq[tuple(i)]:02x} ref=0x{rq[tuple(i)]:02x}"
            for i in bad))


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(128, 128), (1, 1), (1, 7), (3, 130), (129, 130), (300, 513),
                                   (255, 1024), (128, 512), (1000, 4),
                                   # more blocks than four per SM (the 3-stage streaming launch):
                                   # one block per row of blocks, and rows of three blocks that
                                   # the grid's stride wraps unevenly
                                   (80000, 100), (30000, 300),
                                   # on 152 SMs: at most three blocks per SM (three CTAs per SM,
                                   # the tile re-read from shared memory), whole and ragged ...
                                   (4096, 1536), (3000, 1500),
                                   # ... and four blocks per SM (two CTAs per SM)
                                   (4096, 2048), (4000, 2000)])
def test_quantize_bit_exact(oracle_mod, shape, mode):
    _check(synthetic.lognormal_rows(shape, seed=101 + shape[0] + shape[1]), mode, oracle_mod)


@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_special_values(oracle_mod, mode):
    rng = np.random.default_rng(102)
    x = np.zeros((384, 640), np.float32)
    x[0, :128] = -0.0                                          # block of signed zeros
    x[128:256, 0:128] = rng.standard_normal((128, 128)) * 1e-40   # subnormal inputs
    x[130, 200] = 1e-44                                        # scale underflows to 0 -> 1
    x[256:, 256:384] = rng.standard_normal((128, 128)) * 1e37      # large magnitudes
    x[200:220, 400:500] = rng.uniform(-1, 1, (20, 100)).astype(np.float32) * 3.0e38
    # values that land on E4M3 midpoints when the scale is 1 (amax = 448)
    t = oracle_mod.e4m3_table()[:0x7F]
    mids = (0.5 * (t[:-1] + t[1:])).astype(np.float32)
    x[0, 128:128 + mids.size] = mids
    x[1, 128] = 448.0
    x[2, 128:128 + mids.size] = -np.nextafter(mids, np.float32(np.inf))
    _check(x, mode, oracle_mod)


@pytest.mark.parametrize("ld_pad", [0, 4, 3])
def test_quantize_strided_input(oracle_mod, ld_pad):
    """A row stride wider than the row: 4-multiples take the vector path, others the scalar one."""
    dev = device()
    rows, cols = 200, 260
    full = synthetic.normal((rows, cols + ld_pad), seed=103)
    xd = to_dev(full, dev)[:, :cols]
    _check(np.ascontiguousarray(full[:, :cols]), 0, oracle_mod, x_dev=xd)


@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_full_activation_shape(oracle_mod, mode):
    """The 16384 x 7168 activation that the quantizer benchmark times."""
    x = synthetic.normal(synthetic.QUANT_SHAPE, seed=synthetic.seed_for(3, 9))
    _check(x, mode, oracle_mod)


def test_quantize_empty_is_noop():
    dev = device()
    q, s = bq.dg_quantize_fp8_block(torch.empty((0, 64), device=dev))
    assert q.shape == (0, 64) and s.shape == (0, 1)
