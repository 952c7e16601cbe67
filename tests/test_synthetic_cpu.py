"""The seeded input recipes: deterministic draws, the documented seed scheme,
the per-row magnitude spread of the log-normal recipe, and the MoE grouping
(seed 0 group sizes, 128-row padding, one expert id per 128-row block; the
contiguous layout of pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §2.3, §3.3)."""
import numpy as np

import synthetic


def test_seed_scheme():
    assert synthetic.seed_for(2, 3) == 2003 and synthetic.seed_for(1) == 1000


def test_draws_are_deterministic_per_seed():
    a = synthetic.normal((64, 256), 7)
    assert a.dtype == np.float32 and np.array_equal(a, synthetic.normal((64, 256), 7))
    assert not np.array_equal(a, synthetic.normal((64, 256), 8))
    b = synthetic.lognormal_rows((64, 256), 7)
    assert np.array_equal(b, synthetic.lognormal_rows((64, 256), 7))


def test_lognormal_rows_spread_row_magnitudes():
    """One log-normal factor per row: row RMS values spread over orders of
    magnitude, so 128x128 block scales differ from block to block."""
    x = synthetic.lognormal_rows((512, 1024), 11).astype(np.float64)
    rms = np.sqrt((x ** 2).mean(axis=1))
    assert rms.max() / rms.min() > 50
    # The factor is per row, not per element: each row divided by its RMS has unit spread.
    z = x / rms[:, None]
    assert abs(z.std() - 1.0) < 0.01


def test_moe_group_sizes_seed_zero():
    mo = synthetic.MOE
    sizes = synthetic.moe_group_sizes(mo["experts"], mo["tokens"], mo["topk"], 0)
    assert list(sizes) == [1033, 1551, 36, 6, 873, 2462, 1027, 1204]
    assert sizes.sum() == mo["tokens"] * mo["topk"]


def test_moe_layout_pads_each_group_to_128_rows():
    sizes = np.array([1033, 1551, 36, 6, 873, 2462, 1027, 1204])
    m_idx, offsets = synthetic.moe_layout(sizes)
    assert m_idx.dtype == np.int32 and m_idx.size == 8960 == offsets[-1]
    assert np.all(offsets % 128 == 0)
    for g, n in enumerate(sizes):
        rows = m_idx[offsets[g]:offsets[g + 1]]
        assert np.all(rows[:n] == g) and np.all(rows[n:] == -1)
    # Every 128-row block carries one expert id (padding rows are -1).
    for blk in m_idx.reshape(-1, 128):
        ids = set(blk[blk >= 0].tolist())
        assert len(ids) <= 1


def test_moe_layout_empty_group():
    m_idx, offsets = synthetic.moe_layout([0, 5, 0])
    assert list(offsets) == [0, 0, 128, 128] and m_idx.size == 128
    assert np.all(m_idx[:5] == 1) and np.all(m_idx[5:] == -1)
