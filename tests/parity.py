"""Helpers shared by the GPU parity tests: device set-up, the parity bound,
and conversions between torch CUDA tensors and the oracle's numpy arrays."""
import numpy as np
import pytest
import torch

# Per-element GEMM bound: |C_gpu - C_ref| <= REL * |C_ref| + MAG * sum_k |a~ b~|.
REL = 8e-3
MAG = 1e-4


def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantize_gb300 as bq
    bq.lib()
    return torch.device("cuda", 0)


def to_dev(x, dev):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def host(t):
    return t.cpu().numpy()


def assert_within_bound(got_bf16, ref, mag, what=""):
    got = got_bf16.float().cpu().numpy().astype(np.float64) if isinstance(got_bf16, torch.Tensor) \
        else np.asarray(got_bf16, np.float64)
    bound = REL * np.abs(ref) + MAG * mag
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: got {got[tuple(i)]:.6g} ref {ref[tuple(i)]:.6g} "
                           f"bound {bound[tuple(i)]:.3g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements beyond the "
                             f"parity bound; first: {detail}")
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


def sample_rows(m, count, seed=0):
    """Deterministic row sample: first, last, block edges and random rows."""
    rng = np.random.default_rng(seed)
    fixed = [0, m - 1, min(127, m - 1), min(128, m - 1), m // 2]
    rest = rng.choice(m, size=min(count, m), replace=False)
    return np.unique(np.concatenate([fixed, rest])).astype(np.int64)


def rows_per_block(m, block=128, seed=0, valid=None):
    """One random row in every `block`-row block of [0, m) (the tiles of every
    CTA of a launch), plus the first and last rows of the first and the final
    block. With `valid` (a boolean mask) the random row is drawn from the valid
    rows of its block, and blocks without one are skipped."""
    rng = np.random.default_rng(seed)
    rows = [0, min(block - 1, m - 1), (m - 1) // block * block, m - 1]
    for b0 in range(0, m, block):
        cand = np.arange(b0, min(b0 + block, m))
        if valid is not None:
            cand = cand[valid[cand]]
        if cand.size:
            rows.append(int(rng.choice(cand)))
    rows = np.unique(np.asarray(rows, np.int64))
    return rows if valid is None else rows[valid[rows]]


def _expand_scales(s, m, n, block_rows):
    s = np.asarray(s, np.float64)
    if block_rows == 1:
        return np.repeat(s, 128, axis=1)[:m, :n]
    return np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)[:m, :n]


def _block_max(x, block_rows):
    """Max of x over each block_rows x 128 block (zero padding at the edges)."""
    m, n = x.shape
    br = 1 if block_rows == 1 else 128
    mp, np_ = -(-m // br) * br, -(-n // 128) * 128
    pad = np.zeros((mp, np_), np.float64)
    pad[:m, :n] = x
    return pad.reshape(mp // br, br, np_ // 128, 128).max(axis=(1, 3))


def assert_requant_within_bound(q, s, ref, mag, block_rows, pow2, what, oracle_mod):
    """Parity of a requantized GEMM output (E4M3 codes q, scales s) with the
    float64 result ref of the oracle, given the per-element GEMM bound
    e = REL |ref| + MAG mag on the kernel's FP32 accumulator v:
    * scale: s * 448 lies within the block's max|ref| +- max e (FP32 scales,
      up to FP32 rounding); with power-of-two scales s is a power of two with
      s * 448 >= max|v| > s * 224; an all-zero block has s = 1;
    * codes: q is the E4M3 rounding of v / s for some v in [ref - e, ref + e]
      (rounding is monotone, so q lies between the codes of the two ends);
    * FP32 scales: each non-zero block holds a code of magnitude 448."""
    q = np.asarray(q, np.uint8)
    s = np.asarray(s, np.float64)
    ref = np.asarray(ref, np.float64)
    m, n = ref.shape
    e = REL * np.abs(ref) + MAG * np.asarray(mag, np.float64)
    amax = _block_max(np.abs(ref), block_rows)
    emax = _block_max(e, block_rows)
    assert s.shape == amax.shape, (s.shape, amax.shape)
    zero = (amax == 0) & (emax == 0)
    assert np.all(s[zero] == 1.0), f"{what}: all-zero block without scale 1"
    nz = ~zero
    lo, hi = (amax - emax) * (1 - 2.0 ** -22), (amax + emax) * (1 + 2.0 ** -22)
    if pow2:
        mant, _ = np.frexp(s)
        assert np.all(mant == 0.5), f"{what}: scale not a power of two"
        ok = (s * 448 >= lo) & (s * 224 < hi)
    else:
        ok = (s * 448 >= lo) & (s * 448 <= hi)
    bad = nz & ~ok
    assert not bad.any(), f"{what}: {int(bad.sum())} scales outside the bound; first {np.argwhere(bad)[:3].tolist()}"

    t = oracle_mod.e4m3_table()
    S = _expand_scales(s, m, n, block_rows)
    lo_v, hi_v = (ref - e) / S, (ref + e) / S
    lo_v = lo_v - np.abs(lo_v) * 2.0 ** -20
    hi_v = hi_v + np.abs(hi_v) * 2.0 ** -20
    c_lo = t[oracle_mod.e4m3_encode(lo_v.astype(np.float32))]
    c_hi = t[oracle_mod.e4m3_encode(hi_v.astype(np.float32))]
    val = t[q]
    bad = ~((val >= c_lo) & (val <= c_hi))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: code {q[tuple(i)]:#04x} ({val[tuple(i)]:.6g}) allowed "
                           f"[{c_lo[tuple(i)]:.6g}, {c_hi[tuple(i)]:.6g}]" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} codes outside the bound; {detail}")
    if not pow2:
        top = _block_max(np.abs(val), block_rows)
        assert np.all(top[nz & (amax > emax)] == 448.0), f"{what}: a block's largest code is not 448"
