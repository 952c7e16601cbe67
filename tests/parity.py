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
