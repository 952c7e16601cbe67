"""Bounded in-kernel waits: a wait that nothing completes runs out after a short
limit, the kernel records the timeout in the device status word and returns,
and the CUDA context stays usable (no fault, no hang)."""
import numpy as np
import pytest
import torch

import block_quantize_gb300 as bq
import synthetic
from parity import assert_within_bound, device, to_dev

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives(oracle_mod):
    dev = device()
    assert bq.dg_get_device_status() == bq.DG_OK
    bq.dg_selftest_wait_timeout(2_000_000)            # 2 ms
    assert bq.dg_get_device_status() == bq.DG_ERR_TIMEOUT
    assert bq.dg_get_device_status() == bq.DG_OK      # the word was cleared
    a = synthetic.normal((128, 256), seed=301)
    b = synthetic.normal((128, 256), seed=302)
    qa, sa = oracle_mod.quantize(a)
    qb, sb = oracle_mod.quantize(b)
    c = torch.empty((128, 128), dtype=torch.bfloat16, device=dev)
    bq.dg_fp8_gemm_nt(c, to_dev(qa, dev), to_dev(qb, dev), to_dev(sa, dev), to_dev(sb, dev))
    assert bq.dg_get_device_status() == bq.DG_OK
    ref, mag = oracle_mod.gemm_nt(qa, sa, qb, sb)
    assert_within_bound(c, ref, mag, "after timeout")
