"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method (no scaling, rounding or
accumulation): it only draws random numbers and lays out the MoE expert
grouping. Both the CUDA path and the CPU oracle consume what it returns.

Workload recipes (sizes and value distributions of the DeepGEMM pages' use
cases: LLM projections, small-M decode, MoE experts, large squares):

* ``normal``: x ~ N(0, 1), float32.
* ``lognormal_rows``: x[i, :] = N(0, 1) * exp(z_i) with z_i ~ N(0, 1), one z per
  row, so that 128x128 block scales differ from block to block.
* ``moe_group_sizes``: expert probabilities p ~ Dirichlet(1, ..., 1) over G
  experts, group sizes n ~ Multinomial(tokens * topk, p); each group is then
  padded to a multiple of 128 rows. Seed 0 gives, for 4096 tokens, top-2 and 8
  experts, n = [1033, 1551, 36, 6, 873, 2462, 1027, 1204] and M_tot = 8960.
"""
from __future__ import annotations

import numpy as np

ALIGN = 128

# Dense GEMM shapes (M, N, K).
TINY = (128, 256, 512)
LLM_M = 4096
LLM_NK = ((7168, 2048), (2112, 7168), (24576, 1536), (4096, 7168))
SMALL_M = (1, 16, 64, 128)
SMALL_NK = ((24576, 1536), (7168, 16384))
QUANT_SHAPE = (16384, 7168)
MOE = dict(experts=8, tokens=4096, topk=2, hidden=4096, intermediate=11008)
SQUARES = (4096, 8192, 16384)


def seed_for(workload: int, index: int = 0) -> int:
    """Seed of shape `index` of numbered workload `workload` (1000 * workload + index)."""
    return 1000 * int(workload) + int(index)


def normal(shape, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape, dtype=np.float32)


def lognormal_rows(shape, seed: int, sigma: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape, dtype=np.float32)
    z = rng.standard_normal((shape[0], 1), dtype=np.float32) * np.float32(sigma)
    x *= np.exp(z)
    return x


def moe_group_sizes(experts: int, tokens: int, topk: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(experts))
    return rng.multinomial(tokens * topk, p).astype(np.int64)


def moe_layout(group_sizes, align: int = ALIGN):
    """Contiguous grouped layout: returns (m_indices int32 [M_tot], offsets).

    Group g owns rows [offsets[g], offsets[g] + pad(n_g)); its first n_g rows
    carry index g and the padding rows carry -1.
    """
    sizes = np.asarray(group_sizes, dtype=np.int64)
    padded = (sizes + align - 1) // align * align
    offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    m_tot = int(offsets[-1])
    m_indices = np.full(m_tot, -1, dtype=np.int32)
    for g, n in enumerate(sizes):
        m_indices[offsets[g]:offsets[g] + n] = g
    return m_indices, offsets


def moe_inputs(seed: int = 0, experts: int = 8, tokens: int = 4096, topk: int = 2,
               hidden: int = 4096, intermediate: int = 11008, value_seed: int = 4000):
    """Activations A [M_tot, K] (padding rows zero), expert weights B [G, N, K]."""
    sizes = moe_group_sizes(experts, tokens, topk, seed)
    m_indices, offsets = moe_layout(sizes)
    m_tot = m_indices.size
    a = lognormal_rows((m_tot, hidden), value_seed)
    a[m_indices < 0] = 0.0
    b = lognormal_rows((experts * intermediate, hidden), value_seed + 1).reshape(
        experts, intermediate, hidden)
    return a, b, m_indices, sizes
