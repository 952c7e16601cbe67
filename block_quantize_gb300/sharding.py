"""Column sharding of the block-scaled GEMM across ranks (host logic only).

Output tiles are independent (there is no split-K), so a GEMM whose N columns are
divided among ranks needs no exchange: each rank multiplies the full A by its slice
of B. Slices are whole 128-column scale blocks, so each rank's B scales are whole
rows of sb and every column's arithmetic is unchanged by the split.
"""
from __future__ import annotations

BLOCK = 128


def shard_columns(n: int, world: int, rank: int, align: int = BLOCK) -> tuple[int, int]:
    """[lo, hi) columns of `rank`: contiguous, `align`-aligned, as even as possible."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    blocks = (n + align - 1) // align
    base, extra = divmod(blocks, world)
    first = rank * base + min(rank, extra)
    count = base + (1 if rank < extra else 0)
    lo = min(n, first * align)
    hi = min(n, (first + count) * align)
    return lo, hi


def scale_rows(lo: int, hi: int, align: int = BLOCK) -> tuple[int, int]:
    """Rows of sb that cover columns [lo, hi)."""
    return lo // align, (hi + align - 1) // align
