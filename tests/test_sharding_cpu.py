"""Multi-rank host logic on CPU (gloo, world size 2): column sharding of the GEMM
and the benchmark's max-over-ranks timing. Each rank computes its shard with the
CPU oracle; the gathered shards must equal the full result bit for bit, because
output tiles are independent (no split-K)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_quantize_gb300.sharding import scale_rows, shard_columns


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        import synthetic
        m, n, k = 130, 600, 384
        a = synthetic.lognormal_rows((m, k), seed=701)
        b = synthetic.lognormal_rows((n, k), seed=702)
        qa, sa = oracle.quantize(a)
        qb, sb = oracle.quantize(b)
        lo, hi = shard_columns(n, world, rank)
        r0, r1 = scale_rows(lo, hi)
        part, _ = oracle.gemm_nt(qa, sa, qb[lo:hi], sb[r0:r1], want_e=False)
        pieces = [None] * world
        dist.all_gather_object(pieces, (lo, hi, part))
        timing = bench.max_over_ranks([1.0 + rank, 5.0 - rank], world)
        if rank == 0:
            full, _ = oracle.gemm_nt(qa, sa, qb, sb, want_e=False)
            got = np.concatenate([p for _, _, p in sorted(pieces, key=lambda x: x[0])], axis=1)
            spans = sorted((lo_, hi_) for lo_, hi_, _ in pieces)
            out.put((np.array_equal(got, full), spans, timing))
    finally:
        dist.destroy_process_group()


def test_shard_columns_properties():
    for n in (1, 127, 128, 129, 600, 2112, 24576):
        for world in (1, 2, 3, 8):
            spans = [shard_columns(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
            for lo, hi in spans:
                assert (lo % 128 == 0 or lo == hi == n) and lo <= hi
                assert hi == n or hi % 128 == 0


def test_two_rank_gloo_sharding_is_exact():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    exact, spans, timing = out.get(timeout=5)
    assert exact
    assert spans == [(0, 384), (384, 600)]
    assert timing == [2.0, 5.0]
