"""The N > 1 path on CPU with world_size 2 over gloo.

The checksum needs no data exchange between GPUs: each rank of the benchmark
checksums its own replica (weak scaling) and only the timing is reduced.  The
page's statement that partials from tensor-parallel ranks sum to the
unsharded checksum is checked across processes: each rank computes the
oracle partial of its own head shard and an all-reduce SUM over int64
(two's complement, so wrapping like uint64) gives the unsharded value."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from helpers import W, OracleCache, c_form, oracle_requests
        # replica timing: rank r pretends to take 1 + r seconds for 10 + r GB
        gbs = bench.job_throughput((10 + rank) * 1e9, 1.0 + rank, world)
        # TP partials: rank r owns heads [2r, 2r+2) of every layer
        wl = W.random_case(5, "cpu", layers=3, heads=4, head_bytes=16,
                           block_size=4, lengths=(13, 7))
        part = []
        for c in wl.caches:
            v = c.pool.numpy().reshape(2, c.num_blocks, 4, 4, 16)
            sub = np.ascontiguousarray(v[:, :, :, 2 * rank:2 * rank + 2, :]).reshape(-1)
            part.append(OracleCache(sub, c.num_blocks, c.layout, c.layer,
                                    2 * rank, 2, c.head_bytes))
        vals, _ = c_form(part, wl.block_size, oracle_requests(wl))
        t = torch.tensor(np.array(vals, dtype=np.uint64).view(np.int64))
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        if rank == 0:
            from helpers import oracle_caches
            full, _ = c_form(oracle_caches(wl.caches), wl.block_size, oracle_requests(wl))
            q.put((gbs, t.numpy().view(np.uint64).tolist(), full))
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gbs, summed, full = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert gbs == pytest.approx((10 + 11) / 2.0)
    assert [int(v) for v in summed] == [int(v) for v in full]
