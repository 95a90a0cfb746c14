"""The multi-rank plumbing of bench.py, on CPU with two gloo ranks.

Rows are independent and the deterministic path is batch-invariant, so the
path shards by rows with no exchange: every rank runs its own batch (weak
scaling) and only the timing is reduced across ranks (max of the step
times, sum of the processed tokens). Here two ranks check those reductions
and that sharding one batch's rows over the ranks, each computing its shard
alone, reproduces the single-rank result of the FP64 oracle bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outq):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        import synth
        got_max = bench.max_over_ranks(float(rank + 1), world, "cpu")
        got_sum = bench.sum_over_ranks(float(10 * (rank + 1)), world, "cpu")
        # shard the rows of one batch; each rank computes its shard alone
        p = synth.make_problem(24, 256, 64, 8, slices=2, L=3, seed=5, none_frac=0.2)

        def b(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)

        lo, hi = rank * 12, (rank + 1) * 12
        idx = p.idx.numpy()
        z, _, _, y = oracle.apply(b(p.x)[lo:hi], b(p.y)[lo:hi], idx[lo:hi], b(p.A), b(p.B),
                                  p.scale)
        shard = torch.from_numpy(y.astype(np.int32))
        parts = [torch.empty_like(shard) for _ in range(world)]
        dist.all_gather(parts, shard)   # test-only check, not part of the path
        if rank == 0:
            _, _, _, y_full = oracle.apply(b(p.x), b(p.y), idx, b(p.A), b(p.B), p.scale)
            same = bool(np.array_equal(torch.cat(parts).numpy(), y_full.astype(np.int32)))
        else:
            same = True
        outq.put((rank, got_max, got_sum, same))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_timing_reduction_and_row_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for pr in procs:
        pr.join(timeout=30)
        assert pr.exitcode == 0
    for rank, got_max, got_sum, same in res:
        assert got_max == 2.0
        assert got_sum == 30.0
        assert same
