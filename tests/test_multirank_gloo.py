"""The N > 1 host logic with world_size 2 over gloo on CPU.

(1) What the single-GPU emulation stands for: two processes each holding one
replica of a bucket, pre-scaled by 1/2 and summed by torch.distributed's
all_reduce, end with the same bits as the oracle's two-rank ring.  (2) The
benchmark's whole-job aggregation: the maximum elapsed time over ranks and
the whole-job throughput."""
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
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path[:0] = [root, os.path.join(root, "tests")]
    import bench
    import oracle
    import workloads as WL

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        orc = oracle.load()
        wl = WL.c1_mlp()
        plan = orc.assign(wl.numels, None, wl.cap_bytes, wl.first_cap_bytes, wl.order)
        mem = plan["members"][0]
        offs = [int(plan["offset_of"][p]) for p in mem]
        n = int(plan["bucket_numel"][0])
        mine = orc.pack([[WL.grad_np(wl, p, rank) for p in mem]], offs, n)[0]
        t = torch.from_numpy(mine.copy()) * (1.0 / world)
        dist.all_reduce(t)
        both = orc.pack([[WL.grad_np(wl, p, w) for p in mem] for w in range(world)], offs, n)
        ring, _ = orc.ring(both)
        same = np.array_equal(t.numpy().view(np.uint32), ring[rank].view(np.uint32))
        elapsed = [10.0, 12.5][rank]
        m = bench.max_over_ranks(elapsed, dist, "cpu")
        v = bench.job_value(world, 1_000_000_000, 10, m)
        q.put((rank, same, m, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, same, m, v in out:
        assert same, f"rank {rank}: gloo allreduce differs from the oracle's ring"
        assert m == 12.5
        assert v == pytest.approx(2 * 1e9 * 10 / 12.5e-3 / 1e9)
