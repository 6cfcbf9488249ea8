"""The multi-rank host logic of bench.py on CPU (gloo, two ranks): the path
shards by whole calls with no data-path collective, so the only collectives
are the barrier and the max of the per-rank timings; the reference arm runs
on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    try:
        got = bench.max_over_ranks(10.0 * (rank + 1))
        dist.barrier()
        ref = bench.run_reference(_Args(), rank, world)
        out.put((rank, got, ref is None))
    finally:
        dist.destroy_process_group()


class _Args:
    steps = 1
    warmup = 0


def test_max_over_ranks_and_reference_rank_gating():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1] == 20.0
    # rank 1 does no reference work and prints nothing; rank 0 does the work
    assert res[1][2] is True


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
