"""The benchmark's multi-GPU form is replicas only: every rank runs the whole
workload on its own GPU and the job's numbers are the slowest rank's time and
the sum of all ranks' tokens.  This runs that combination step with two gloo
ranks on the CPU (the data path has no collective)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    times, counts = bench.combine_ranks([10.0 + rank, 5.0 * (rank + 1), 1.0], [256.0 + rank, 152.0], w)
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, w, local, times, counts))


def test_two_rank_combination():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, local, times, counts in res:
        assert w == 2 and local == r
        assert times == [11.0, 10.0, 1.0]          # max over ranks
        assert counts == [513.0, 304.0]            # sum over ranks


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    times, counts = bench.combine_ranks([3.0, 2.0], [7.0], 1)
    assert times == [3.0, 2.0] and counts == [7.0]
