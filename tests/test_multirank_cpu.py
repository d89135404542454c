"""The benchmark's multi-rank logic on CPU with gloo, world size 2: every
rank runs its own copy of the workload (different seeds), and the only
cross-rank traffic is a max over the ranks' times and a sum of their bytes."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    t = bench.reduce_over_ranks(10.0 + 5.0 * rank, "max")   # per-rank times
    b = bench.reduce_over_ranks(100.0 * (rank + 1), "sum")  # per-rank bytes
    q.put((r, ws, local, t, b, bench.rank_seed(r)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reductions_and_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    for r, ws, local, t, b, seed in got:
        assert ws == 2 and local == r
        assert t == 15.0            # max over ranks
        assert b == 300.0           # sum over ranks
    assert got[0][5] != got[1][5]   # independent workloads per rank


def test_single_process_reduction_is_identity():
    assert bench.reduce_over_ranks(3.5, "max") == 3.5
    assert bench.rank_seed(0) == 4
