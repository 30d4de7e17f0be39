"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each timing a different amount of work.

The hot path shards by request (every (request, KV head) is independent), so N GPUs run N replicas with no
collective on the data path. The only cross-rank steps are the timing reductions: the step time is the maximum over
ranks and the byte count is the sum over ranks.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.reduce_max(10.0 + 5.0 * rank, dist)
    b = bench.reduce_sum(1000.0 * (rank + 1), dist)
    out[rank] = torch.tensor([t, b], dtype=torch.float64)
    dist.barrier()
    dist.destroy_process_group()


def test_reductions_two_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        t, b = out[r].tolist()
        assert t == 15.0          # slowest rank's time
        assert b == 3000.0        # all ranks' bytes


def test_reductions_single_process_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.reduce_sum(7.0, None) == 7.0


def test_reference_arm_other_ranks_exit_clean():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args, world=2, rank=1) == 0
