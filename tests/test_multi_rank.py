"""The host side of a multi-GPU run, on CPU: two `gloo` ranks in spawned processes.

Requests are independent, so N GPUs run N replicas of the step with no collective on the data
path.  What the ranks share is the timing: `bench.max_over_ranks` takes the slowest rank's time
(an all-reduce MAX), and the job's throughput is every rank's units over that time.  The oracle
arm (`--impl reference`) runs on rank 0 alone; the other ranks leave without work.
"""
import io
import contextlib
import os
import socket
import sys
import types

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t_rank = 0.25 * (rank + 1)                   # rank 1 is the slower one
        t = bench.max_over_ranks(t_rank, world, "cpu")
        units = 1000                                 # every rank's own units (weak scaling)
        value, tmax = bench.aggregate([t], [units * world], world)
        # the oracle arm: rank 0 alone works; here only the other ranks run it, and must print nothing
        out = io.StringIO()
        if rank != 0:
            args = types.SimpleNamespace(workload="membound", sample_requests=1, steps=1, warmup=0, gpus=world)
            with contextlib.redirect_stdout(out):
                bench.run_reference(args)
        dist.barrier()
        q.put((rank, t, value, tmax, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, t, value, tmax, printed in res:
        assert t == 0.5, (rank, t)                   # both ranks see the slowest rank's time
        assert tmax == 0.5
        assert abs(value - 2000 / 0.5) < 1e-9        # all ranks' units / the slowest time
        assert printed == ""                         # rank 1 ran no oracle and printed nothing


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.125, 1, "cpu") == 0.125
    assert bench.aggregate([0.5], [100], 1) == (200.0, 0.5)
