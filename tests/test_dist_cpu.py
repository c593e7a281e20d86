"""The benchmark's multi-process path on CPU: two gloo ranks each time an
independent replica; the job's time is the slowest rank's and its throughput
counts both ranks' steps (the replicas-only scaling of a problem that is not
sharded)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t, v = bench.job_throughput(10.0 * (rank + 1), steps=5, flops_per_step=1e12)
    out.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # slowest rank: 20 ms for 5 steps; 2 ranks x 5 steps x 1e12 flop in 20 ms
    for rank, t, v in res:
        assert t == pytest.approx(20.0)
        assert v == pytest.approx(2 * 5 * 1e12 / 0.020 / 1e12)


def test_single_process_is_its_own_job():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    t, v = bench.job_throughput(4.0, steps=2, flops_per_step=1e12)
    assert t == 4.0 and v == pytest.approx(2 * 1e12 / 0.004 / 1e12)
