"""The multi-rank host logic of bench.py (replicas only: barrier, max-over-ranks
time, whole-job value) on CPU with the gloo backend, world size 2."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    slowest = bench.aggregate_max(ms, world)
    out.put((rank, slowest, bench.dist_env()))
    dist.destroy_process_group()


def test_two_rank_max_time_and_env():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    assert [r[2][:2] for r in res] == [(0, 2), (1, 2)]
    # whole-job value: particles of all ranks at the slowest rank's time
    n = 1000
    assert n * 2 / (15.0 * 1e-3) == pytest.approx(133333.33, rel=1e-6)
