"""The N > 1 path of the benchmark runs independent replicas (the path has
no exchange step); only the timing is reduced across ranks.  Checked here
with two gloo ranks on the CPU: max over ranks and the aggregate value."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    t_local = 1.0 + rank  # rank 1 is the slow one
    t = bench.max_over_ranks(t_local)
    val = bench.aggregate_tflops(2e12, 10, t, ws)
    q.put((rank, ws, r, local, t, val))
    dist.destroy_process_group()


def test_two_replicas_max_time_and_aggregate():
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
    for rank, ws, r, local, t, val in res:
        assert ws == 2 and r == rank and local == rank
        assert t == 2.0                      # the slowest rank's time
        assert val == pytest.approx(2 * 2e12 * 10 / 2.0 / 1e12)


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_tflops(1e12, 4, 2.0, 1) == pytest.approx(2.0)
