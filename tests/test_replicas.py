"""The N > 1 bench path on CPU: two gloo ranks, each timing its own replica;
the job time is the max over ranks and the throughput counts every rank's
tokens (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [1.5, 2.5][rank]
    ms = bench.max_over_ranks(ms_local)
    q.put((rank, ms, bench.job_throughput(8, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value in res:
        assert ms == 2.5                      # the slowest rank
        assert value == pytest.approx(2 * 8 / 2.5e-3)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_throughput(8, 1, 2.0) == 4000.0
