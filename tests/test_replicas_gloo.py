"""The N>1 path of bench.py is replicas only (DWDP ranks share no data-path
collective): each rank times its own steps, the job's time is the max over
ranks and the value counts every rank's tokens.  Checked with two gloo ranks
on CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.0, 150.0][rank]
    m = bench.max_over_ranks(ms, world, device="cpu")
    v = bench.whole_job_rate(8192, 10, world, m)
    q.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_timing_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, m, v in got:
        assert m == 150.0
        assert v == pytest.approx(2 * 10 * 8192 / 0.150)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(100, 4, 1, 2000.0) == pytest.approx(200.0)
