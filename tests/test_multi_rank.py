"""The benchmark's multi-GPU path on two CPU ranks (gloo): the job's time is
the slowest rank's, taken by an all-reduce MAX after a barrier, and the
whole-job throughput counts every rank's units over that time (replicas,
weak scaling)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=ws)
    try:
        import bench
        env_ws, env_rank, _ = bench.dist_env()
        dist.barrier()
        t = bench.max_over_ranks(times[rank], ws, torch.device("cpu"))
        out.put((rank, env_ws, env_rank, t, bench.job_throughput(1000.0, ws, t)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ws, times = 2, [3.0, 5.5]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, times, out)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env_ws, env_rank, t, v in res:
        assert (env_ws, env_rank) == (ws, rank)
        assert t == 5.5
        assert v == pytest.approx(1000.0 * 2 / 5.5e-3)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(4.25, 1, torch.device("cpu")) == 4.25
    assert bench.job_throughput(10.0, 1, 2.0) == pytest.approx(5000.0)
