"""The benchmark's multi-rank path on CPU: two gloo ranks reduce their step
times to the slowest rank's and report the aggregate throughput of both
(replicas, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    try:
        assert bench.dist_env() == (ws, rank, rank)
        ms = bench.job_time(local_ms[rank], ws, "cpu")
        value = bench.job_value(240, ws, ms / 10)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("local_ms", [(2.5, 3.75), (4.0, 1.0)])
def test_two_gloo_ranks_take_the_slowest_time(local_ms):
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, local_ms, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    slowest = max(local_ms)
    for rank, ms, value in res:
        assert ms == slowest  # every rank reports the job's time
        assert value == pytest.approx(240 * ws / (slowest / 10 / 1e3))


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.job_time(1.25, 1) == 1.25
    assert bench.job_value(100, 1, 2.0) == pytest.approx(50000.0)
