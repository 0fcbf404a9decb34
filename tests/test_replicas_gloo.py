"""bench.py's N-GPU path runs independent replicas (the layer does not shard
on these boxes): the only cross-rank step is the max over ranks of the timed
span.  Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]
    results[rank] = (bench.reduce_max(ms, "cpu"), bench.aggregate_rate(world, 100.0, 10, bench.reduce_max(ms, "cpu")))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        mx, rate = results[r]
        assert mx == 5.0                       # the slowest rank's time
        assert rate == pytest.approx(2 * 100.0 * 10 / 5e-3)  # both ranks' work over it


def test_single_process_without_group():
    import bench
    assert bench.reduce_max(7.0, "cpu") == 7.0
