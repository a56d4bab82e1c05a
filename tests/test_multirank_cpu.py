"""The benchmark's multi-rank bookkeeping on CPU with the gloo backend (two
ranks): the step time is the slowest rank's, and the whole-job rate counts
every rank's bytes (replicas, weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(times[rank], world, "cpu")
    out[rank] = (ms, bench.whole_job_gbs(1e9, world, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    times = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    ms, gbs = out[0]
    assert ms == 20.0
    assert abs(gbs - 2 * 1e9 / 20e-3 / 1e9) < 1e-9


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_gbs(2e9, 1, 4.0) == pytest.approx(500.0)
