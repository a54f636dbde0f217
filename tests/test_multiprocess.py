"""Host logic of the multi-GPU (replica) path, run as two gloo ranks on CPU:
the whole-job throughput is the units of all ranks over the slowest rank's
step time, identical on every rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r processes 1000*(r+1) units per step in (2 + r) ms
        value, ms = bench.whole_job(1000.0 * (rank + 1), 2.0 + rank, world, dist, "cpu")
        out[rank] = (value, ms)
    finally:
        dist.destroy_process_group()


def test_whole_job_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        res = dict(out)
    # units 1000 + 2000 over the slowest rank's 3 ms
    for r in range(2):
        value, ms = res[r]
        assert ms == pytest.approx(3.0)
        assert value == pytest.approx(3000.0 / 3e-3)


def test_whole_job_single_rank():
    import bench
    value, ms = bench.whole_job(500.0, 4.0, 1)
    assert ms == 4.0 and value == pytest.approx(500.0 / 4e-3)
