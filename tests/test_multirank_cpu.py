"""The multi-rank benchmark path on CPU: two gloo ranks run independent replicas;
the job's step time is the maximum over ranks and its throughput the sum of the
ranks' work over that time (no collective touches the data path)."""
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


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]
    dist.barrier()
    ms = bench.reduce_max_ms(local_ms, world, "cpu")
    out[rank] = (ms, bench.job_throughput(1000.0, ms, world))
    dist.destroy_process_group()


def test_two_rank_max_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, thr = out[r]
        assert ms == 20.0
        assert thr == pytest.approx(2 * 1000.0 / 0.020)
