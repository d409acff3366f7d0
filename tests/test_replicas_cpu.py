"""The multi-GPU path is replicas only (rows shard with no data-path
collective).  Its host logic -- the slowest rank's step time and the
whole-job throughput -- runs here as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.5][rank]  # the second replica is slower
    got = bench.max_over_ranks(ms, "cpu")
    gbs = bench.job_throughput(10 ** 9, world, got)
    dist.barrier()
    out[rank] = (got, gbs)
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    ms, gbs = out[0]
    assert ms == 5.5
    assert gbs == pytest.approx(2 * 1e9 / 5.5e-3 / 1e9)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(4.25, "cpu") == 4.25
    assert bench.job_throughput(2 * 10 ** 9, 1, 1.0) == pytest.approx(2000.0)
