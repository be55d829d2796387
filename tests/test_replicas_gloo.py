"""Replica (multi-GPU) bookkeeping of bench.py on two gloo ranks on the CPU:
the path has no data-path collective, so N GPUs run N independent blocks and
the whole-job throughput is all ranks' positions over the slowest rank's
time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r processed (r + 1) * 32 positions in (r + 1) * 0.5 s
    units, secs = (rank + 1) * 32.0, (rank + 1) * 0.5
    out[rank] = (bench._max_over_ranks(secs, dist), bench._sum_over_ranks(units, dist),
                 bench.replica_throughput(units, secs, dist))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        mx, sm, thr = out[r]
        assert mx == pytest.approx(1.0)
        assert sm == pytest.approx(96.0)
        assert thr == pytest.approx(96.0)


def test_single_rank_is_identity():
    import bench
    assert bench.replica_throughput(32.0, 0.25, None) == pytest.approx(128.0)
