"""Host logic of the multi-GPU benchmark path, on CPU ranks (gloo, world size 2).

Under weak scaling every rank runs the whole per-GPU workload and no data is
exchanged; the only cross-rank steps are the barrier and the max over ranks
of the timed region, and the job throughput is world_size x per-rank FLOPs
over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms)
    out[rank] = (m, bench.job_throughput(world, 1e12, m))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_throughput():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        m, tput = out[r]
        assert m == 15.0
        assert tput == pytest.approx(2 * 1e12 / 15e-3 / 1e12)


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(1, 2e12, 1.0) == pytest.approx(2000.0)
