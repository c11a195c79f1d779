"""The multi-GPU path of bench.py on CPU: world size 2 over gloo.  Every rank times its own
batch; the job throughput is all ranks' units over the slowest rank's time."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units = [320.0, 480.0][rank]
    seconds = [0.5, 2.0][rank]
    value, t = bench.aggregate(units, seconds)
    out[rank] = value
    out[world + rank] = t
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_sums_units_over_slowest_rank():
    world, port = 2, _free_port()
    out = torch.zeros(2 * world, dtype=torch.float64).share_memory_()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == pytest.approx((320 + 480) / 2.0)
    assert out[1] == pytest.approx((320 + 480) / 2.0)
    assert out[2] == 2.0 and out[3] == 2.0


def test_aggregate_without_process_group_is_local():
    import bench
    assert bench.aggregate(100.0, 0.5) == (200.0, 0.5)
