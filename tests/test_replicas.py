"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks.

On several GPUs the benchmark runs one independent replica of the workload per rank (the
loss has no exchange step), times each rank on its own device, and reports the slowest
rank's time. These tests run that host logic with the gloo backend.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = (bench.max_over_ranks(values[rank]), bench.replica_seed(0, rank), bench.dist_env()[:2])
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("values", [(12.5, 40.0), (7.0, 3.0)])
def test_slowest_rank_time_reaches_every_rank(values):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), values, out), nprocs=world, start_method="spawn")
    assert out[0][0] == out[1][0] == max(values)
    # every rank draws its own replica
    assert out[0][1] != out[1][1]
    assert out[0][2] == (0, 2) and out[1][2] == (1, 2)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
