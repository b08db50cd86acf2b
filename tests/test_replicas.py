"""The multi-GPU path of the benchmark is replicas only (each rank runs the
whole forward on its own GPU; there is no exchange).  These CPU tests run two
gloo ranks through the same rank aggregation the benchmark uses: the slowest
rank's time decides, and the job value counts every rank's work."""
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
    ms = [2.0, 3.5][rank]
    got = bench.reduce_max(ms, dist, torch.device("cpu"))
    out[rank] = (got, bench.job_tflops(1e12, world, got))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0][0] == 3.5 and out[1][0] == 3.5
    # 2 ranks x 1 TFLOP each over 3.5 ms
    assert out[0][1] == pytest.approx(2 * 1e12 / 3.5e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(1.25, None, torch.device("cpu")) == 1.25
    assert bench.job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)
