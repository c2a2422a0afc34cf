"""The multi-GPU path is replicas only (every box has one GPU and the step
has no exchange): bench.py's whole-job value over N ranks is every rank's
tokens over the slowest rank's time.  Checked with 2 gloo ranks on CPU."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [40.0, 55.0][rank]            # rank 1 is the slow replica
    value, max_ms = bench.replica_value(local_ms, tokens=128, world=world, dist=dist, device="cpu")
    dist.barrier()
    out[rank] = (value, max_ms)
    dist.destroy_process_group()


def test_replica_value_takes_the_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        value, max_ms = out[r]
        assert max_ms == pytest.approx(55.0)
        assert value == pytest.approx(2 * 128 / 0.055)


def test_replica_value_single_process():
    import bench
    value, ms = bench.replica_value(40.0, tokens=128, world=1)
    assert ms == 40.0 and value == pytest.approx(128 / 0.040)
