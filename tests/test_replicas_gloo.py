"""CPU, world size 2 over gloo: bench.py's replica aggregation.  N GPUs run independent
replicas (the op has no exchange step); the job's time is the slowest rank's and its work
the sum of all ranks' -- every rank must see the same two numbers after the all-reduces."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(w, device_is_cuda=False)
    device = torch.device("cpu")
    bench.barrier(dist, device)
    elapsed = 1.0 + 0.5 * rank          # rank 1 is the slow one
    units = 1000.0 * (rank + 1)
    t, u = bench.aggregate(dist, elapsed, units, device)
    bench.barrier(dist, device)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"t": t, "u": u}, f)
    dist.destroy_process_group()


def test_aggregate_takes_max_time_and_summed_work(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for rank in range(world):
        with open(tmp_path / f"rank{rank}.json") as f:
            d = json.load(f)
        assert d["t"] == pytest.approx(1.5)
        assert d["u"] == pytest.approx(3000.0)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, device_is_cuda=False) is None
    assert bench.aggregate(None, 2.0, 7.0, None) == (2.0, 7.0)
