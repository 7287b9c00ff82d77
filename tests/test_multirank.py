"""The multi-rank (replica) path of the benchmark on CPU: two gloo ranks agree on
the slowest rank's times, and the whole-job µs per layer counts every replica."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [1.0 + rank, 5.0 - rank, 2.5]
    got = bench.reduce_max(mine, torch.device("cpu"), world)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == [2.0, 5.0, 2.5]


def test_us_per_layer_counts_replicas():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from semantic_paged_kv_head_gb300 import synth
    w = synth.WORKLOADS["llama8b_36k"]
    one = bench.us_per_layer(0.064, w, 1)
    assert one == pytest.approx(64.0 / 32)
    assert bench.us_per_layer(0.064, w, 4) == pytest.approx(one / 4)
    assert bench.reduce_max([3.0, 1.0], torch.device("cpu"), 1) == [3.0, 1.0]
