"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each timing its own
replica of the layer (the layer does not shard), reduce to the slowest rank's
time and a whole-job tokens/s; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [10.0, 12.5][rank]          # rank 1 is the slower one
        value, ms = bench.whole_job(ms_local, tokens_per_rank=8, steps=100, world=world)
        bench.barrier(world)
        out[rank] = (value, ms)
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_to_slowest_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        value, ms = out[r]
        assert ms == 12.5                                  # max over ranks
        assert value == pytest.approx(2 * 100 * 8 / 12.5e-3)   # tokens of both ranks / slowest time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.whole_job(4.0, tokens_per_rank=16, steps=10, world=1)
    assert ms == 4.0 and value == pytest.approx(10 * 16 / 4e-3)


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from moe_ffn_layer_gb300 import synth
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(steps=1, warmup=0, seed=0, gpus=2))()
    assert bench.run_reference(args, synth.workload("tiny")) is None
