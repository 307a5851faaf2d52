"""The multi-rank host path of bench.py on CPU: two gloo ranks, each timing its own
replica of a workload (independent sequences, no collective on the data path), combined
by the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from linear_recurrent_sequence_causal_gb300 import inputs as I


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = I.get_workload("tiny_f32")
        # replicas: different inputs per rank, same shapes
        inp = I.generate(wl, seed=bench.replica_seed(wl, rank))
        first = float(inp["v"].flatten()[0])
        firsts = [None] * world
        dist.all_gather_object(firsts, first)
        # each rank reports a different local time; all get the slowest
        local_ms = 10.0 + 5.0 * rank
        ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        value = bench.job_throughput(wl.B * wl.T, world, ms)
        out[rank] = (ms, value, firsts)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_tokens():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    wl = I.get_workload("tiny_f32")
    for rank in range(world):
        ms, value, firsts = out[rank]
        assert ms == pytest.approx(15.0)
        assert value == pytest.approx(wl.B * wl.T * world / 15e-3)
        assert firsts[0] != firsts[1], "replicas must draw different inputs"


def test_single_process_is_unchanged():
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5
    assert bench.job_throughput(100, 1, 2.0) == pytest.approx(5e4)
