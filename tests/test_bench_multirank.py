"""The multi-GPU path of bench.py is data-parallel replicas: no collective on
the data path, only the timing aggregation (max over ranks) and barriers.
Exercise that aggregation with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [3.0, 5.0][rank]
        ms = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
        value = bench.job_throughput(world, bench.step_flops(), ms)
        dist.barrier()
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_is_max_and_value_is_whole_job():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 5.0
    expect = world * bench.step_flops() / 5e-3
    assert abs(out[0][1] - expect) / expect < 1e-12 and out[0][1] == out[1][1]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    assert bench.job_throughput(1, 10.0, 1000.0) == 10.0
