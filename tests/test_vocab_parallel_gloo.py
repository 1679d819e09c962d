"""The exchange step of vocab-parallel logprob across ranks: each rank's chunk
statistics for its contiguous, chunk-aligned vocabulary shard, all-gathered in
rank order, are the full vocabulary's chunk statistics.  Two gloo ranks on the
CPU compute their shard's statistics with the float64 oracle and exchange them."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from parallelism_invariant_logprob_gb300 import inputs

V, T, H, L = 2432 * 3 + 640, 6, 64, 4
SPLITS = [0, 2432 * 2]  # rank 0 owns chunks 0-1, rank 1 chunks 2-3 (the last one ragged)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        h, W, ids = inputs.logprob_inputs(T, H, V, seed=9)
        v0, v1 = SPLITS[rank], (SPLITS + [V])[rank + 1]
        loc = oracle.selected_logprob(_bits(h), _bits(W[:, v0:v1]), np.clip(ids.numpy() - v0, 0, v1 - v0 - 1), L,
                                      chunk_stats=True)
        mine = torch.from_numpy(np.stack([loc["chunk_m"], loc["chunk_s"]], -1).transpose(1, 0, 2).copy())
        sizes = [None] * world
        dist.all_gather_object(sizes, mine.shape[0])
        parts = [torch.empty(n, T, 2, dtype=torch.float64) for n in sizes]
        dist.all_gather(parts, mine)
        out[rank] = torch.cat(parts, 0).numpy()
    finally:
        dist.destroy_process_group()


def test_two_rank_gather_of_shard_chunk_stats_is_the_full_chunk_stats():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=9)
    full = oracle.selected_logprob(_bits(h), _bits(W), ids.numpy(), L, chunk_stats=True)
    want = np.stack([full["chunk_m"], full["chunk_s"]], -1).transpose(1, 0, 2)
    for r in range(world):
        assert np.array_equal(out[r], want)
