"""Expert parallelism for the MoE layer [IsoExec blog, "Parallelism-invariant kernels": expert
outputs are combined in a fixed routing order, not in rank order].

Two gloo ranks on the CPU own disjoint expert sets (a seeded partition).  Each computes, with the
float64 oracle, the routing-slot outputs of its own experts only (the other experts' weights are
zero on that rank), the ranks all-gather the slot tensors (transport only), every slot is taken
from the rank owning its expert, and the slots are combined in routing order.  The result equals
the single-rank layer bit for bit."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from parallelism_invariant_logprob_gb300 import inputs

T, H, E, F, K_TOP, L = 24, 64, 8, 32, 4, 4


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _problem():
    x, W1, W2, logits = inputs.moe_inputs(T, H, E, F, seed=31)
    ids, w = oracle.moe_route(logits.numpy(), K_TOP)
    owner = inputs.random_partition(E, 2, seed=32).numpy()
    return _bits(x), _bits(W1), _bits(W2), ids, w, owner


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, W1, W2, ids, w, owner = _problem()
        mine = owner == rank
        W1r, W2r = W1.copy(), W2.copy()
        W1r[~mine] = 0
        W2r[~mine] = 0
        slots = oracle.moe_layer(x, ids, w, W1r, W2r, L, with_slots=True)["y_slots"]  # [T, k, H]
        # bf16 bit patterns travel widened to int32 (gloo moves no 16-bit integers); exact
        gathered = [torch.empty(T, K_TOP, H, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(gathered, torch.from_numpy(slots.astype(np.int32)))
        # each slot from the rank that owns its expert, in routing order
        full = np.empty_like(slots)
        for r in range(world):
            sel = owner[ids] == r
            full[sel] = gathered[r].numpy().astype(np.uint16)[sel]
        out[rank] = oracle.moe_combine(full, w)
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_combine_equals_single_rank():
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
    x, W1, W2, ids, w, owner = _problem()
    assert 0 < owner.sum() < E  # both ranks own experts
    assert len(np.unique(owner[ids])) == 2  # and both serve routed slots
    ref = oracle.moe_layer(x, ids, w, W1, W2, L)["out"]
    for r in range(world):
        assert np.array_equal(out[r], ref), r
