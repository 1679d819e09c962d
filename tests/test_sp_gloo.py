"""Sequence parallelism for the row-parallel GEMM [IsoExec blog, "Parallelism-invariant kernels":
with SP the row-parallel reduction becomes a reduce-scatter; the same reduction tree as without
SP is reused and each rank keeps its own output slice].

R gloo ranks on the CPU each hold a contiguous K slice (R a power of two dividing the 8
leaves) and compute its subtree root with the float64 oracle.  The reduce-scatter only
transports: rank q receives row slice q of every rank's partial (point-to-point, no arithmetic
in the collective) and applies the top tree levels in rank order.  Its rows equal the same
rows of the single-rank result bit for bit, for ragged slices too (M not divisible by R)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from parallelism_invariant_logprob_gb300 import inputs

M, K, N, L = 13, 512, 40, 8


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def row_slice(q, R):
    """Rows kept by rank q: [floor(q M / R), floor((q + 1) M / R))."""
    return (q * M) // R, ((q + 1) * M) // R


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        A, B = inputs.gemm_inputs(M, K, N, seed=12)
        Kl = K // world
        part = oracle.gemm_leaf_partial(_bits(A[:, rank * Kl:(rank + 1) * Kl]), _bits(B[rank * Kl:(rank + 1) * Kl]), L,
                                        world)
        part = torch.from_numpy(part)
        # reduce-scatter as transport: send row slice q to rank q, receive mine from everyone
        r0, r1 = row_slice(rank, world)
        recv = [torch.empty(r1 - r0, N, dtype=torch.float64) for _ in range(world)]
        recv[rank] = part[r0:r1].clone()
        reqs = []
        for q in range(world):
            if q == rank:
                continue
            q0, q1 = row_slice(q, world)
            reqs.append(dist.isend(part[q0:q1].contiguous(), dst=q))
            reqs.append(dist.irecv(recv[q], src=q))
        for rq in reqs:
            rq.wait()
        root = oracle.tree_combine(torch.stack(recv).numpy())  # the top log2(R) levels, rank order
        out[rank] = oracle.round_bf16(root)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_sp_reduce_scatter_slice_equals_rows_of_the_full_result(world):
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
    A, B = inputs.gemm_inputs(M, K, N, seed=12)
    full = oracle.gemm(_bits(A), _bits(B), L)  # single rank, no SP
    for q in range(world):
        r0, r1 = row_slice(q, world)
        assert np.array_equal(out[q], full[r0:r1]), q
    # the slices tile the rows exactly once
    assert sum(row_slice(q, world)[1] - row_slice(q, world)[0] for q in range(world)) == M
