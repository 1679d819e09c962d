"""The exchange steps of ``exchange.py`` with the library's own partials: two processes, each
a rank with its own CUDA context on the same GPU, exchange the fp32 subtree roots, the vocab
shards' chunk statistics and the experts' slot rows over gloo (through host memory: the ranks'
kernels never wait on one another), and every rank's result must equal the single-call result
bit for bit (IsoExec blog, "Parallelism-invariant kernels": the collectives only transport;
RL-Kernel blog, §6 table row 06 and §7 "LogP")."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _same(a, b):
    return bool(torch.equal(a.contiguous().view(torch.int16) if a.dtype == torch.bfloat16 else a,
                            b.contiguous().view(torch.int16) if b.dtype == torch.bfloat16 else b))


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from parallelism_invariant_logprob_gb300 import binding as B
        from parallelism_invariant_logprob_gb300 import exchange, inputs
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        c = B.Contract(8)
        ops = exchange.LibraryOps(c)
        # row-parallel and sequence-parallel GEMM: M = 300 rows (ragged SP slices), K = 1024
        M, K, N = 300, 1024, 392
        A, Bm = inputs.gemm_inputs(M, K, N, seed=41, device=dev)
        Kl = K // world
        A_r, B_r = A[:, rank * Kl:(rank + 1) * Kl].contiguous(), Bm[rank * Kl:(rank + 1) * Kl].contiguous()
        C = B.gemm(c, A, Bm)
        out[("tp", rank)] = _same(exchange.row_parallel_gemm(A_r, B_r, ops), C)
        r0, r1 = exchange.sp_row_slice(rank, world, M)
        out[("sp", rank)] = _same(exchange.sequence_parallel_gemm(A_r, B_r, ops), C[r0:r1])
        # vocab-parallel logprob: 4 chunks of 2432 columns (the last ragged), contiguous shards
        T, H, V = 33, 256, 2432 * 3 + 640
        h, W, ids = inputs.logprob_inputs(T, H, V, seed=42, device=dev)
        chunks = [(4 * q) // world for q in range(world + 1)]
        v0, v1 = chunks[rank] * 2432, min(chunks[rank + 1] * 2432, V)
        lp = exchange.vocab_parallel_selected_logprob(h, W[:, v0:v1].contiguous(), ids, V, v0, ops)
        out[("vp", rank)] = _same(lp, B.selected_logprob(c, h, W, ids))
        # expert-parallel MoE layer: a seeded expert -> rank map
        T, H, E, F, k = 64, 256, 16, 128, 4
        x, W1, W2, logits = inputs.moe_inputs(T, H, E, F, seed=43, device=dev)
        eids, ew = B.moe_route(c, logits, k)
        owner = inputs.random_partition(E, world, seed=44).tolist()
        y = exchange.expert_parallel_moe(x, eids, ew, W1, W2, [o == rank for o in owner], ops)
        out[("ep", rank)] = _same(y, B.grouped_gemm_moe(c, x, eids, ew, W1, W2))
        torch.cuda.synchronize()
        out[("status", rank)] = B.last_device_status(c)
    finally:
        dist.destroy_process_group()


def test_exchange_with_library_partials_two_processes():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    for r in range(world):
        for form in ("tp", "sp", "vp", "ep"):
            assert out[(form, r)], (form, r)
        assert out[("status", r)] == 0
