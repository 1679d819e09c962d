"""The exchange steps of ``exchange.py`` across real processes (gloo ranks on the CPU), with the
float64 oracle standing in for the library's compute steps: row-parallel GEMM (TP over K-leaves),
its sequence-parallel reduce-scatter form, vocab-parallel logprob and expert-parallel MoE must give
exactly the single-rank results for 2 and 4 ranks.  The collectives only move data (IsoExec blog,
"Parallelism-invariant kernels": NCCL transports the partials, the contract's tree combines them),
so the float64 results are identical, not merely close."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from parallelism_invariant_logprob_gb300 import exchange, inputs

L = 8
M, K, N = 13, 512, 40                      # GEMM (ragged row slices for SP)
V, T, H = 2432 * 3 + 640, 6, 64            # logprob: 4 chunks, the last ragged
TM, HM, EM, FM, KM = 10, 64, 8, 64, 4      # MoE


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


class OracleOps:
    """The compute steps of the parallel forms from the float64 oracle (test infrastructure)."""

    def gemm_leaf_partial(self, rank, R, A_r, B_r):
        return torch.from_numpy(oracle.gemm_leaf_partial(_bits(A_r), _bits(B_r), L, R))

    def tree_combine(self, S):
        return _bf16(oracle.round_bf16(oracle.tree_combine(S.numpy())))

    def selected_logprob_partial(self, h, W_r, ids, V_, v0):
        V_r = W_r.shape[1]
        loc = oracle.selected_logprob(_bits(h), _bits(W_r), np.clip(ids.numpy() - v0, 0, V_r - 1), L, chunk_stats=True)
        stats = torch.from_numpy(np.stack([loc["chunk_m"], loc["chunk_s"]], -1).transpose(1, 0, 2).copy())
        mine = (ids.numpy() >= v0) & (ids.numpy() < v0 + V_r)
        return stats, torch.from_numpy(np.where(mine, loc["z_sel"], 0.0))

    def selected_logprob_combine(self, shard_v0, stats, zsel, ids, V_):
        # the chunk tree (pairwise, odd node carried up) over the gathered chunk statistics
        nodes = [(stats[c, :, 0].numpy(), stats[c, :, 1].numpy()) for c in range(stats.shape[0])]
        while len(nodes) > 1:
            nxt = []
            for i in range(0, len(nodes) - 1, 2):
                m = np.empty(T)
                s = np.empty(T)
                for t in range(T):
                    m[t], s[t] = oracle.lse_merge(nodes[i][0][t], nodes[i][1][t], nodes[i + 1][0][t], nodes[i + 1][1][t])
                nxt.append((m, s))
            if len(nodes) % 2:
                nxt.append(nodes[-1])
            nodes = nxt
        lse = nodes[0][0] + np.log(nodes[0][1])
        owner = np.searchsorted(np.array(shard_v0), ids.numpy(), side="right") - 1
        return torch.from_numpy(zsel.numpy()[owner, np.arange(T)] - lse)

    def moe_experts_partial(self, x, ids, W1, W2, expert_mask):
        ys = oracle.moe_layer(_bits(x), ids.numpy(), np.ones(ids.shape), _bits(W1), _bits(W2), L,
                              with_slots=True)["y_slots"].reshape(-1, x.shape[1])
        own = np.array([bool(expert_mask[e]) for e in ids.numpy().reshape(-1)])
        return _bf16(np.where(own[:, None], ys, 0).astype(np.uint16))

    def moe_combine(self, y_slots, w):
        return _bf16(oracle.moe_combine(_bits(y_slots), w.double().numpy()))


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ops = OracleOps()
        A, Bm = inputs.gemm_inputs(M, K, N, seed=31)
        Kl = K // world
        A_r, B_r = A[:, rank * Kl:(rank + 1) * Kl].contiguous(), Bm[rank * Kl:(rank + 1) * Kl].contiguous()
        out[("tp", rank)] = _bits(exchange.row_parallel_gemm(A_r, B_r, ops))
        out[("sp", rank)] = _bits(exchange.sequence_parallel_gemm(A_r, B_r, ops))
        h, W, ids = inputs.logprob_inputs(T, H, V, seed=32)
        chunk_cols = 2432
        shard_chunks = [(4 * q) // world for q in range(world + 1)]  # contiguous chunk ranges
        v0, v1 = shard_chunks[rank] * chunk_cols, min(shard_chunks[rank + 1] * chunk_cols, V)
        out[("vp", rank)] = exchange.vocab_parallel_selected_logprob(h, W[:, v0:v1].contiguous(), ids, V, v0, ops).numpy()
        x, W1, W2, logits = inputs.moe_inputs(TM, HM, EM, FM, seed=33)
        eids, ew = oracle.moe_route(logits.numpy(), KM)
        owner = inputs.random_partition(EM, world, seed=34).tolist()
        mask = [o == rank for o in owner]
        out[("ep", rank)] = _bits(exchange.expert_parallel_moe(x, torch.from_numpy(eids), torch.from_numpy(ew), W1, W2,
                                                               mask, ops))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_exchange_forms_equal_single_rank(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(240)
        assert p.exitcode == 0
    A, Bm = inputs.gemm_inputs(M, K, N, seed=31)
    C = oracle.gemm(_bits(A), _bits(Bm), L)
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=32)
    lp = oracle.selected_logprob(_bits(h), _bits(W), ids.numpy(), L)["out"]
    x, W1, W2, logits = inputs.moe_inputs(TM, HM, EM, FM, seed=33)
    eids, ew = oracle.moe_route(logits.numpy(), KM)
    moe = oracle.moe_layer(_bits(x), eids, ew, _bits(W1), _bits(W2), L)["out"]
    for r in range(world):
        assert np.array_equal(out[("tp", r)], C), r
        r0, r1 = exchange.sp_row_slice(r, world, M)
        assert np.array_equal(out[("sp", r)], C[r0:r1]), r
        assert np.array_equal(out[("vp", r)], lp), r
        assert np.array_equal(out[("ep", r)], moe), r
