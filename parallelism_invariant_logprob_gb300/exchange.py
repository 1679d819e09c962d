"""The exchange steps of the parallel forms, over ``torch.distributed``.

Every collective here only moves data: all-gathers and all-to-alls, never a
reduction.  The arithmetic of each form -- the rank's partial, and the fixed
tree over the gathered partials in rank order -- runs in the library's kernels
through ``LibraryOps`` (the C ABI), so a rank's result is the single-GPU
result bit for bit whatever the rank count:

  row-parallel GEMM (TP over K)   [IsoExec blog, "Parallelism-invariant kernels":
      each rank owns contiguous K-leaves, NCCL only transports the partial
      results, the contract's tree combines them; RL-Kernel blog, §6 table
      row 06: one fixed balanced tree for TP1/2/4/8]
  sequence-parallel GEMM          [IsoExec blog, same section: with SP the
      reduction becomes a reduce-scatter that reuses the non-SP tree and keeps
      each rank's output slice]
  vocab-parallel logprob          [RL-Kernel blog, §7 "LogP": each shard's local
      statistics, merged in a fixed vocab tile order]
  expert-parallel MoE             [IsoExec blog, "Parallelism-invariant kernels":
      expert outputs combined in a fixed routing order, not in rank order]

With the NCCL backend the tensors stay on the GPU; with gloo they go through
host memory (gloo moves CPU tensors).  A caller may pass another ``ops``
object with the same methods (the tests pass the float64 oracle to check the
exchange logic on machines without a GPU).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as B


class LibraryOps:
    """The compute steps of the parallel forms, through the library's C ABI."""

    def __init__(self, contract: B.Contract, stream=None):
        self.c = contract
        self.stream = stream

    def gemm_leaf_partial(self, rank, R, A_r, B_r):
        return B.gemm_leaf_partial(self.c, rank, R, A_r, B_r, stream=self.stream)

    def tree_combine(self, S):
        return B.tree_combine(self.c, S, stream=self.stream)

    def selected_logprob_partial(self, h, W_r, ids, V, v0):
        return B.selected_logprob_partial(self.c, h, W_r, ids, V, v0, stream=self.stream)

    def selected_logprob_combine(self, shard_v0, stats, zsel, ids, V):
        return B.selected_logprob_combine(self.c, shard_v0, stats, zsel, ids, V, stream=self.stream)

    def moe_experts_partial(self, x, ids, W1, W2, expert_mask):
        T, k = ids.shape
        y = torch.zeros(T * k, x.shape[1], dtype=torch.bfloat16, device=x.device)
        return B.moe_experts_partial(self.c, x, ids, W1, W2, expert_mask, y_slots=y, stream=self.stream)

    def moe_combine(self, y_slots, w):
        return B.moe_combine(self.c, y_slots, w, stream=self.stream)


def _on_host(group) -> bool:
    return dist.get_backend(group) == "gloo"


def all_gather_stack(t: torch.Tensor, group=None) -> torch.Tensor:
    """[R, *t.shape]: every rank's tensor, in rank order (transport only)."""
    R = dist.get_world_size(group)
    src = t.detach().contiguous()
    dev = src.device
    if _on_host(group):
        src = src.cpu()
    parts = [torch.empty_like(src) for _ in range(R)]
    dist.all_gather(parts, src, group=group)
    return torch.stack(parts).to(dev)


def all_gather_ragged(t: torch.Tensor, group=None) -> list:
    """Every rank's tensor (first dimensions may differ), in rank order (transport only)."""
    R = dist.get_world_size(group)
    n = all_gather_stack(torch.tensor([t.shape[0]], dtype=torch.int64, device=t.device), group).view(R).tolist()
    width = max(n)
    pad = torch.zeros((width,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    pad[: t.shape[0]] = t
    full = all_gather_stack(pad, group)
    return [full[r, : n[r]] for r in range(R)]


def row_parallel_gemm(A_r, B_r, ops, group=None):
    """C = A B with K split over the ranks: rank r holds A_r = A[:, K_r] and B_r = B[K_r, :] (its
    contiguous leaves), computes its fp32 subtree root, and every rank combines the gathered roots
    in rank order with the top log2 R levels of the tree.  Returns C (bf16) on every rank."""
    R, r = dist.get_world_size(group), dist.get_rank(group)
    S_r = ops.gemm_leaf_partial(r, R, A_r, B_r)
    return ops.tree_combine(all_gather_stack(S_r, group))


def sp_row_slice(q: int, R: int, M: int):
    """Rows kept by rank q in the sequence-parallel form: [q M / R, (q + 1) M / R)."""
    return (q * M) // R, ((q + 1) * M) // R


def sequence_parallel_gemm(A_r, B_r, ops, group=None):
    """The reduce-scatter form of ``row_parallel_gemm``: rank q receives row slice q of every rank's
    partial (an all-to-all, no arithmetic) and combines only those rows; it returns rows
    sp_row_slice(q, R, M) of C."""
    R, r = dist.get_world_size(group), dist.get_rank(group)
    S_r = ops.gemm_leaf_partial(r, R, A_r, B_r)
    M, N = S_r.shape
    bounds = [sp_row_slice(q, R, M) for q in range(R)]
    r0, r1 = bounds[r]
    dev = S_r.device
    src = S_r.detach().contiguous()
    if _on_host(group):
        src = src.cpu()
    send = [src[q0:q1].contiguous() for q0, q1 in bounds]
    recv = [torch.empty(r1 - r0, N, dtype=src.dtype, device=src.device) for _ in range(R)]
    _all_to_all(recv, send, group)
    return ops.tree_combine(torch.stack(recv).to(dev))


def _all_to_all(recv, send, group):
    """recv[q] <- rank q's send[me], for every q (gloo has no all-to-all: point-to-point there)."""
    if not _on_host(group):
        dist.all_to_all(recv, send, group=group)
        return
    me = dist.get_rank(group)
    peer = (lambda q: q) if group is None else (lambda q: dist.get_global_rank(group, q))
    recv[me].copy_(send[me])
    reqs = []
    for q in range(dist.get_world_size(group)):
        if q != me:
            reqs.append(dist.isend(send[q], dst=peer(q), group=group))
            reqs.append(dist.irecv(recv[q], src=peer(q), group=group))
    for rq in reqs:
        rq.wait()


def vocab_parallel_selected_logprob(h, W_r, ids, V: int, v0: int, ops, group=None):
    """Selected-token logprobs with the vocabulary split over the ranks: rank r holds the LM-head
    columns [v0, v0 + V_r) (chunk-aligned, shards contiguous in rank order), computes its chunk
    statistics and the logits of the ids it owns; the statistics are gathered in rank order and
    every rank runs the chunk tree.  Returns the logprobs [T] on every rank."""
    R = dist.get_world_size(group)
    stats_r, zsel_r = ops.selected_logprob_partial(h, W_r, ids, V, v0)
    v0s = all_gather_stack(torch.tensor([v0], dtype=torch.int64, device=h.device), group).view(R).tolist()
    stats = torch.cat(all_gather_ragged(stats_r, group), 0)
    zsel = all_gather_stack(zsel_r, group)
    return ops.selected_logprob_combine([int(v) for v in v0s], stats, zsel, ids, V)


def expert_parallel_moe(x, ids, w, W1, W2, expert_mask, ops, group=None):
    """The expert layer with the experts split over the ranks (expert_mask: this rank's experts;
    every expert has exactly one owner): each rank computes the slot rows of its experts, the
    rows are gathered, each slot takes the row of its expert's owner (a selection, no
    arithmetic), and every rank runs the slot-tree combine in routing order."""
    R = dist.get_world_size(group)
    T, k = ids.shape
    mask = torch.tensor([1 if m else 0 for m in expert_mask], dtype=torch.int64, device=x.device)
    masks = all_gather_stack(mask, group)  # [R, E]
    if not bool((masks.sum(0) == 1).all()):
        raise ValueError("every expert needs exactly one owning rank")
    owner = masks.argmax(0)  # [E]
    y_r = ops.moe_experts_partial(x, ids, W1, W2, expert_mask)
    Y = all_gather_stack(y_r, group)  # [R, T k, H]
    slot_owner = owner[ids.reshape(-1).long()]
    y = Y[slot_owner, torch.arange(T * k, device=Y.device)]
    return ops.moe_combine(y.view(T, k, -1), w)
