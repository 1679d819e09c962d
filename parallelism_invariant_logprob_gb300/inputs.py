"""Seeded synthetic input generators shared by the tests, the benchmark and the
smoke check.

This module holds no arithmetic of the method: it only draws random numbers
with ``torch.Generator`` and rounds them to the storage dtype.  Both the CUDA
path and the CPU oracle consume what it returns.

Recipes (shapes and distributions of the workloads on the pages; the pages'
datasets and model weights are not used):
  gemm      A ~ N(0,1) bf16 [M,K];  B ~ N(0, 0.02^2) bf16 [K,N]
  logprob   h ~ N(0,1) bf16 [T,H] (rows of i.i.d. unit normals have RMS ~1,
            which stands in for RMS-normalised hidden states);
            W ~ N(0, 0.02^2) bf16 [H,V]; ids ~ U[0,V) int32
  rmsnorm   x ~ N(0,1) bf16 [T,H]; gamma = bf16(1 + 0.1 N(0,1)) [H]
  moe       x ~ N(0,1) bf16 [T,H]; W1 ~ N(0,0.02^2) bf16 [E,H,2F];
            W2 ~ N(0,0.02^2) bf16 [E,F,H]; router logits ~ N(0,1) fp32 [T,E]
  rollout   64 sequence lengths ~ U[1,8192]; states ~ N(0,1) bf16 [sum,H]
  attention packed sequences (query rows at positions pos0.., keys = cache +
            own rows + unseen tail); Q, K, V ~ N(0,1) bf16 [T, heads, 128]
Exact-integer variants draw small integers so every summation order is exact.
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def small_int_bf16(shape, lo: int, hi: int, seed: int, device="cpu") -> torch.Tensor:
    """Integers in [lo, hi] stored as bf16 (exact)."""
    g = _gen(seed, device)
    return torch.randint(lo, hi + 1, shape, generator=g, device=device, dtype=torch.int32).to(torch.bfloat16)


def uniform_ids(n: int, V: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randint(0, V, (n,), generator=g, device=device, dtype=torch.int32)


def gemm_inputs(M: int, K: int, N: int, seed: int, device="cpu"):
    A = normal_bf16((M, K), 1.0, seed * 2 + 0, device)
    B = normal_bf16((K, N), 0.02, seed * 2 + 1, device)
    return A, B


def logprob_inputs(T: int, H: int, V: int, seed: int, device="cpu"):
    h = normal_bf16((T, H), 1.0, seed * 3 + 0, device)
    W = normal_bf16((H, V), 0.02, seed * 3 + 1, device)
    ids = uniform_ids(T, V, seed * 3 + 2, device)
    return h, W, ids


def rmsnorm_inputs(T: int, H: int, seed: int, device="cpu"):
    x = normal_bf16((T, H), 1.0, seed * 2 + 0, device)
    g = _gen(seed * 2 + 1, device)
    gamma = (1.0 + 0.1 * torch.randn(H, generator=g, device=device, dtype=torch.float32)).to(torch.bfloat16)
    return x, gamma


def moe_inputs(T: int, H: int, E: int, F: int, seed: int, device="cpu"):
    x = normal_bf16((T, H), 1.0, seed * 5 + 0, device)
    W1 = normal_bf16((E, H, 2 * F), 0.02, seed * 5 + 1, device)
    W2 = normal_bf16((E, F, H), 0.02, seed * 5 + 2, device)
    g = _gen(seed * 5 + 3, device)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    return x, W1, W2, logits


def sequence_lengths(n: int, max_len: int, seed: int) -> list:
    g = _gen(seed, "cpu")
    return [int(v) for v in torch.randint(1, max_len + 1, (n,), generator=g)]


def random_partition(E: int, P: int, seed: int) -> torch.Tensor:
    """A seeded expert -> partition map (int32 [E]) with values in [0, P)."""
    g = _gen(seed, "cpu")
    return torch.randint(0, P, (E,), generator=g, dtype=torch.int32)


def attention_inputs(q_lens, pos0, Hq: int, Hkv: int, d: int, seed: int, extra_keys=None, device="cpu"):
    """Packed causal-attention inputs (CPU tensors).  Sequence b has q_lens[b] query rows at
    positions pos0[b], pos0[b]+1, ... and pos0[b] + q_lens[b] + extra_keys[b] keys (the KV
    cache of earlier positions, then the keys of its query rows, then keys no row sees).
    Q, K, V ~ N(0,1) bf16; returns Q, K, V, q_start, k_start, pos0 (int32)."""
    B = len(q_lens)
    extra = list(extra_keys) if extra_keys is not None else [0] * B
    k_lens = [int(pos0[b]) + int(q_lens[b]) + int(extra[b]) for b in range(B)]
    q_start = torch.zeros(B + 1, dtype=torch.int32)
    k_start = torch.zeros(B + 1, dtype=torch.int32)
    q_start[1:] = torch.tensor([int(v) for v in q_lens], dtype=torch.int64).cumsum(0).to(torch.int32)
    k_start[1:] = torch.tensor(k_lens, dtype=torch.int64).cumsum(0).to(torch.int32)
    Tq, Tk = int(q_start[-1]), int(k_start[-1])
    Q = normal_bf16((Tq, Hq, d), 1.0, seed * 3 + 0, device)
    K = normal_bf16((Tk, Hkv, d), 1.0, seed * 3 + 1, device)
    V = normal_bf16((Tk, Hkv, d), 1.0, seed * 3 + 2, device)
    p0 = torch.tensor([int(v) for v in pos0], dtype=torch.int32)
    return Q, K, V, q_start.to(device), k_start.to(device), p0.to(device)
