"""GPU parity and invariance of the 16-leaf contract.

The tree over 16 K-leaves is the same balanced binary tree as for 8 (IsoExec blog,
"Parallelism-invariant kernels": leaves combined by the contract's fixed binary schedule;
RL-Kernel blog, §6 table row 06: one fixed balanced tree for TP1/2/4/8, here extended to 16
ranks).  Its eager merge stack needs a fifth accumulator, so the engine parks the root of leaves
[0, 8) in shared memory and makes the tree's top add as it reads the root of leaves [8, 16).
These tests check that path against the float64 oracle (exactly where the arithmetic is exact,
within the row-norm bound elsewhere) and against the other schedules, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
L = 16


def bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.fixture(scope="module")
def c16():
    return B.Contract(L)


def test_tree_shape_sixteen_leaves(c16):
    # one product per leaf: leaf 0 = 2^24, leaf 8 = 1, leaf 15 = -2^24, the rest 0.  The balanced
    # tree adds (2^24) + (1 + -2^24) = 1 at its top; a left fold, or the parked half added one
    # level too low ((2^24 + 1) rounds to 2^24), gives 0.
    K = L * 16
    A = torch.zeros(1, K, dtype=torch.bfloat16)
    Bm = torch.zeros(K, 8, dtype=torch.bfloat16)
    for l, v in ((0, 2.0 ** 24), (8, 1.0), (15, -(2.0 ** 24))):
        A[0, l * 16] = 1.0
        Bm[l * 16, :] = v
    root = oracle.gemm_root(bits(A), bits(Bm), L)
    assert root[0, 0] == 1.0
    C = B.gemm(c16, A.to(DEV), Bm.to(DEV))
    assert torch.all(C.float().cpu() == 1.0)
    S = B.gemm_leaf_partial(c16, 0, 1, A.to(DEV), Bm.to(DEV))
    assert torch.all(S.cpu() == 1.0)
    # two ranks of 8 leaves: their fp32 subtree roots, combined at the top
    S2 = torch.stack([B.gemm_leaf_partial(c16, r, 2, A[:, r * 128:(r + 1) * 128].contiguous().to(DEV),
                                          Bm[r * 128:(r + 1) * 128].contiguous().to(DEV)) for r in range(2)])
    assert torch.all(S2[0].cpu() == 2.0 ** 24) and torch.all(S2[1].cpu() == -(2.0 ** 24) + 1.0)
    assert torch.all(B.tree_combine(c16, S2).float().cpu() == 1.0)


# leaves of 16, 128, 256 and 512 k; one row block (small A boxes) and many (CTA pairs at 512-k
# leaves with more than 128 rows); ragged N
@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (7, 392, 2048), (300, 136, 4096), (300, 256, 8192)])
def test_exact_integer_bits_equal_oracle(c16, M, N, K):
    A = inputs.small_int_bf16((M, K), -3, 3, seed=M + 1)
    Bm = inputs.small_int_bf16((K, N), -3, 3, seed=N + 2)
    C = B.gemm(c16, A.to(DEV), Bm.to(DEV))
    assert np.array_equal(bits(C), oracle.gemm(bits(A), bits(Bm), L))


@pytest.mark.parametrize("K", [4096, 8192])
def test_normal_inputs_invariance(c16, K):
    M, N = 300, 512
    A, Bm = inputs.gemm_inputs(M, K, N, seed=K // 64)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    full = B.gemm(c16, Ad, Bd)
    root = oracle.gemm_root(bits(A), bits(Bm), L)
    got = oracle.bf16_to_f64(bits(full))
    assert np.all(np.abs(got - root).max(axis=1) <= 2e-2 * np.linalg.norm(root, axis=1))
    ulp = np.spacing(np.abs(oracle.bf16_to_f64(oracle.round_bf16(root))).astype(np.float32)) * 65536
    assert np.all(np.abs(got - root) <= ulp + 1e-5 * np.linalg.norm(root, axis=1, keepdims=True))
    # a row alone, and the rows shuffled: the same bits
    for r in (0, 150, 299):
        assert same_bits(B.gemm(c16, Ad[r:r + 1].contiguous(), Bd), full[r:r + 1]), r
    perm = torch.randperm(M, generator=torch.Generator().manual_seed(K)).to(DEV)
    assert same_bits(B.gemm(c16, Ad[perm].contiguous(), Bd), full[perm])
    # every simulated rank count: partials of L/R leaves, then the top log2 R levels
    for R in (1, 2, 4, 8, 16):
        Kl = K // R
        S = torch.stack([B.gemm_leaf_partial(c16, r, R, Ad[:, r * Kl:(r + 1) * Kl].contiguous(), Bd[r * Kl:(r + 1) * Kl])
                         for r in range(R)])
        assert same_bits(B.tree_combine(c16, S), full), R
    # leaf groups over more SMs (one row block): the same bits as the single pass
    few = Ad[:7].contiguous()
    assert same_bits(B.gemm_ws(c16, few, Bd), full[:7])


def test_selected_logprob_sixteen_leaves(c16):
    T, H, V = 150, 2048, 5000
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=61)
    hd, Wd, idd = h.to(DEV), W.to(DEV), ids.to(DEV)
    out = B.selected_logprob(c16, hd, Wd, idd)
    ref = oracle.selected_logprob(bits(h), bits(W), ids.numpy(), L)["out"]
    assert np.max(np.abs(out.cpu().double().numpy() - ref)) <= 1e-3
    # chunk units (the minimum workspace) and tile units: the same bits; one row alone too
    ws_min = torch.empty(B.selected_logprob_min_workspace(c16, T, V), dtype=torch.uint8, device=DEV)
    assert torch.equal(B.selected_logprob(c16, hd, Wd, idd, ws=ws_min), out)
    assert torch.equal(B.selected_logprob(c16, hd[77:78].contiguous(), Wd, idd[77:78].contiguous()), out[77:78])
    assert B.last_device_status(c16) == B.ISO_OK


def test_moe_layer_sixteen_leaves(c16):
    # gate/up leaves of 16 k (H = 256), down leaves of 16 k (F = 256)
    T, H, E, F, k = 64, 256, 8, 256, 4
    x, W1, W2, logits = inputs.moe_inputs(T, H, E, F, seed=62)
    xd, W1d, W2d = x.to(DEV), W1.to(DEV), W2.to(DEV)
    ids, w = B.moe_route(c16, logits.to(DEV), k)
    out = B.grouped_gemm_moe(c16, xd, ids, w, W1d, W2d)
    ref = oracle.moe_layer(bits(x), ids.cpu().numpy(), w.cpu().double().numpy(), bits(W1), bits(W2), L, exact=True,
                           with_slots=True)
    oe = ref["out_exact"]
    assert np.all(np.abs(oracle.bf16_to_f64(bits(out)) - oe).max(axis=1) <= 2e-2 * np.linalg.norm(oe, axis=1))
    y = B.moe_experts_partial(c16, xd, ids, W1d, W2d, [1] * E).view(T, k, H)
    got, yr = oracle.bf16_to_f64(bits(y)), oracle.bf16_to_f64(ref["y_slots"])
    ulp = np.spacing(np.abs(yr).astype(np.float32)).astype(np.float64) * 65536.0
    rms = np.sqrt((yr ** 2).mean(axis=-1, keepdims=True))
    assert np.all(np.abs(got - yr) <= ulp + 2.0 ** -9 * rms)
    assert same_bits(B.grouped_gemm_moe(c16, xd, ids, w, W1d, W2d, expert_partition=[e % 3 for e in range(E)]), out)
    assert B.last_device_status(c16) == B.ISO_OK


def test_rmsnorm_prologue_sixteen_leaves(c16):
    M, K, N = 200, 4096, 384
    x, gamma = inputs.rmsnorm_inputs(M, K, seed=63)
    _, Bm = inputs.gemm_inputs(1, K, N, seed=64)
    xd, gd, Bd = x.to(DEV), gamma.to(DEV), Bm.to(DEV)
    sep = B.gemm(c16, B.rmsnorm(c16, xd, gd, 1e-6), Bd)
    assert same_bits(B.rmsnorm_gemm(c16, xd, gd, 1e-6, Bd), sep)
