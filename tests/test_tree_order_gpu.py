"""The contract's leaf tree, add by add, on the GPU for every leaf count.

Each leaf of row m, column n holds exactly one nonzero product, chosen from values
whose fp32 sums round differently under different associations (+-2^24, +-2^23, 1,
2, 3, ...).  A leaf's MMA chain then yields that value exactly, and the GEMM's
result is the fp32 balanced tree over the L leaf values (level by level, left =
lower leaf, round to nearest) rounded once to bf16 [IsoExec blog,
"Parallelism-invariant kernels": contiguous K-leaves combined by a fixed
balanced binary tree].  The expectation below evaluates that tree in numpy
float32 directly from its definition; any other grouping of the adds (an
epilogue that evaluates the tree in another order) changes some of these
results.  Leaf lengths 128 (8 epilogue warps) and 512 (CTA pairs when M > 128,
cluster leaf groups when M <= 128) cover the engine's epilogue forms."""
import numpy as np
import pytest
import torch

from parallelism_invariant_logprob_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"
VALUES = np.array([2.0 ** 24, -2.0 ** 24, 2.0 ** 23, -2.0 ** 23, 1.0, -1.0, 2.0, 3.0, -3.0, 0.0, 0.5],
                  dtype=np.float32)
J = 64  # distinct row patterns: row m uses slot m % J of every leaf


def balanced_tree_f32(v):
    """fp32 balanced tree over the last axis (length a power of two), left = lower index."""
    v = v.astype(np.float32)
    while v.shape[-1] > 1:
        v = (v[..., 0::2] + v[..., 1::2]).astype(np.float32)
    return v[..., 0]


@pytest.mark.parametrize("L", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("leaf_len", [128, 512])
@pytest.mark.parametrize("M", [7, 300])
def test_leaf_tree_order(L, leaf_len, M):
    N = 256
    K = L * leaf_len
    rng = np.random.default_rng(1000 * L + leaf_len + M)
    vals = rng.choice(VALUES, size=(L, J, N))  # value of leaf l, slot j, column n
    Bm = np.zeros((K, N), dtype=np.float32)
    for l in range(L):
        Bm[l * leaf_len:l * leaf_len + J] = vals[l]
    A = np.zeros((M, K), dtype=np.float32)
    rows = np.arange(M)
    for l in range(L):
        A[rows, l * leaf_len + rows % J] = 1.0
    c = B.Contract(L)
    C = B.gemm(c, torch.from_numpy(A).to(torch.bfloat16).to(DEV), torch.from_numpy(Bm).to(torch.bfloat16).to(DEV))
    leaf_values = np.moveaxis(vals[:, rows % J, :], 0, -1)  # [M, N, L]
    root = balanced_tree_f32(leaf_values)
    want = torch.from_numpy(root).to(torch.bfloat16)
    got = C.cpu()
    bad = (got.view(torch.int16) != want.view(torch.int16)).nonzero()
    assert len(bad) == 0, f"{len(bad)} elements differ, first {bad[0].tolist()}: got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"
    # the fixture does tell association orders apart: left to right differs somewhere
    seq = leaf_values[..., 0].astype(np.float32)
    for l in range(1, L):
        seq = (seq + leaf_values[..., l]).astype(np.float32)
    if L >= 4:
        assert not np.array_equal(seq, root)
    assert B.last_device_status(c) == B.ISO_OK
