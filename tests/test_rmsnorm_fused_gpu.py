"""RMSNorm fused into the A prologue of the leaf-tree GEMM [IsoExec blog, "Parallelism-invariant
kernels"; RL-Kernel blog, §6 table row 02 (RMSNorm) and §7]: the fused calls must give the bits of
the separate stages, iso_rmsnorm followed by iso_gemm or iso_selected_logprob."""
import numpy as np
import pytest
import torch

import oracle
from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-6


def _bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.fixture(scope="module")
def c8():
    return B.Contract(8)


# (M, K, N): one ragged row block; several row blocks; a K whose leaves (144) end in a partial
# 16-column stage; the 8B-class projection width
@pytest.mark.parametrize("M,K,N", [(1, 1024, 200), (33, 2048, 520), (300, 4096, 264), (40, 1152, 136),
                                   (257, 4096, 4096)])
def test_rmsnorm_gemm_equals_separate_stages(c8, M, K, N):
    x, gamma = inputs.rmsnorm_inputs(M, K, seed=M + K)
    _, Wt = inputs.gemm_inputs(1, K, N, seed=N)
    xd, gd, Wd = x.to(DEV), gamma.to(DEV), Wt.to(DEV)
    sep = B.gemm(c8, B.rmsnorm(c8, xd, gd, EPS), Wd)
    fused = B.rmsnorm_gemm(c8, xd, gd, EPS, Wd)
    assert _same_bits(fused, sep)
    assert B.last_device_status(c8) == B.ISO_OK


def test_rmsnorm_gemm_rows_are_invariant_and_match_the_oracle(c8):
    M, K, N = 200, 2048, 136
    x, gamma = inputs.rmsnorm_inputs(M, K, seed=3)
    _, Wt = inputs.gemm_inputs(1, K, N, seed=4)
    xd, gd, Wd = x.to(DEV), gamma.to(DEV), Wt.to(DEV)
    full = B.rmsnorm_gemm(c8, xd, gd, EPS, Wd)
    for r in (0, 127, 128, 199):
        assert _same_bits(B.rmsnorm_gemm(c8, xd[r:r + 1].contiguous(), gd, EPS, Wd), full[r:r + 1]), r
    y = oracle.rmsnorm(_bits(x[:8]), _bits(gamma), EPS)  # bf16 bits of the normalised rows
    ref = oracle.gemm_root(y, _bits(Wt), 8)
    got = oracle.bf16_to_f64(_bits(full[:8]))
    assert np.all(np.abs(got - ref).max(axis=1) <= 2e-2 * np.linalg.norm(ref, axis=1))


@pytest.mark.parametrize("T,H,V", [(1, 1024, 2432 * 3 + 640), (77, 2048, 2432 * 2 + 8), (300, 1024, 5000)])
def test_rmsnorm_selected_logprob_equals_separate_stages(c8, T, H, V):
    x, gamma = inputs.rmsnorm_inputs(T, H, seed=T + 1)
    _, W, ids = inputs.logprob_inputs(T, H, V, seed=T + 2)
    xd, gd, Wd, idd = x.to(DEV), gamma.to(DEV), W.to(DEV), ids.to(DEV)
    sep = B.selected_logprob(c8, B.rmsnorm(c8, xd, gd, EPS), Wd, idd)
    fused = B.rmsnorm_selected_logprob(c8, xd, gd, EPS, Wd, idd)
    assert torch.equal(fused, sep)
    # the chunk-unit schedule (workspace of the factors plus the minimum) gives the same bits
    ws_min = torch.empty(B.selected_logprob_min_workspace(c8, T, V) + ((T * 4 + 255) // 256) * 256,
                         dtype=torch.uint8, device=DEV)
    assert torch.equal(B.rmsnorm_selected_logprob(c8, xd, gd, EPS, Wd, idd, ws=ws_min), sep)


def test_fused_workspace_errors(c8):
    lib = B.load()
    x, gamma = inputs.rmsnorm_inputs(8, 1024, seed=5)
    _, W, ids = inputs.logprob_inputs(8, 1024, 2432, seed=6)
    xd, gd, Wd, idd = x.to(DEV), gamma.to(DEV), W.to(DEV), ids.to(DEV)
    out = torch.empty(8, dtype=torch.float32, device=DEV)
    small = torch.empty(64, dtype=torch.uint8, device=DEV)
    st = lib.iso_rmsnorm_selected_logprob(c8.handle, B._ptr(xd), B._ptr(gd), EPS, B._ptr(Wd), B._ptr(idd),
                                          B._ptr(out), 8, 1024, 2432, B._ptr(small), 64, B._stream())
    assert st == B.ISO_ERR_WORKSPACE
    C = torch.empty(8, 136, dtype=torch.bfloat16, device=DEV)
    Wg = W[:, :136].contiguous().to(DEV)
    st = lib.iso_rmsnorm_gemm(c8.handle, B._ptr(xd), B._ptr(gd), EPS, B._ptr(Wg), 136, B._ptr(C), 136, 8, 136, 1024,
                              B._ptr(small), 16, B._stream())
    assert st == B.ISO_ERR_WORKSPACE
    st = lib.iso_rmsnorm_gemm(c8.handle, B._ptr(xd), None, EPS, B._ptr(Wg), 136, B._ptr(C), 136, 8, 136, 1024,
                              B._ptr(small), 64, B._stream())
    assert st == B.ISO_ERR_INVALID_ARG


@pytest.mark.slow
def test_rmsnorm_selected_logprob_full_vocab(c8):
    """The logprob config's H and V at T = 512: fused equals separate bit for bit."""
    T, H, V = 512, 4096, 151936
    x, gamma = inputs.rmsnorm_inputs(T, H, seed=8)
    _, W, ids = inputs.logprob_inputs(T, H, V, seed=9, device=DEV)
    xd, gd = x.to(DEV), gamma.to(DEV)
    sep = B.selected_logprob(c8, B.rmsnorm(c8, xd, gd, EPS), W, ids)
    fused = B.rmsnorm_selected_logprob(c8, xd, gd, EPS, W, ids)
    assert torch.equal(fused, sep)
