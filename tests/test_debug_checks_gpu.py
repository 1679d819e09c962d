"""The bounds-checked debug build (libiso_debug.so, -DISO_DEBUG) on the GPU: every data-dependent
global store and gather of the kernels is guarded by a check that records ISO_ERR_DEVICE_CHECK and
skips the access instead of trapping (the memory checker is closed on this machine; this is what
stands in for it).  Each workload below -- the small-M cluster GEMM, CTA pairs, short leaves,
16 leaves, leaf partials and the tree combine, logprob in both schedules and vocab shards, the MoE
layer with its whole-leaf stages, attention with ragged packed sequences, RMSNorm and the
diagnostics -- must finish with no check failed and give the normal build's bits."""
import math

import numpy as np
import pytest
import torch

from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _same(a, b):
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    return torch.equal(a, b)


@pytest.fixture(scope="module")
def libs():
    return B.load(), B.load(debug=True)


def _both(libs, L, fn):
    rel, dbg = (B.Contract(L, lib) for lib in libs)
    a = fn(rel)
    b = fn(dbg)
    torch.cuda.synchronize()
    assert dbg.lib.iso_last_device_status(None) == B.ISO_OK
    assert rel.lib.iso_last_device_status(None) == B.ISO_OK
    return a, b


@pytest.mark.parametrize("M,K,N,L", [(1, 4096, 4096, 8), (300, 4096, 392, 8), (7, 768, 4096, 8), (200, 8192, 256, 16),
                                     (129, 256, 136, 1)])
def test_gemm_debug_build(libs, M, K, N, L):
    A, Bm = inputs.gemm_inputs(M, K, N, seed=M + K, device=DEV)
    a, b = _both(libs, L, lambda c: B.gemm(c, A, Bm))
    assert _same(a, b)
    R = 2 if L >= 2 else 1
    Kl = K // R

    def tp(c):
        S = torch.stack([B.gemm_leaf_partial(c, r, R, A[:, r * Kl:(r + 1) * Kl].contiguous(), Bm[r * Kl:(r + 1) * Kl])
                         for r in range(R)])
        return B.tree_combine(c, S)
    a, b = _both(libs, L, tp)
    assert _same(a, b)


def test_logprob_and_rmsnorm_debug_build(libs):
    T, H, V = 200, 1024, 2432 * 3 + 640
    x, gamma = inputs.rmsnorm_inputs(T, H, seed=51, device=DEV)
    _, W, ids = inputs.logprob_inputs(T, H, V, seed=52, device=DEV)

    def run(c):
        h = B.rmsnorm(c, x, gamma, 1e-6)
        full = B.selected_logprob(c, h, W, ids)
        ws = torch.empty(B.selected_logprob_min_workspace(c, T, V), dtype=torch.uint8, device=DEV)
        chunk = B.selected_logprob(c, h, W, ids, ws=ws)
        parts = [B.selected_logprob_partial(c, h, W[:, v0:v1].contiguous(), ids, V, v0)
                 for v0, v1 in ((0, 4864), (4864, V))]
        vp = B.selected_logprob_combine(c, [0, 4864], torch.cat([p[0] for p in parts], 0),
                                        torch.stack([p[1] for p in parts]), ids, V)
        return torch.cat([h.view(torch.int16).float().flatten(), full, chunk, vp])
    a, b = _both(libs, 8, run)
    assert torch.equal(a, b)


def test_moe_debug_build(libs):
    T, H, E, F, k = 200, 256, 16, 768, 8
    x, W1, W2, logits = inputs.moe_inputs(T, H, E, F, seed=53, device=DEV)

    def run(c):
        ids, w = B.moe_route(c, logits, k)
        out = B.grouped_gemm_moe(c, x, ids, w, W1, W2, expert_partition=[e % 3 for e in range(E)])
        y = B.moe_experts_partial(c, x, ids, W1, W2, [e % 2 == 0 for e in range(E)],
                                  y_slots=torch.zeros(T * k, H, dtype=torch.bfloat16, device=DEV))
        return torch.cat([out.flatten(), y.flatten()])
    a, b = _both(libs, 8, run)
    assert _same(a, b)


def test_attention_and_diagnostics_debug_build(libs):
    Q, K, V, qs, ks, p0 = inputs.attention_inputs([130, 1, 0, 257], [0, 300, 7, 5], 8, 2, 128, seed=54,
                                                  extra_keys=[3, 0, 2, 129], device=DEV)
    lp_a = -torch.rand(500, generator=torch.Generator().manual_seed(55)).to(DEV)
    lp_b = lp_a + (torch.arange(500, device=DEV) % 7 == 0) * 1e-3
    offs = torch.tensor([0, 100, 100, 377, 500], dtype=torch.int32, device=DEV)

    def run(c):
        o, l = B.attention(c, Q, K, V, qs, ks, p0, 1.0 / math.sqrt(128))
        d = B.mismatch_diagnostics(c, lp_a, lp_b, offs)
        return o, l, d
    (oa, la, da), (ob, lb, db) = _both(libs, 8, run)
    assert _same(oa, ob) and torch.equal(la, lb)
    for key in da:
        assert torch.equal(da[key], db[key]), key
