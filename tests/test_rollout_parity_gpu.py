"""Rollout-vs-trainer logprob parity: the same token's logprob through
iso_rmsnorm + iso_selected_logprob must have identical bits whether it is
computed in a packed prefill batch of many sequences, in one-token decode
calls (M = 1), or in decode-step batches of varying size.
[VeXact paper, §2 Eq. (1): delta_t = log pi_train - log pi_rollout must be 0]
[RL-Kernel blog, §5 "The Absolute Consistency Requirement"]"""
import numpy as np
import pytest
import torch

import oracle
from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f32_bits(t):
    return t.contiguous().view(torch.int32)


def run(c, states, gamma, W, ids):
    h = B.rmsnorm(c, states, gamma, 1e-6)
    return B.selected_logprob(c, h, W, ids)


def _parity(c, n_seq, max_len, H, V, seed, n_decode_samples):
    lens = inputs.sequence_lengths(n_seq, max_len, seed)
    total = sum(lens)
    states = inputs.normal_bf16((total, H), 1.0, seed + 1, device=DEV)
    _, gamma = inputs.rmsnorm_inputs(1, H, seed + 2)
    gamma = gamma.to(DEV)
    W = inputs.normal_bf16((H, V), 0.02, seed + 3, device=DEV)
    ids = inputs.uniform_ids(total, V, seed + 4, device=DEV)
    packed = run(c, states, gamma, W, ids)  # trainer: one packed batch
    # rollout decode: one token per call (one workspace and output buffer reused, compared at the end)
    g = torch.Generator().manual_seed(seed + 5)
    sample = torch.randperm(total, generator=g)[:n_decode_samples].tolist()
    ws1 = torch.empty(B.selected_logprob_workspace(c, 1, V), dtype=torch.uint8, device=DEV)
    h1 = torch.empty(1, H, dtype=torch.bfloat16, device=DEV)
    dec = torch.empty(len(sample), 4, dtype=torch.float32, device=DEV)  # a 16-byte row per result (out alignment)
    for i, t in enumerate(sample):
        B.rmsnorm(c, states[t:t + 1], gamma, 1e-6, out=h1)
        B.selected_logprob(c, h1, W, ids[t:t + 1], out=dec[i, :1], ws=ws1)
    idx = torch.tensor(sample, device=DEV)
    diff = (f32_bits(dec[:, 0]) != f32_bits(packed[idx])).nonzero()
    assert diff.numel() == 0, sample[int(diff[0])]
    # the fused RMSNorm + logprob call, one token per call, on part of the sample
    wsf = torch.empty(B.rmsnorm_selected_logprob_workspace(c, 1, V), dtype=torch.uint8, device=DEV)
    nf = min(64, len(sample))
    fused = torch.empty(nf, 4, dtype=torch.float32, device=DEV)
    for i, t in enumerate(sample[:nf]):
        B.rmsnorm_selected_logprob(c, states[t:t + 1], gamma, 1e-6, W, ids[t:t + 1], out=fused[i, :1], ws=wsf)
    assert torch.equal(f32_bits(fused[:, 0]), f32_bits(packed[idx[:nf]]))
    # decode-step emulation: step s batches token s of every sequence longer than s
    starts = np.cumsum([0] + lens[:-1])
    for s in list(range(0, min(max_len, 24))) + [max(lens) - 1]:
        rows = [int(st + s) for st, L in zip(starts, lens) if L > s]
        if not rows:
            continue
        r = torch.tensor(rows, device=DEV)
        step = run(c, states[r].contiguous(), gamma, W, ids[r].contiguous())
        assert torch.equal(f32_bits(step), f32_bits(packed[r])), s
    return states, gamma, W, ids, packed


def test_packed_prefill_vs_decode_small():
    c = B.Contract(8)
    states, gamma, W, ids, packed = _parity(c, n_seq=16, max_len=96, H=512, V=2440, seed=40, n_decode_samples=64)
    # and the packed values match the oracle
    idx = torch.tensor([0, 5, len(ids) - 1], device=DEV)
    h = B.rmsnorm(c, states, gamma, 1e-6)
    hb = h[idx].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    Wb = W.cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.selected_logprob(hb, Wb, ids[idx].cpu().numpy(), 8)
    assert np.max(np.abs(packed[idx].cpu().double().numpy() - ref["out"])) <= 1e-3


@pytest.mark.slow
def test_config5_packed_prefill_vs_decode_full():
    c = B.Contract(8)
    _parity(c, n_seq=64, max_len=8192, H=4096, V=151936, seed=4, n_decode_samples=4096)
