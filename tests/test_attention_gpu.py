"""GPU parity and invariance of iso_attention, the causal attention kernel with a fixed
KV-chunk merge (RL-Kernel blog, §4 "Focus: The Shared Dependency of Attention and Linear LogP
on LogSumExp", §6 row 03 and §7 "Attention"; VeXact paper, §3.1: KV splitting disabled).

Tolerance, from the arithmetic: the kernel rounds the softmax weights P to bf16 before the
P.V product (relative error <= 2^-9 per weight, so <= 2^-9 max|v| on the weighted sum) and
rounds the output to bf16 (<= 2^-9 |out|); the fp32 score and sum errors are far smaller.  So
|out - exact| <= 2^-8 (max|V| + |exact|) element by element, and |lse - exact| <= 1e-4.  The
lse bound also catches a single key let in or left out at any tested length (that moves lse
by log(1 + e^(s - lse)) >= ~1e-3 here)."""
import math

import numpy as np
import pytest
import torch

import oracle
from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128
SCALE = 1.0 / math.sqrt(D)


def _bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.fixture(scope="module")
def c8():
    return B.Contract(8)


def _run(c, Q, K, V, qs, ks, p0, **kw):
    return B.attention(c, Q.to(DEV), K.to(DEV), V.to(DEV), qs.to(DEV), ks.to(DEV), p0.to(DEV), SCALE, **kw)


def _check_vs_oracle(out, lse, Q, K, V, qs, ks, p0):
    ref = oracle.attention(_bits(Q), _bits(K), _bits(V), qs.numpy(), ks.numpy(), p0.numpy(), SCALE)
    got = out.float().cpu().numpy().astype(np.float64)
    vmax = float(V.float().abs().max())
    err = np.abs(got - ref["out_exact"])
    bound = 2.0 ** -8 * (vmax + np.abs(ref["out_exact"]))
    assert np.all(err <= bound), float((err - bound).max())
    lerr = np.abs(lse.cpu().numpy().astype(np.float64) - ref["lse"])
    assert lerr.max() <= 1e-4, float(lerr.max())
    return ref


# G = Hq / Hkv query heads per KV head: 4, 1, 4; 8 and 16 pack 16 and 8 tokens per tile;
# 3 does not divide 128 and runs one head per tile
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (4, 1), (8, 1), (16, 1), (6, 2)])
def test_attention_vs_oracle_ragged(c8, Hq, Hkv):
    # several tiles and KV chunks, ragged tails, a KV cache before the rows (pos0 > 0),
    # keys past the last row, a one-row sequence and an empty one
    q_lens = [130, 1, 0, 257, 64]
    pos0 = [0, 300, 7, 5, 190]
    extra = [3, 0, 2, 129, 0]
    Q, K, V, qs, ks, p0 = inputs.attention_inputs(q_lens, pos0, Hq, Hkv, D, seed=21, extra_keys=extra)
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    _check_vs_oracle(out, lse, Q, K, V, qs, ks, p0)


def test_attention_exact_tile_and_chunk_boundaries(c8):
    # rows and positions that sit exactly on the 128-row tile and the 80-key chunk grid
    q_lens = [128, 256, 127, 129, 81, 160]
    pos0 = [0, 80, 1, 79, 159, 240]
    Q, K, V, qs, ks, p0 = inputs.attention_inputs(q_lens, pos0, 2, 1, D, seed=22)
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    _check_vs_oracle(out, lse, Q, K, V, qs, ks, p0)


def test_attention_prefill_equals_decode_bitwise(c8):
    # prefill over 300 rows of one sequence, then each sampled row alone as a decode step
    # (one query row, its KV prefix only): the same bits
    Hq, Hkv = 8, 2
    Q, K, V, qs, ks, p0 = inputs.attention_inputs([300], [0], Hq, Hkv, D, seed=23)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    out, lse = B.attention(c8, Qd, Kd, Vd, qs.to(DEV), ks.to(DEV), p0.to(DEV), SCALE)
    for r in (0, 1, 79, 80, 81, 126, 127, 128, 129, 159, 160, 200, 239, 240, 255, 256, 299):
        one = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
        kv = torch.tensor([0, r + 1], dtype=torch.int32, device=DEV)
        o1, l1 = B.attention(c8, Qd[r:r + 1].contiguous(), Kd[:r + 1].contiguous(), Vd[:r + 1].contiguous(), one, kv,
                             torch.tensor([r], dtype=torch.int32, device=DEV), SCALE)
        assert _same_bits(o1[0], out[r]), r
        assert torch.equal(l1[0], lse[r]), r


def test_attention_batch_composition_invariant(c8):
    # a sequence's rows are the same bits alone, packed with others, or after other sequences
    Hq, Hkv = 4, 2
    q_lens, pos0, extra = [77, 140, 3, 200], [10, 0, 250, 60], [0, 5, 1, 0]
    Q, K, V, qs, ks, p0 = inputs.attention_inputs(q_lens, pos0, Hq, Hkv, D, seed=24, extra_keys=extra)
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    for b in range(len(q_lens)):
        q0, q1, k0, k1 = int(qs[b]), int(qs[b + 1]), int(ks[b]), int(ks[b + 1])
        o1, l1 = _run(c8, Q[q0:q1].contiguous(), K[k0:k1].contiguous(), V[k0:k1].contiguous(),
                      torch.tensor([0, q1 - q0], dtype=torch.int32), torch.tensor([0, k1 - k0], dtype=torch.int32),
                      p0[b:b + 1].clone())
        assert _same_bits(o1, out[q0:q1]), b
        assert torch.equal(l1, lse[q0:q1]), b


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (16, 2), (6, 2)])
def test_attention_batched_decode_matches_prefill(c8, Hq, Hkv):
    # one decode call over several sequences (one row each, at different positions) against
    # the prefill of each sequence; the decode tiles pack the heads of a KV group differently
    # from the prefill tiles, the bits must not change
    q_lens = [150, 33, 260]
    Q, K, V, qs, ks, p0 = inputs.attention_inputs(q_lens, [0, 0, 0], Hq, Hkv, D, seed=25)
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    last = [int(qs[b + 1]) - 1 for b in range(3)]
    Qd = Q[last].contiguous()
    dq = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    dpos = torch.tensor([q_lens[b] - 1 for b in range(3)], dtype=torch.int32)
    o1, l1 = _run(c8, Qd, K, V, dq, ks, dpos)
    assert _same_bits(o1, out[last])
    assert torch.equal(l1, lse[last])


def test_attention_without_lse_and_empty(c8):
    Q, K, V, qs, ks, p0 = inputs.attention_inputs([40, 9], [3, 0], 2, 2, D, seed=26)
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    out2, none = _run(c8, Q, K, V, qs, ks, p0, want_lse=False)
    assert none is None and _same_bits(out, out2)
    # no sequences / no rows: no-ops
    e, _ = _run(c8, Q[:0], K, V, torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
                torch.zeros(0, dtype=torch.int32))
    assert e.numel() == 0
    assert B.load().iso_last_device_status(None) == B.ISO_OK


def test_attention_argument_errors(c8):
    lib = B.load()
    Q, K, V, qs, ks, p0 = inputs.attention_inputs([4], [0], 2, 1, D, seed=27)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    qd, kd, pd = qs.to(DEV), ks.to(DEV), p0.to(DEV)
    out = torch.empty(4, 2, D, dtype=torch.bfloat16, device=DEV)
    P = B._ptr
    s = B._stream()

    def call(Qp=P(Qd), d=D, Hq=2, Hkv=1, outp=P(out)):
        return lib.iso_attention(c8.handle, Qp, P(Kd), P(Vd), P(qd), P(kd), P(pd), 1, 4, 4, Hq, Hkv, d, 4, SCALE, outp,
                                 None, s)

    assert call(d=64) == B.ISO_ERR_UNSUPPORTED
    assert call(Hq=3, Hkv=2) == B.ISO_ERR_SHAPE
    assert call(Qp=B._vp(Qd.data_ptr() + 2)) == B.ISO_ERR_ALIGNMENT
    assert call(outp=None) == B.ISO_ERR_INVALID_ARG
    assert call() == B.ISO_OK
    # a sequence table whose rows need keys past the sequence: flagged on the device, rows
    # of that sequence left alone, nothing launched for them
    bad_pos = torch.tensor([1], dtype=torch.int32, device=DEV)
    out.fill_(0)
    st = lib.iso_attention(c8.handle, P(Qd), P(Kd), P(Vd), P(qd), P(kd), P(bad_pos), 1, 4, 4, 2, 1, D, 4, SCALE,
                           P(out), None, s)
    assert st == B.ISO_OK
    assert lib.iso_last_device_status(s) == B.ISO_ERR_SHAPE
    assert int(out.view(torch.int16).abs().sum()) == 0
    assert lib.iso_last_device_status(s) == B.ISO_OK


def _ramp_keys(K, ks, a):
    """Key j of each sequence (j counted from the sequence's first key) scaled by 1 + a j / 80, then
    rounded to bf16: the chunk maxima of the scores grow along the sequence, so the running
    maximum of the chunk merge has to move after chunk 0 (input generation only)."""
    Kf = K.float().clone()
    for b in range(ks.numel() - 1):
        k0, k1 = int(ks[b]), int(ks[b + 1])
        j = torch.arange(k1 - k0, dtype=torch.float32)
        Kf[k0:k1] *= (1.0 + a * j / 80.0)[:, None, None]
    return Kf.to(torch.bfloat16)


def _lazy_moves(Q, K, qs, ks, p0, Hq, Hkv):
    """CPU replay of the merge's lazy maximum, for every (query row, head): the number of chunks
    after chunk 0 at which the running maximum moves.  The kernel's rule: t_c = the chunk's largest
    visible score times c2 = fp32(scale log2 e); m starts at t_0 and moves to t_c only when
    t_c > m + 8.  Scores are taken in float64 here, so a decision within rounding distance of the
    threshold may differ from the kernel's; the counts are only used in aggregate."""
    G = Hq // Hkv
    c2 = np.float32(np.float32(SCALE) * np.float32(math.log2(math.e)))
    out = []
    Qd, Kd = Q.double().numpy(), K.double().numpy()
    for b in range(qs.numel() - 1):
        q0, q1, k0 = int(qs[b]), int(qs[b + 1]), int(ks[b])
        if q1 == q0:
            continue
        pos = int(p0[b]) + np.arange(q1 - q0)
        nk = int(pos[-1]) + 1
        nc = (nk + 79) // 80
        Kh = np.repeat(Kd[k0:k0 + nk], G, axis=1)                    # [keys, Hq, d]
        S = np.einsum("rhd,khd->rhk", Qd[q0:q1], Kh)                  # [rows, Hq, keys]
        S = np.where(np.arange(nk)[None, None, :] > pos[:, None, None], -np.inf, S)
        S = np.concatenate([S, np.full(S.shape[:2] + (nc * 80 - nk,), -np.inf)], axis=2)
        t = (S.reshape(S.shape[0], Hq, nc, 80).max(axis=3).astype(np.float32) * c2).astype(np.float64)
        m = t[:, :, 0].copy()
        moves = np.zeros(m.shape, np.int64)
        for c in range(1, nc):
            mv = t[:, :, c] > m + 8.0
            m = np.where(mv, t[:, :, c], m)
            moves += mv
        out.append(moves)
    return np.concatenate(out, axis=0)


def _decode_row_equals_prefill(c, Qd, Kd, Vd, k0, r, pos, out, lse, row):
    one = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    kv = torch.tensor([0, pos + 1], dtype=torch.int32, device=DEV)
    o1, l1 = B.attention(c, Qd[row:row + 1].contiguous(), Kd[k0:k0 + pos + 1].contiguous(),
                         Vd[k0:k0 + pos + 1].contiguous(), one, kv, torch.tensor([pos], dtype=torch.int32, device=DEV),
                         SCALE)
    return _same_bits(o1[0], out[row]) and torch.equal(l1[0], lse[row])


def test_attention_lazy_rescale_vs_oracle(c8):
    """Rows whose running maximum moves by more than 8 (base 2) after chunk 0, many of them in
    several chunks: the O and l rescale of the merge runs, and its results must still match the
    plain softmax of the oracle and be the same bits in a one-row decode call.
    (RL-Kernel blog, §4 "Causal Chain: How Block Merge Order Alters LSE": the rescale-merge.)"""
    Hq, Hkv = 8, 2
    lens = [300, 700, 1200]
    Q, K, V, qs, ks, p0 = inputs.attention_inputs(lens, [0, 0, 0], Hq, Hkv, D, seed=31)
    K = _ramp_keys(K, ks, 1.5)
    moves = _lazy_moves(Q, K, qs, ks, p0, Hq, Hkv)
    assert (moves >= 1).mean() > 0.6 and (moves >= 2).mean() > 0.4 and moves.max() >= 5
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    _check_vs_oracle(out, lse, Q, K, V, qs, ks, p0)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    many = np.nonzero(moves.max(axis=1) >= 3)[0]
    g = torch.Generator().manual_seed(32)
    pick = many[torch.randint(0, many.size, (10,), generator=g).numpy()].tolist() + [299, 999, 2199]
    for row in pick:
        b = int(np.searchsorted(qs.numpy(), row, side="right")) - 1
        pos = row - int(qs[b])
        assert _decode_row_equals_prefill(c8, Qd, Kd, Vd, int(ks[b]), row, pos, out, lse, row), row
    assert B.last_device_status(c8) == B.ISO_OK


def test_attention_lazy_rescale_long_sequence(c8):
    """The last rows of a 4096-key sequence (52 chunks, a KV cache before the rows) with keys
    ramped so the maximum keeps moving, next to a short sequence in the same call: within the
    oracle's bounds, and decode = prefill bit for bit."""
    Hq, Hkv = 4, 1
    Q, K, V, qs, ks, p0 = inputs.attention_inputs([8, 90], [4088, 0], Hq, Hkv, D, seed=33)
    K = _ramp_keys(K, ks, 0.4)
    moves = _lazy_moves(Q, K, qs, ks, p0, Hq, Hkv)
    assert moves[:8].min() >= 1 and moves[:8].max() >= 4
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    _check_vs_oracle(out, lse, Q, K, V, qs, ks, p0)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    for row in (0, 3, 7):
        assert _decode_row_equals_prefill(c8, Qd, Kd, Vd, 0, row, 4088 + row, out, lse, row), row
    assert B.last_device_status(c8) == B.ISO_OK


@pytest.mark.slow
def test_attention_full_size_sampled(c8):
    """The bench's workload (packed prefill, 4096 query rows in 4 sequences of 1024, 32 query
    heads over 8 KV heads) in the bench's launch; sampled rows against the oracle, each row
    computed alone there (its KV prefix only)."""
    Hq, Hkv = 32, 8
    q_lens = [1024] * 4
    Q, K, V, qs, ks, p0 = inputs.attention_inputs(q_lens, [0] * 4, Hq, Hkv, D, seed=28)
    out, lse = _run(c8, Q, K, V, qs, ks, p0)
    Kb, Vb, Qb = _bits(K), _bits(V), _bits(Q)
    vmax = float(V.float().abs().max())
    g = torch.Generator().manual_seed(5)
    for row in torch.randint(0, 4096, (12,), generator=g).tolist() + [0, 1023, 1024, 4095]:
        b = row // 1024
        p = row - b * 1024
        k0 = int(ks[b])
        ref = oracle.attention(Qb[row:row + 1], Kb[k0:k0 + p + 1], Vb[k0:k0 + p + 1], np.array([0, 1], np.int32),
                               np.array([0, p + 1], np.int32), np.array([p], np.int32), SCALE)
        got = out[row].float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref["out_exact"][0]) <= 2.0 ** -8 * (vmax + np.abs(ref["out_exact"][0]))), row
        assert np.abs(lse[row].cpu().numpy() - ref["lse"][0]).max() <= 1e-4, row
