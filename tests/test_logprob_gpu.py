"""GPU parity and invariance of iso_selected_logprob and iso_rmsnorm through the
C ABI.  Logprob tolerance: <= 1e-3 absolute against the float64 oracle.
RMSNorm: bf16 outputs within one bf16 ulp of the oracle's exactly rounded
value (the GPU reduces in fp32)."""
import math

import numpy as np
import pytest
import torch

import oracle
from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f32_same(a, b):
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


@pytest.fixture(scope="module")
def c8():
    return B.Contract(8)


# ------------------------------------------------------------------ logprob
@pytest.mark.parametrize("T,H,V", [(300, 512, 2440), (7, 1024, 128 * 19 * 3), (130, 256, 40000), (1, 128, 8)])
def test_logprob_vs_oracle(c8, T, H, V):
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=T)
    out = B.selected_logprob(c8, h.to(DEV), W.to(DEV), ids.to(DEV))
    ref = oracle.selected_logprob(bits(h), bits(W), ids.numpy(), 8)
    got = out.cpu().double().numpy()
    assert np.max(np.abs(got - ref["out"])) <= 1e-3
    assert np.all(got <= 0)
    assert B.last_device_status(c8) == B.ISO_OK


def test_logprob_batch_invariance_bitwise(c8):
    T, H, V = 300, 512, 2440
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=1)
    hd, Wd, idd = h.to(DEV), W.to(DEV), ids.to(DEV)
    full = B.selected_logprob(c8, hd, Wd, idd)
    for t in (0, 1, 127, 128, 299):
        one = B.selected_logprob(c8, hd[t:t + 1].contiguous(), Wd, idd[t:t + 1].contiguous())
        assert f32_same(one, full[t:t + 1]), t
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(3)).to(DEV)
    sh = B.selected_logprob(c8, hd[perm].contiguous(), Wd, idd[perm].contiguous())
    assert f32_same(sh, full[perm])


def test_logprob_zero_weights_uniform(c8):
    T, H, V = 64, 256, 151936
    h, _, ids = inputs.logprob_inputs(T, H, 8, seed=2)
    ids = inputs.uniform_ids(T, V, seed=5)
    W = torch.zeros(H, V, dtype=torch.bfloat16, device=DEV)
    out = B.selected_logprob(c8, h.to(DEV), W, ids.to(DEV))
    assert torch.all(torch.abs(out.double() + math.log(V)) <= 2e-6)
    # every row has the identical computation: identical bits
    assert torch.all(out.view(torch.int32) == out[0].view(torch.int32))


def test_logprob_dominant_logit(c8):
    H, V = 128, 1024
    h = torch.ones(2, H, dtype=torch.bfloat16)
    W = torch.zeros(H, V, dtype=torch.bfloat16)
    W[:, 777] = 0.5  # z[777] = 64
    out = B.selected_logprob(c8, h.to(DEV), W.to(DEV), torch.tensor([777, 3], dtype=torch.int32, device=DEV)).cpu()
    assert abs(float(out[0])) < 1e-6
    assert abs(float(out[1]) + 64.0) < 1e-4


def test_logprob_bad_token_id_reports(c8):
    h, W, _ = inputs.logprob_inputs(4, 128, 256, seed=3)
    ids = torch.tensor([0, 256, -1, 5], dtype=torch.int32, device=DEV)
    out = B.selected_logprob(c8, h.to(DEV), W.to(DEV), ids).cpu()
    assert torch.isnan(out[1]) and torch.isnan(out[2]) and not torch.isnan(out[0]) and not torch.isnan(out[3])
    assert B.last_device_status(c8) == 11  # ISO_ERR_BAD_TOKEN_ID
    assert B.last_device_status(c8) == B.ISO_OK  # read clears


@pytest.mark.slow
def test_logprob_config3_full_size_sampled_rows(c8):
    T, H, V = 4096, 4096, 151936
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=2, device=DEV)
    out = B.selected_logprob(c8, h, W, ids)
    rows = torch.tensor([0, 1, 777, 2048, 4095], device=DEV)
    ref = oracle.selected_logprob(bits(h[rows]), bits(W), ids[rows].cpu().numpy(), 8)
    assert np.max(np.abs(out[rows].cpu().double().numpy() - ref["out"])) <= 1e-3
    assert torch.all(out <= 0) and not torch.any(torch.isnan(out))
    # decode-style M = 1 calls give the packed-prefill bits
    for t in (0, 777, 4095):
        one = B.selected_logprob(c8, h[t:t + 1].contiguous(), W, ids[t:t + 1].contiguous())
        assert f32_same(one, out[t:t + 1])


# ------------------------------------------------------------------ RMSNorm
@pytest.mark.parametrize("T,H", [(33, 4096), (5, 2048), (17, 1000 * 8 // 8), (3, 8192), (64, 776)])
def test_rmsnorm_vs_oracle(c8, T, H):
    x, gamma = inputs.rmsnorm_inputs(T, H, seed=H)
    y = B.rmsnorm(c8, x.to(DEV), gamma.to(DEV), 1e-6)
    ref, ye = oracle.rmsnorm(bits(x), bits(gamma), 1e-6, exact=True)
    got = oracle.bf16_to_f64(bits(y))
    ulp = np.spacing(np.abs(oracle.bf16_to_f64(ref)).astype(np.float32)) * 65536
    assert np.all(np.abs(got - ye) <= ulp * 1.01)
    assert np.mean(bits(y) == ref) > 0.99


def test_rmsnorm_batch_invariance_bitwise(c8):
    x, gamma = inputs.rmsnorm_inputs(1000, 4096, seed=4)
    xd, gd = x.to(DEV), gamma.to(DEV)
    full = B.rmsnorm(c8, xd, gd, 1e-6)
    for t in (0, 5, 999):
        assert torch.equal(B.rmsnorm(c8, xd[t:t + 1].contiguous(), gd, 1e-6).view(torch.int16),
                           full[t:t + 1].view(torch.int16))
    perm = torch.randperm(1000, generator=torch.Generator().manual_seed(0)).to(DEV)
    assert torch.equal(B.rmsnorm(c8, xd[perm].contiguous(), gd, 1e-6).view(torch.int16), full[perm].view(torch.int16))


@pytest.mark.parametrize("H", [1024, 2048, 4096])
def test_rmsnorm_large_batch_bulk_staged(c8, H):
    """Batches of >= 32768 rows run the bulk-staged kernel (rows copied into shared memory by
    bulk copies): sampled rows within one bf16 ulp of the oracle, rows computed alone (the
    register kernel) equal their rows of the batch bitwise, and so does a shuffled batch."""
    T = 40000
    x, gamma = inputs.rmsnorm_inputs(T, H, seed=H + 7)
    xd, gd = x.to(DEV), gamma.to(DEV)
    full = B.rmsnorm(c8, xd, gd, 1e-6)
    rows = torch.tensor([0, 1, 7, 8, 1215, 1216, 20011, T - 2, T - 1])
    sub = full[rows.to(DEV)]
    ref, ye = oracle.rmsnorm(bits(x[rows]), bits(gamma), 1e-6, exact=True)
    got = oracle.bf16_to_f64(bits(sub))
    ulp = np.spacing(np.abs(oracle.bf16_to_f64(ref)).astype(np.float32)) * 65536
    assert np.all(np.abs(got - ye) <= ulp * 1.01)
    for t in rows.tolist():
        assert torch.equal(B.rmsnorm(c8, xd[t:t + 1].contiguous(), gd, 1e-6).view(torch.int16),
                           full[t:t + 1].view(torch.int16)), t
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(1)).to(DEV)
    assert torch.equal(B.rmsnorm(c8, xd[perm].contiguous(), gd, 1e-6).view(torch.int16), full[perm].view(torch.int16))
    assert B.last_device_status(c8) == B.ISO_OK


def test_rmsnorm_constant_row(c8):
    H = 4096
    x = torch.full((2, H), 2.0, dtype=torch.bfloat16, device=DEV)
    g = torch.ones(H, dtype=torch.bfloat16, device=DEV)
    y = B.rmsnorm(c8, x, g, 0.0)
    assert torch.all(y.float() == 1.0)
    y0 = B.rmsnorm(c8, torch.zeros_like(x), g, 1e-6)
    assert torch.all(y0.float() == 0.0)


@pytest.mark.parametrize("T", [400, 600])
def test_logprob_cta_pairs_match_single_rows(c8, T):
    """H = 8192 with 8 leaves (1024 k each) runs the LM head on CTA pairs (256-row units;
    T = 400 with one 128-column tile per unit, T = 600 with whole chunks); every row must
    equal its own single-row (one CTA) result, and sampled rows the oracle."""
    H, V = 8192, 128 * 19 * 2 + 40
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=8, device=DEV)
    full = B.selected_logprob(c8, h, W, ids)
    for t in (0, 255, 256, T - 1):
        one = B.selected_logprob(c8, h[t:t + 1].contiguous(), W, ids[t:t + 1].contiguous())
        assert f32_same(one, full[t:t + 1]), t
    rows = torch.tensor([0, 300, T - 1], device=DEV)
    ref = oracle.selected_logprob(bits(h[rows]), bits(W), ids[rows].cpu().numpy(), 8)
    assert np.max(np.abs(full[rows].cpu().double().numpy() - ref["out"])) <= 1e-3


def test_logprob_one_leaf_deep_stage_pairs():
    """A one-leaf contract's logprob GEMM runs on CTA pairs with 128-k stages (H = 1088 ends on a
    half stage): within 1e-3 of the oracle, and rows equal their single-row results bitwise."""
    c1 = B.Contract(1)
    T, H, V = 300, 1088, 2440 * 2
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=77)
    hd, Wd, idd = h.to(DEV), W.to(DEV), ids.to(DEV)
    out = B.selected_logprob(c1, hd, Wd, idd)
    ref = oracle.selected_logprob(bits(h), bits(W), ids.numpy(), 1)
    assert np.max(np.abs(out.cpu().double().numpy() - ref["out"])) <= 1e-3
    for t in (0, 128, 256, 299):
        one = B.selected_logprob(c1, hd[t:t + 1].contiguous(), Wd, idd[t:t + 1].contiguous())
        assert f32_same(one, out[t:t + 1]), t
    assert B.last_device_status(c1) == B.ISO_OK


def test_logprob_tile_units_and_chunk_units_agree_bitwise(c8):
    """With the full workspace every 128-column tile is its own work unit and a fold kernel
    folds each chunk's tiles left to right; with the minimum workspace one CTA folds a whole
    chunk.  Same fold, same order: the bits must agree, for the whole batch and row subsets."""
    T, H, V = 700, 256, 151936
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=77, device=DEV)
    full = B.selected_logprob(c8, h, W, ids)  # tile units
    ws_min = torch.empty(B.selected_logprob_min_workspace(c8, T, V), dtype=torch.uint8, device=DEV)
    assert ws_min.numel() < B.selected_logprob_workspace(c8, T, V)
    assert f32_same(B.selected_logprob(c8, h, W, ids, ws=ws_min), full)  # chunk units
    for lo, hi in ((0, 1), (5, 69), (100, 612), (699, 700)):
        hs, ids_s = h[lo:hi].contiguous(), ids[lo:hi].contiguous()
        assert f32_same(B.selected_logprob(c8, hs, W, ids_s), full[lo:hi]), (lo, hi)
        wsm = torch.empty(B.selected_logprob_min_workspace(c8, hi - lo, V), dtype=torch.uint8, device=DEV)
        assert f32_same(B.selected_logprob(c8, hs, W, ids_s, ws=wsm), full[lo:hi]), (lo, hi)
    rows = torch.tensor([0, 350, 699], device=DEV)
    ref = oracle.selected_logprob(bits(h[rows]), bits(W), ids[rows].cpu().numpy(), 8)
    assert np.max(np.abs(full[rows].cpu().double().numpy() - ref["out"])) <= 1e-3


def test_logprob_workspace_below_minimum_is_rejected(c8):
    T, H, V = 8, 128, 2440
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=5, device=DEV)
    small = torch.empty(B.selected_logprob_min_workspace(c8, T, V) - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(B.IsoError):
        B.selected_logprob(c8, h, W, ids, ws=small)


# ------------------------------------------------------------ vocab-parallel
@pytest.mark.parametrize("T,H,splits", [
    (300, 512, [0]),
    (300, 512, [0, 2432]),
    (700, 256, [0, 2432 * 20, 2432 * 40]),
    (64, 512, [0, 2432 * 10, 2432 * 31, 2432 * 50]),
])
def test_vocab_parallel_partial_combine_equals_single_call_bitwise(c8, T, H, splits):
    """Shards of the vocabulary (simulated ranks on column slices of W) compute their chunk
    statistics and owned selected logits; the combine over the rank-ordered concatenation
    must give the single call's bits, with one-tile or whole-chunk units per shard."""
    V = 151936
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=T + H, device=DEV)
    ref = B.selected_logprob(c8, h, W, ids)
    bounds = splits + [V]
    for tile_units in (True, False):
        stats, zs = [], []
        for r in range(len(splits)):
            v0, v1 = bounds[r], bounds[r + 1]
            ws = None if tile_units else torch.empty(16, dtype=torch.uint8, device=DEV)
            s_r, z_r = B.selected_logprob_partial(c8, h, W[:, v0:v1], ids, V, v0, ws=ws)
            stats.append(s_r)
            zs.append(z_r)
        out = B.selected_logprob_combine(c8, splits, torch.cat(stats, 0), torch.stack(zs), ids, V)
        assert f32_same(out, ref), (splits, tile_units)
    assert B.last_device_status(c8) == B.ISO_OK


def test_vocab_parallel_rejects_unaligned_shards(c8):
    T, H, V = 4, 128, 151936
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=3, device=DEV)
    with pytest.raises(B.IsoError):
        B.selected_logprob_partial(c8, h, W[:, 128:4992], ids, V, 128)  # v0 not chunk-aligned
    with pytest.raises(B.IsoError):
        B.selected_logprob_partial(c8, h, W[:, 0:2560], ids, V, 0)  # ragged shard that does not end at V
    stats = torch.zeros(63, T, 2, device=DEV)
    with pytest.raises(B.IsoError):
        B.selected_logprob_combine(c8, [0, 2500], stats, torch.zeros(2, T, device=DEV), ids, V)


def test_logprob_rows_span_several_l2_groups():
    """T = 7000 rows of H = 4096: more row blocks than one L2 raster group holds (the units run
    group by group, chunk-major inside a group), with a ragged last group.  Each row's logprob is
    the same bits as in a call of that row alone, and within 1e-3 of the oracle."""
    c = B.Contract(8)
    T, H, V = 7000, 4096, 2432 * 2 + 256
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=71, device=DEV)
    full = B.selected_logprob(c, h, W, ids)
    ws_min = torch.empty(B.selected_logprob_min_workspace(c, T, V), dtype=torch.uint8, device=DEV)
    assert torch.equal(B.selected_logprob(c, h, W, ids, ws=ws_min), full)
    rows = [0, 255, 256, 6143, 6144, 6999]
    for r in rows:
        assert torch.equal(B.selected_logprob(c, h[r:r + 1].contiguous(), W, ids[r:r + 1].contiguous()), full[r:r + 1]), r
    idx = torch.tensor(rows, device=DEV)
    ref = oracle.selected_logprob(bits(h[idx]), bits(W), ids[idx].cpu().numpy(), 8)["out"]
    assert np.max(np.abs(full[idx].cpu().double().numpy() - ref)) <= 1e-3
    assert B.last_device_status(c) == B.ISO_OK
