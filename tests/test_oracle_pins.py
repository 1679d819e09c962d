"""Pins of the float64 oracle against things other than itself: exact rational
brute force, exact-integer inputs, closed forms, identities, textbook/library
routines for special cases, and worked examples printed on the pages
(``tests/golden``).  Each pin is chosen so a plausible mistake (a dropped term,
a wrong sign or index, a transposed operand, a wrong tree shape) fails it."""
import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from parallelism_invariant_logprob_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(b):
    return oracle.bf16_to_f64(b)


def bf16_bits_of(values):
    return bits(torch.tensor(values, dtype=torch.float32).to(torch.bfloat16))


# ----------------------------------------------------------------- bf16 round
def _nearest_bf16_exact(x: Fraction) -> Fraction:
    """Brute force: nearest bf16 value (ties to even significand) by search."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = math.floor(math.log2(a)) if a > 0 else 0
    # fix e so 2^e <= a < 2^(e+1)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (max(e, -126) - 7)  # spacing of bf16 values near a
    lo = (a // q) * q
    hi = lo + q
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        r = lo if (lo / q) % 2 == 0 else hi
    return sign * r


def test_round_bf16_matches_library_on_float32_values():
    g = torch.Generator().manual_seed(11)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 8)
    ref = bits(x.to(torch.bfloat16))  # torch's float32 -> bf16 is round-to-nearest-even
    got = oracle.round_bf16(x.double().numpy())
    assert np.array_equal(got, ref)


def test_round_bf16_matches_exact_brute_force_on_doubles():
    rng = np.random.default_rng(5)
    xs = list(rng.standard_normal(300) * 10.0 ** rng.integers(-30, 30, 300))
    # exact midpoints between bf16 neighbours (ties) and values just off them
    for b in [1.0, 1.0 + 2 ** -7, 3.0, 1e-3]:
        mid = b + 2 ** (math.floor(math.log2(b)) - 8)
        xs += [mid, -mid, mid * (1 + 2 ** -40), mid * (1 - 2 ** -40)]
    got = f64(oracle.round_bf16(np.array(xs)))
    for x, g in zip(xs, got):
        assert Fraction(g) == _nearest_bf16_exact(Fraction(x)), x


# ---------------------------------------------------------------------- GEMM
def _exact_dot(a_row, B, j):
    return sum(Fraction(float(a)) * Fraction(float(B[k, j])) for k, a in enumerate(a_row))


@pytest.mark.parametrize("M,K,N,L", [(3, 8, 5, 4), (2, 6, 7, 2), (4, 16, 3, 8), (1, 5, 4, 1)])
def test_gemm_root_exact_brute_force(M, K, N, L):
    A, B = inputs.gemm_inputs(M, K, N, seed=7)
    Ab, Bb = bits(A), bits(B)
    root = oracle.gemm_root(Ab, Bb, L)
    Af, Bf = f64(Ab), f64(Bb)
    for i in range(M):
        for j in range(N):
            exact = _exact_dot(Af[i], Bf, j)
            bound = sum(abs(Af[i, k] * Bf[k, j]) for k in range(K)) * 1e-15 + 1e-300
            assert abs(Fraction(root[i, j]) - exact) <= Fraction(bound), (i, j)


def test_gemm_exact_integer_inputs_equal_integer_matmul():
    A = inputs.small_int_bf16((9, 64), -4, 4, seed=3)
    B = inputs.small_int_bf16((64, 11), -4, 4, seed=4)
    ref = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy()
    for L in (1, 2, 4, 8):
        root = oracle.gemm_root(bits(A), bits(B), L)
        assert np.array_equal(root, ref.astype(np.float64))
        assert np.array_equal(oracle.gemm(bits(A), bits(B), L), bits(torch.tensor(ref, dtype=torch.float32).to(torch.bfloat16)))


def test_gemm_identity_and_permutation():
    A, _ = inputs.gemm_inputs(6, 32, 1, seed=9)
    I = torch.eye(32, dtype=torch.bfloat16)
    assert np.array_equal(oracle.gemm(bits(A), bits(I), 4), bits(A))
    perm = torch.randperm(32, generator=torch.Generator().manual_seed(2))
    Pm = I[:, perm]  # column j of Pm picks row perm[j] of B's identity -> C[:, j] = A[:, perm[j]]
    assert np.array_equal(oracle.gemm(bits(A), bits(Pm), 8), bits(A[:, perm]))


def test_gemm_single_leaf_is_textbook_matmul():
    A, B = inputs.gemm_inputs(17, 96, 23, seed=1)
    root = oracle.gemm_root(bits(A), bits(B), 1)
    ref = f64(bits(A)) @ f64(bits(B))
    assert np.allclose(root, ref, rtol=1e-13, atol=1e-13)


def test_gemm_tree_shape_golden():
    fx = json.load(open(os.path.join(GOLDEN, "tree_shape_fixture.json")))
    leaves = fx["f64_leaves"]
    L = len(leaves)
    A = np.array([bf16_bits_of([1.0] * L)])
    B = bf16_bits_of([[v] for v in leaves])
    assert np.array_equal(f64(B).ravel(), np.array(leaves))
    root = oracle.gemm_root(A, B, L)
    assert root[0, 0] == fx["f64_balanced_tree"]
    assert root[0, 0] != fx["f64_left_fold"] and root[0, 0] != fx["f64_right_fold"]
    # the same tree seen as two simulated ranks of two leaves each
    S = np.stack([oracle.gemm_leaf_partial(A[:, 2 * r:2 * r + 2], B[2 * r:2 * r + 2], L, 2) for r in range(2)])
    assert oracle.tree_combine(S)[0, 0] == fx["f64_balanced_tree"]


def test_gemm_tree_shape_sixteen_leaves():
    # leaf 0 = 2^53, leaf 8 = 1, leaf 15 = -2^53 (float64): the balanced tree's top add is
    # 2^53 + (1 - 2^53) = 1; a left fold gives (2^53 + 1) - 2^53 = 0 (2^53 + 1 rounds to 2^53)
    L = 16
    vals = [0.0] * L
    vals[0], vals[8], vals[15] = 2.0 ** 53, 1.0, -(2.0 ** 53)
    A = np.array([bf16_bits_of([1.0] * L)])
    B = bf16_bits_of([[v] for v in vals])
    assert oracle.gemm_root(A, B, L)[0, 0] == 1.0
    fold = 0.0
    for v in vals:
        fold += v
    assert fold == 0.0
    S = np.stack([oracle.gemm_leaf_partial(A[:, 8 * r:8 * r + 8], B[8 * r:8 * r + 8], L, 2) for r in range(2)])
    assert oracle.tree_combine(S)[0, 0] == 1.0


@pytest.mark.parametrize("R", [1, 2, 4, 8, 16])
def test_gemm_partial_plus_combine_sixteen_leaves(R):
    L = 16
    A, B = inputs.gemm_inputs(3, 256, 11, seed=9)
    Ab, Bb = bits(A), bits(B)
    full = oracle.gemm_root(Ab, Bb, L)
    Kl = 256 // R
    S = np.stack([oracle.gemm_leaf_partial(Ab[:, r * Kl:(r + 1) * Kl], Bb[r * Kl:(r + 1) * Kl], L, R)
                  for r in range(R)])
    assert np.array_equal(oracle.tree_combine(S), full)


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_gemm_partial_plus_combine_equals_single_pass(R):
    L = 8
    A, B = inputs.gemm_inputs(5, 128, 9, seed=4)
    Ab, Bb = bits(A), bits(B)
    full = oracle.gemm_root(Ab, Bb, L)
    Kl = 128 // R
    S = np.stack([oracle.gemm_leaf_partial(Ab[:, r * Kl:(r + 1) * Kl], Bb[r * Kl:(r + 1) * Kl], L, R)
                  for r in range(R)])
    assert np.array_equal(oracle.tree_combine(S), full)
    # rank r's subtree root equals the oracle's own subtree over leaves of rank r
    for r in range(R):
        sub = oracle.gemm_root(Ab, Bb, L, leaf_lo=r * (L // R), leaf_hi=(r + 1) * (L // R))
        assert np.array_equal(S[r], sub)


def test_gemm_rejects_unproven_shapes():
    A, B = inputs.gemm_inputs(2, 12, 3, seed=0)
    with pytest.raises(ValueError):
        oracle.gemm_root(bits(A), bits(B), 3)  # leaf count not a power of two
    with pytest.raises(ValueError):
        oracle.gemm_root(bits(A), bits(B), 8)  # K not divisible by L


# ------------------------------------------------------------------- RMSNorm
def test_rmsnorm_brute_force_decimal():
    getcontext().prec = 50
    x, gamma = inputs.rmsnorm_inputs(3, 40, seed=6)
    eps = 1e-6
    y, ye = oracle.rmsnorm(bits(x), bits(gamma), eps, exact=True)
    xf, gf = f64(bits(x)), f64(bits(gamma))
    for t in range(3):
        ss = sum(Decimal(float(v)) ** 2 for v in xf[t])
        r = 1 / (ss / Decimal(40) + Decimal(eps)).sqrt()
        for i in range(40):
            ref = Decimal(float(xf[t, i])) * r * Decimal(float(gf[i]))
            assert abs(Decimal(ye[t, i]) - ref) <= abs(ref) * Decimal(1e-14) + Decimal(1e-300)
    assert np.array_equal(y, oracle.round_bf16(ye))


def test_rmsnorm_constant_row_closed_form():
    H = 64
    for c in (1.0, -3.0, 0.5):
        x = bf16_bits_of([[c] * H])
        _, gamma = inputs.rmsnorm_inputs(1, H, seed=2)
        y, ye = oracle.rmsnorm(x, bits(gamma), 1e-6, exact=True)
        gf = f64(bits(gamma))
        ref = np.sign(c) * gf * abs(c) / math.sqrt(c * c + 1e-6)
        assert np.allclose(ye[0], ref, rtol=1e-15, atol=0)
    y = oracle.rmsnorm(bf16_bits_of([[2.0] * H]), bf16_bits_of([1.0] * H), 0.0)
    assert np.array_equal(f64(y), np.ones((1, H)))
    y = oracle.rmsnorm(bf16_bits_of([[0.0] * H]), bf16_bits_of([1.0] * H), 1e-6)
    assert np.array_equal(f64(y), np.zeros((1, H)))


# ------------------------------------------------------------------- logprob
def test_lse_merge_closed_form():
    for a, b in [(0.3, -1.2), (5.0, 5.0), (-40.0, 2.0)]:
        m, s = oracle.lse_merge(a, 1.0, b, 1.0)
        assert abs((m + math.log(s)) - math.log(math.exp(a) + math.exp(b))) < 1e-14
    # empty block is the identity
    assert oracle.lse_merge(-math.inf, 0.0, 1.5, 2.0) == (1.5, 2.0)
    assert oracle.lse_merge(1.5, 2.0, -math.inf, 0.0) == (1.5, 2.0)


def _brute_logprob(h, W, ids, L):
    z = oracle.gemm_root(h, W, L)
    out = []
    for t in range(z.shape[0]):
        m = max(z[t])
        lse = m + math.log(math.fsum(math.exp(v - m) for v in z[t]))
        out.append(z[t, ids[t]] - lse)
    return np.array(out), z


@pytest.mark.parametrize("V,tile,chunk", [(3, 128, 19), (129, 128, 19), (128 * 19 + 1, 128, 19), (29, 4, 3), (64, 8, 2)])
def test_selected_logprob_brute_force(V, tile, chunk):
    h, W, ids = inputs.logprob_inputs(4, 32, V, seed=8)
    r = oracle.selected_logprob(bits(h), bits(W), ids.numpy(), 4, tile_cols=tile, chunk_tiles=chunk, chunk_stats=True)
    ref, z = _brute_logprob(bits(h), bits(W), ids.numpy(), 4)
    assert np.allclose(r["out"], ref, rtol=0, atol=1e-12)
    assert np.allclose(r["lse"], r["lse_direct"], rtol=0, atol=1e-12)
    assert np.all(r["out"] <= 0)
    assert r["chunk_m"].shape[1] == oracle.num_chunks(V, tile, chunk)


def test_logprob_full_distribution_sums_to_one():
    V = 77
    h, W, _ = inputs.logprob_inputs(3, 64, V, seed=12)
    for t in range(3):
        ids = np.arange(V, dtype=np.int32)
        hh = np.repeat(bits(h)[t:t + 1], V, axis=0)
        r = oracle.selected_logprob(hh, bits(W), ids, 8, tile_cols=8, chunk_tiles=3)
        assert abs(math.log(math.fsum(math.exp(v) for v in r["out"]))) < 1e-12
        assert np.all(r["out"] <= 0)


def test_logprob_zero_weights_is_uniform():
    V = 1000
    h, _, ids = inputs.logprob_inputs(5, 16, V, seed=1)
    W = np.zeros((16, V), np.uint16)
    r = oracle.selected_logprob(bits(h), W, ids.numpy(), 2, tile_cols=128, chunk_tiles=3)
    assert np.allclose(r["out"], -math.log(V), rtol=0, atol=1e-13)


def test_logprob_dominant_logit():
    V, H = 50, 16
    h = bf16_bits_of([[1.0] * H])
    Wf = np.zeros((H, V), np.float32)
    Wf[:, 7] = 8.0  # z[7] = 128, others 0
    r = oracle.selected_logprob(h, bf16_bits_of(Wf), np.array([7], np.int32), 4, tile_cols=8, chunk_tiles=2)
    assert abs(r["out"][0]) < 1e-50
    r2 = oracle.selected_logprob(h, bf16_bits_of(Wf), np.array([3], np.int32), 4, tile_cols=8, chunk_tiles=2)
    assert abs(r2["out"][0] + 128.0) < 1e-12


def test_logprob_invalid_id_is_nan():
    h, W, _ = inputs.logprob_inputs(1, 16, 10, seed=3)
    r = oracle.selected_logprob(bits(h), bits(W), np.array([10], np.int32), 2)
    assert math.isnan(r["out"][0])


# ----------------------------------------------------------------------- MoE
def test_moe_route_matches_library_sort_with_ties():
    T, E, k = 40, 16, 4
    g = torch.Generator().manual_seed(4)
    logits = torch.randint(-3, 4, (T, E), generator=g).float()  # many ties
    ids, w = oracle.moe_route(logits.numpy(), k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].numpy()))  # primary: logit desc, then id asc
        assert list(ids[t]) == list(order[:k])
        full = np.exp(logits[t].double().numpy() - logits[t].max().item())
        ren = full[order[:k]] / full[order[:k]].sum()
        assert np.allclose(w[t], ren, rtol=1e-14, atol=0)
        assert abs(w[t].sum() - 1.0) < 1e-14


def test_moe_permute_is_stable_sort():
    T, E, k = 33, 8, 2
    _, _, _, logits = inputs.moe_inputs(T, 8, E, 8, seed=2)
    ids, _ = oracle.moe_route(logits.numpy(), k)
    perm, offs = oracle.moe_permute(ids, E)
    ref = np.argsort(ids.ravel(), kind="stable")
    assert np.array_equal(perm, ref)
    assert np.array_equal(np.diff(offs), np.bincount(ids.ravel(), minlength=E))
    mask = np.array([1, 0, 1, 0, 0, 1, 1, 0], np.uint8)
    pm, om = oracle.moe_permute(ids, E, mask)
    keep = mask[ids.ravel()] == 1
    assert np.array_equal(pm, np.arange(T * k)[keep][np.argsort(ids.ravel()[keep], kind="stable")])
    assert om[-1] == keep.sum()


def _silu_ffn_reference(x, W1, W2, L):
    """k = 1, gate 1: the expert layer reduces to a dense SwiGLU FFN.  Matmuls
    by numpy; bf16 rounding by the separately pinned helper."""
    F = W2.shape[0]
    G = f64(x) @ f64(W1)
    g = f64(oracle.round_bf16(G[:, :F]))
    u = f64(oracle.round_bf16(G[:, F:]))
    h = oracle.round_bf16(g / (1.0 + np.exp(-g)) * u)
    return oracle.round_bf16(f64(h) @ f64(W2))


def test_moe_single_slot_reduces_to_dense_ffn():
    T, H, E, F = 6, 32, 3, 16
    x, W1, W2, _ = inputs.moe_inputs(T, H, E, F, seed=5)
    W1 = (W1.float() * 20).to(torch.bfloat16)  # larger weights so SwiGLU is far from linear
    ids = np.array([[t % E] for t in range(T)], np.int32)
    w = np.ones((T, 1))
    r = oracle.moe_layer(bits(x), ids, w, bits(W1), bits(W2), 4)
    for t in range(T):
        e = ids[t, 0]
        ref = _silu_ffn_reference(bits(x)[t:t + 1], bits(W1)[e], bits(W2)[e], 4)
        assert np.array_equal(r["out"][t:t + 1], ref)


def test_moe_combine_onehot_and_equal_gates():
    T, k, H = 4, 8, 24
    y = bits(inputs.normal_bf16((T, k, H), 1.0, seed=3))
    for j in range(k):
        w = np.zeros((T, k))
        w[:, j] = 1.0
        assert np.array_equal(oracle.moe_combine(y, w), y[:, j])
    same = np.repeat(y[:, :1], k, axis=1)
    assert np.array_equal(oracle.moe_combine(same, np.full((T, k), 1.0 / k)), y[:, 0])


def test_moe_layer_slots_match_combine():
    T, H, E, F, k = 5, 16, 4, 8, 2
    x, W1, W2, logits = inputs.moe_inputs(T, H, E, F, seed=9)
    ids, w = oracle.moe_route(logits.numpy(), k)
    r = oracle.moe_layer(bits(x), ids, w, bits(W1), bits(W2), 2, with_slots=True)
    assert np.array_equal(oracle.moe_combine(r["y_slots"], w), r["out"])


# ------------------------------------------------------------------- delta_t
def test_delta_matches_vexact_table1():
    fx = json.load(open(os.path.join(GOLDEN, "vexact_table1_delta.json")))
    d = oracle.delta(np.array(fx["logp_train"]), np.array(fx["logp_rollout"]))
    tol = 10.0 ** -fx["printed_decimals"] * 1.01  # both printed operands and the printed delta are rounded
    assert np.all(np.abs(d - np.array(fx["delta"])) <= tol)
    assert np.argmax(np.abs(d)) == 3


def test_delta_matches_rlkernel_minimal_example():
    fx = json.load(open(os.path.join(GOLDEN, "rlkernel_minimal_example.json")))
    d = oracle.delta(np.array([fx["train_logp"]]), np.array([fx["rollout_logp"]]))[0]
    assert abs(d - fx["delta"]) < 1e-12
    assert abs(math.exp(d) - fx["ratio_single_token_approx"]) < 5e-4
    assert abs(fx["tokens"] * d - fx["cumulative_delta"]) < 1e-9
    assert abs(math.exp(fx["tokens"] * d) - fx["ratio_cumulative_approx"]) < 5e-3


# ------------------------------------------------------- mismatch diagnostics
# VeXact paper: delta_t (§2 Eq. 1), K1 / K3 (§4.1), TIS min(r_corr, tau_tok) (§4.2 Eq. 6),
# sequence rejection 1[sum_t K(r_corr,t) <= tau_seq] (Eq. 7-11, tau_tok = 2, tau_seq = 0.001).
def _f32(x):
    return float(np.float32(x))


def test_mismatch_table1_delta_and_identity_rows():
    g = json.load(open(os.path.join(GOLDEN, "vexact_table1_delta.json")))
    tr = np.array(g["logp_train"], np.float32)
    ro = np.array(g["logp_rollout"], np.float32)
    r = oracle.mismatch(tr, ro, [0, len(tr)])
    assert np.allclose(np.round(r["delta"], 3), g["delta"], atol=1e-12)
    # the printed 3-decimal values differ in 3 of 8 positions
    assert r["seq_mismatches"][0] == 3
    assert r["seq_max_abs_delta"][0] == pytest.approx(0.133, abs=1e-6)
    same = oracle.mismatch(tr, tr, [0, 4, 8])
    assert np.all(same["delta"] == 0) and np.all(same["tis_weight"] == 1.0)
    assert np.all(same["seq_k1"] == 0) and np.all(same["seq_k3"] == 0)
    assert list(same["accept_k1"]) == [1, 1] and list(same["accept_k3"]) == [1, 1]
    assert list(same["seq_mismatches"]) == [0, 0]


def test_mismatch_closed_forms_and_truncation():
    # rollout assigns a third of the training probability: r_corr = 3 -> weight truncated at tau_tok = 2
    tr = np.array([0.0, -1.0, -0.5], np.float32)
    ro = np.array([_f32(-math.log(3.0)), -1.25, -0.25], np.float32)
    r = oracle.mismatch(tr, ro, [0, 3])
    d = [float(tr[i]) - float(ro[i]) for i in range(3)]
    assert list(r["delta"]) == d  # train minus rollout, in that order
    rc = [math.exp(x) for x in d]
    assert r["tis_weight"][0] == 2.0 and rc[0] > 2.0
    assert r["tis_weight"][1] == pytest.approx(rc[1], rel=1e-15) and rc[1] < 2.0
    assert r["tis_weight"][2] == pytest.approx(rc[2], rel=1e-15) and rc[2] < 1.0
    k1 = math.fsum(-x for x in d)
    k3 = math.fsum((math.exp(x) - 1.0) - x for x in d)
    assert r["seq_k1"][0] == pytest.approx(k1, abs=1e-15)
    assert r["seq_k3"][0] == pytest.approx(k3, rel=1e-14)
    assert r["seq_k3"][0] > 0  # K3 is a non-negative estimator
    assert r["seq_k1"][0] == pytest.approx(-0.0 - sum(d), abs=1e-15)


def test_mismatch_sequence_sums_brute_force_and_masks():
    rng = np.random.default_rng(7)
    lens = [0, 1, 5, 300, 17, 2049]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = int(offs[-1])
    ro = (-np.abs(rng.standard_normal(n)) * 2).astype(np.float32)
    tr = (ro + (rng.standard_normal(n) * 1e-3)).astype(np.float32)
    r = oracle.mismatch(tr, ro, offs)
    for b in range(len(lens)):
        seg = range(offs[b], offs[b + 1])
        d = [float(tr[t]) - float(ro[t]) for t in seg]
        s1 = math.fsum(-x for x in d)
        s3 = math.fsum((math.exp(x) - 1.0) - x for x in d)
        assert r["seq_k1"][b] == pytest.approx(s1, abs=1e-12)
        assert r["seq_k3"][b] == pytest.approx(s3, rel=1e-9, abs=1e-18)
        assert r["accept_k1"][b] == (1 if s1 <= 0.001 else 0)
        assert r["accept_k3"][b] == (1 if s3 <= 0.001 else 0)
        assert r["seq_max_abs_delta"][b] == (max(abs(x) for x in d) if d else 0.0)
        assert r["seq_mismatches"][b] == sum(1 for t in seg if tr[t] != ro[t])
    assert r["accept_k1"][0] == 1 and r["seq_k1"][0] == 0.0  # an empty sequence is accepted
    # K3 ~ delta^2 / 2 for small delta
    small = oracle.mismatch(np.array([1e-3], np.float32), np.array([0.0], np.float32), [0, 1])
    dd = float(np.float32(1e-3))
    assert small["seq_k3"][0] == pytest.approx(dd * dd / 2 + dd ** 3 / 6, rel=1e-6)


def test_mismatch_rejection_threshold_sides():
    # S_K1 = -sum(delta): 0.0005 is accepted, 0.002 is rejected (tau_seq = 0.001)
    ro = np.zeros(4, np.float32)
    acc = oracle.mismatch(np.full(4, -0.000125, np.float32), ro, [0, 4])
    rej = oracle.mismatch(np.full(4, -0.0005, np.float32), ro, [0, 4])
    assert acc["accept_k1"][0] == 1 and acc["seq_k1"][0] == pytest.approx(0.0005, rel=1e-6)
    assert rej["accept_k1"][0] == 0 and rej["seq_k1"][0] == pytest.approx(0.002, rel=1e-6)


# ------------------------------------------------------------------- attention
# RL-Kernel blog §4: softmax over the visible keys (causal), the LSE statistic.
def _bf16_np(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _from_bits(b):
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().double().numpy()


def _attn_case(seed, lens_q, lens_k, pos0, Hq=4, Hkv=2, d=16):
    rng = np.random.default_rng(seed)
    Tq, Tk = sum(lens_q), sum(lens_k)
    Q = _bf16_np(rng.standard_normal((Tq, Hq, d)))
    K = _bf16_np(rng.standard_normal((Tk, Hkv, d)))
    V = _bf16_np(rng.standard_normal((Tk, Hkv, d)))
    qs = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ks = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    return Q, K, V, qs, ks, np.array(pos0, np.int32)


def test_attention_matches_numpy_brute_force():
    Q, K, V, qs, ks, p0 = _attn_case(3, [5, 3], [5, 9], [0, 6])
    scale = 0.25
    r = oracle.attention(Q, K, V, qs, ks, p0, scale)
    Qf, Kf, Vf = _from_bits(Q), _from_bits(K), _from_bits(V)
    for b in range(2):
        for i in range(qs[b + 1] - qs[b]):
            row, p = qs[b] + i, p0[b] + i
            for h in range(4):
                g = h // 2  # 4 query heads over 2 KV heads
                keys = Kf[ks[b]:ks[b] + p + 1, g]
                s = scale * (keys @ Qf[row, h])
                w = np.exp(s - s.max())
                want = (w[:, None] * Vf[ks[b]:ks[b] + p + 1, g]).sum(0) / w.sum()
                assert np.allclose(r["out_exact"][row, h], want, rtol=1e-12, atol=1e-12)
                assert r["lse"][row, h] == pytest.approx(s.max() + math.log(w.sum()), abs=1e-12)
    # bf16 output is the round-to-nearest of the exact value (round_bf16 is pinned above)
    assert np.array_equal(r["out"], oracle.round_bf16(r["out_exact"]))


def test_attention_special_cases():
    Q, K, V, qs, ks, p0 = _attn_case(4, [6], [6], [0])
    r = oracle.attention(Q, K, V, qs, ks, p0, 0.3)
    # position 0 sees one key: the output is that value row exactly
    assert np.array_equal(r["out"][0], V[0, [0, 0, 1, 1]])
    # zero queries give equal scores: the mean of the visible values, lse = log(count)
    Z = np.zeros_like(Q)
    rz = oracle.attention(Z, K, V, qs, ks, p0, 0.3)
    Vf = _from_bits(V)
    for i in range(6):
        assert np.allclose(rz["out_exact"][i, 0], Vf[:i + 1, 0].mean(0), atol=1e-12)
        assert rz["lse"][i, 0] == pytest.approx(math.log(i + 1), abs=1e-12)
    # causality: changing keys / values past a row's position leaves the row unchanged
    K2, V2 = K.copy(), V.copy()
    K2[4:] ^= 0x0100
    V2[4:] ^= 0x0100
    r2 = oracle.attention(Q, K2, V2, qs, ks, p0, 0.3)
    assert np.array_equal(r2["out_exact"][:4], r["out_exact"][:4])
    assert not np.array_equal(r2["out_exact"][4:], r["out_exact"][4:])
