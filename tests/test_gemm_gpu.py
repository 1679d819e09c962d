"""GPU parity and invariance of iso_gemm / iso_gemm_leaf_partial /
iso_tree_combine, through the C ABI, against the float64 oracle.

Tolerance (floating point): per row, max |C_gpu - C_oracle| <= 2e-2 * ||C_oracle row||_2.
Exact-integer inputs and single-term (identity / permutation) products are
exact in every summation order, so there the bits must be equal."""
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


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def first_diff(a, b):
    x, y = bits(a), bits(b)
    idx = np.argwhere(x != y)
    if len(idx) == 0:
        return None
    i = tuple(idx[0])
    return f"first differing element {i}: {x[i]:#06x} vs {y[i]:#06x} ({len(idx)} differ)"


def check_row_tolerance(C, root):
    got = oracle.bf16_to_f64(bits(C))
    err = np.abs(got - root).max(axis=1)
    bound = 2e-2 * np.linalg.norm(root, axis=1)
    bad = np.nonzero(err > bound)[0]
    assert len(bad) == 0, f"rows {bad[:8]} exceed 2e-2 * row norm: err {err[bad[:4]]} bound {bound[bad[:4]]}"
    # tighter: one bf16 ulp of the defined value, plus fp32-accumulation slack
    ulp = np.spacing(np.abs(oracle.bf16_to_f64(oracle.round_bf16(root))).astype(np.float32)) * 65536
    slack = 1e-5 * np.linalg.norm(root, axis=1, keepdims=True)
    assert np.all(np.abs(got - root) <= ulp + slack)


@pytest.fixture(scope="module")
def c4():
    return B.Contract(4)


@pytest.fixture(scope="module")
def c8():
    return B.Contract(8)


@pytest.mark.parametrize("M", [1, 7, 32])
def test_config1_exact_integer_bits_equal_oracle(c4, M):
    A = inputs.small_int_bf16((M, 2048), -4, 4, seed=10 + M)
    Bm = inputs.small_int_bf16((2048, 512), -4, 4, seed=20 + M)
    C = B.gemm(c4, A.to(DEV), Bm.to(DEV))
    ref = oracle.gemm(bits(A), bits(Bm), 4)
    assert np.array_equal(bits(C), ref), first_diff(C, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16))


@pytest.mark.parametrize("M,N,K,L", [(300, 392, 1024, 8), (129, 136, 256, 1), (5, 1024, 4096, 8), (64, 256, 768, 8)])
def test_exact_integer_multi_tile_ragged(M, N, K, L):
    c = B.Contract(L)
    A = inputs.small_int_bf16((M, K), -3, 3, seed=M)
    Bm = inputs.small_int_bf16((K, N), -3, 3, seed=N)
    C = B.gemm(c, A.to(DEV), Bm.to(DEV))
    assert np.array_equal(bits(C), oracle.gemm(bits(A), bits(Bm), L))


@pytest.mark.parametrize("M,K", [(1, 1024), (7, 768), (16, 512), (33, 1024)])
def test_short_leaves_small_m_exact_and_row_invariant(c8, M, K):
    # leaves of 64-128 k with few rows: 8 epilogue warps, A boxes of 16-64 rows, and (for
    # 16- and 32-row boxes) the unstaged store path; exact integers equal the oracle, and the
    # rows have the same bits as inside a 300-row product (staged stores, 128-row boxes)
    N = 392
    A = inputs.small_int_bf16((300, K), -3, 3, seed=K + M)
    Bm = inputs.small_int_bf16((K, N), -3, 3, seed=K)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    C = B.gemm(c8, Ad[:M].contiguous(), Bd)
    assert np.array_equal(bits(C), oracle.gemm(bits(A[:M]), bits(Bm), 8))
    An = inputs.gemm_inputs(300, K, N, seed=M)[0].to(DEV)
    Bn = inputs.gemm_inputs(300, K, N, seed=M + 1)[1].to(DEV)
    big = B.gemm(c8, An, Bn)
    assert same_bits(B.gemm(c8, An[:M].contiguous(), Bn), big[:M])


def test_identity_and_permutation_are_exact(c8):
    A, _ = inputs.gemm_inputs(200, 256, 1, seed=3)
    I = torch.eye(256, dtype=torch.bfloat16)
    assert same_bits(B.gemm(c8, A.to(DEV), I.to(DEV)).cpu(), A)
    perm = torch.randperm(256, generator=torch.Generator().manual_seed(1))
    assert same_bits(B.gemm(c8, A.to(DEV), I[:, perm].contiguous().to(DEV)).cpu(), A[:, perm])


def test_tree_shape_on_gpu(c4):
    # leaves (2^24, 1, 1, -2^24): the balanced tree gives 1, a left fold 0.
    K = 4 * 16
    A = torch.zeros(1, K, dtype=torch.bfloat16)
    Bm = torch.zeros(K, 8, dtype=torch.bfloat16)
    for l, v in enumerate([2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)]):
        A[0, l * 16] = 1.0
        Bm[l * 16, :] = v
    C = B.gemm(c4, A.to(DEV), Bm.to(DEV))
    assert torch.all(C.float().cpu() == 1.0)
    S = B.gemm_leaf_partial(B.Contract(4), 0, 1, A.to(DEV), Bm.to(DEV))
    assert torch.all(S.cpu() == 1.0)


@pytest.mark.parametrize("M,N,K", [(32, 512, 2048), (300, 392, 1024), (1000, 1024, 1536)])
def test_normal_inputs_within_tolerance(c8, M, N, K):
    A, Bm = inputs.gemm_inputs(M, K, N, seed=M + N)
    C = B.gemm(c8, A.to(DEV), Bm.to(DEV))
    check_row_tolerance(C, oracle.gemm_root(bits(A), bits(Bm), 8))


def test_config1_bitwise_invariance(c4):
    A, Bm = inputs.gemm_inputs(32, 2048, 512, seed=0)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    full = B.gemm(c4, Ad, Bd)
    check_row_tolerance(full, oracle.gemm_root(bits(A), bits(Bm), 4))
    for M in (1, 7):
        for start in (0, 3, 32 - M):
            part = B.gemm(c4, Ad[start:start + M].contiguous(), Bd)
            assert same_bits(part, full[start:start + M]), (M, start)
    perm = torch.randperm(32, generator=torch.Generator().manual_seed(5)).to(DEV)
    shuf = B.gemm(c4, Ad[perm].contiguous(), Bd)
    assert same_bits(shuf, full[perm])
    # rows embedded in a much larger batch, at other tile positions
    big = torch.cat([inputs.gemm_inputs(700, 2048, 1, seed=9)[0].to(DEV), Ad, Ad[:5]], dim=0)
    Cb = B.gemm(c4, big.contiguous(), Bd)
    assert same_bits(Cb[700:732], full) and same_bits(Cb[732:], full[:5])


@pytest.mark.parametrize("R", [1, 2, 4])
def test_config1_partial_combine_equals_single_pass(c4, R):
    A, Bm = inputs.gemm_inputs(32, 2048, 512, seed=0)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    full = B.gemm(c4, Ad, Bd)
    Kl = 2048 // R
    S = torch.stack([B.gemm_leaf_partial(c4, r, R, Ad[:, r * Kl:(r + 1) * Kl].contiguous(), Bd[r * Kl:(r + 1) * Kl])
                     for r in range(R)])
    C = B.tree_combine(c4, S)
    assert same_bits(C, full), first_diff(C, full)
    # the rank subtree roots match the oracle's subtree roots within fp32 rounding of the tree
    for r in range(R):
        sub = oracle.gemm_root(bits(A), bits(Bm), 4, leaf_lo=r * (4 // R), leaf_hi=(r + 1) * (4 // R))
        assert np.allclose(S[r].cpu().double().numpy(), sub, rtol=0, atol=1e-4 * np.abs(sub).max() + 1e-6)


@pytest.mark.parametrize("K,N", [(4096, 4096), (4096, 12288), (12288, 4096)])
def test_config2_shapes_sampled_rows_and_ranks(c8, K, N):
    M = 512
    A, Bm = inputs.gemm_inputs(M, K, N, seed=1)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    full = B.gemm(c8, Ad, Bd)
    rows = torch.tensor([0, 1, 127, 128, 300, 511])
    ref = oracle.gemm_root(bits(A[rows]), bits(Bm), 8)
    check_row_tolerance(full[rows.to(DEV)], ref)
    for M1 in (1, 8, 64):
        assert same_bits(B.gemm(c8, Ad[:M1].contiguous(), Bd), full[:M1])
    for R in (2, 4, 8):
        Kl = K // R
        S = torch.stack([B.gemm_leaf_partial(c8, r, R, Ad[:, r * Kl:(r + 1) * Kl].contiguous(),
                                             Bd[r * Kl:(r + 1) * Kl]) for r in range(R)])
        assert same_bits(B.tree_combine(c8, S), full), R


@pytest.mark.parametrize("R", [2, 4, 8])
def test_sp_reduce_scatter_slices_equal_rows_of_iso_gemm(c8, R):
    """Sequence parallelism [IsoExec blog, "Parallelism-invariant kernels": the row-parallel
    reduction becomes a reduce-scatter over the same tree; each rank keeps its output slice].
    Rank q's slice is the top tree levels over rows [q M / R, (q+1) M / R) of every rank's
    partial (iso_tree_combine on the row-offset view; the exchange only moves rows): the bits
    equal those rows of iso_gemm, for ragged slices (M = 1000 is not a multiple of 8)."""
    M, K, N = 1000, 4096, 520
    A, Bm = inputs.gemm_inputs(M, K, N, seed=77)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    full = B.gemm(c8, Ad, Bd)
    Kl = K // R
    S = torch.stack([B.gemm_leaf_partial(c8, r, R, Ad[:, r * Kl:(r + 1) * Kl].contiguous(), Bd[r * Kl:(r + 1) * Kl])
                     for r in range(R)])
    for q in range(R):
        r0, r1 = (q * M) // R, ((q + 1) * M) // R
        # in place on the rank-strided view, and after the exchange packs the slices contiguously
        Cq = B.tree_combine(c8, S[:, r0:r1])
        assert same_bits(Cq, full[r0:r1]), (R, q)
        assert same_bits(B.tree_combine(c8, S[:, r0:r1].contiguous()), full[r0:r1]), (R, q)


@pytest.mark.parametrize("M,K", [(129, 8192), (200, 8192), (257, 8192), (384, 8192), (129, 4096), (300, 4096)])
def test_cta_pair_units_ragged_exact(c8, M, K):
    """Leaves of 512 k and more (K = 4096 or 8192, 8 leaves) run on CTA pairs: a unit is 256
    rows, the second CTA's 128 rows may be partly or wholly past M.  Exact integer inputs: the
    bits must equal the oracle's, and every row must equal its single-row (one CTA) result."""
    N = 136
    A = inputs.small_int_bf16((M, K), -3, 3, seed=M)
    Bm = inputs.small_int_bf16((K, N), -3, 3, seed=N + M)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    C = B.gemm(c8, Ad, Bd)
    assert np.array_equal(bits(C), oracle.gemm(bits(A), bits(Bm), 8)), first_diff(
        C, torch.from_numpy(oracle.gemm(bits(A), bits(Bm), 8).view(np.int16)).view(torch.bfloat16))
    for r in (0, 128, M - 1):
        assert same_bits(B.gemm(c8, Ad[r:r + 1].contiguous(), Bd), C[r:r + 1]), r


@pytest.mark.parametrize("M,K", [(129, 576), (300, 1024), (257, 2048), (200, 528), (520, 640)])
def test_cta_pair_one_leaf_deep_stages_exact(M, K):
    """A one-leaf contract on CTA pairs stages 128 k at a time (A through the 3-D chunk view):
    K = 576 and 640 end on a half stage whose second chunk lies past K (zero-filled, unused);
    K = 528 is not a whole number of 64-k chunks and keeps 64-k stages.  Exact integers: the bits
    equal the oracle's one-leaf chain, and rows equal their single-row results."""
    c1 = B.Contract(1)
    N = 264
    A = inputs.small_int_bf16((M, K), -3, 3, seed=M + K)
    Bm = inputs.small_int_bf16((K, N), -3, 3, seed=N + K)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    C = B.gemm(c1, Ad, Bd)
    ref = oracle.gemm(bits(A), bits(Bm), 1)
    assert np.array_equal(bits(C), ref), first_diff(C, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16))
    for r in (0, 128, 255 if M > 255 else M - 1, M - 1):
        assert same_bits(B.gemm(c1, Ad[r:r + 1].contiguous(), Bd), C[r:r + 1]), r


def test_cta_pair_one_leaf_normal_inputs_partial_and_repeats():
    """Normal inputs on the one-leaf deep-stage pairs: sampled rows within tolerance of the
    oracle, repeated launches give the same bits, and the R = 1 leaf partial (fp32 root through
    the same pairs) + combine reproduces the single pass."""
    c1 = B.Contract(1)
    M, K, N = 1024, 4096, 1024
    A, Bm = inputs.gemm_inputs(M, K, N, seed=43)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    full = B.gemm(c1, Ad, Bd)
    rows = torch.tensor([0, 255, 256, 700, 1023])
    check_row_tolerance(full[rows.to(DEV)], oracle.gemm_root(bits(A[rows]), bits(Bm), 1))
    for _ in range(2):
        assert same_bits(B.gemm(c1, Ad, Bd), full)
    S = B.gemm_leaf_partial(c1, 0, 1, Ad, Bd)
    assert same_bits(B.tree_combine(c1, S[None]), full)
    assert B.last_device_status(c1) == B.ISO_OK


def test_cta_pair_repeatable_many_tiles(c8):
    """Many 256-row tiles per CTA pair (K = 4096, 512-k leaves): repeated launches give the
    same bits, and rows equal their one-CTA results (guards the pair's TMEM-buffer release
    protocol, where a race would show as tiles that differ between runs)."""
    M, K, N = 2048, 4096, 2048
    A, Bm = inputs.gemm_inputs(M, K, N, seed=41, device=DEV)
    base = B.gemm(c8, A, Bm)
    for _ in range(3):
        assert same_bits(B.gemm(c8, A, Bm), base)
    for r in (0, 255, 256, 1029, 2047):
        assert same_bits(B.gemm(c8, A[r:r + 1].contiguous(), Bm), base[r:r + 1]), r


def test_cta_pair_normal_inputs_and_partials(c8):
    """Normal inputs through CTA pairs: tolerance against the oracle on sampled rows, and
    the R-rank partial + combine path (also on pairs while K / (8 / R) >= 512) reproduces the
    single pass bit for bit."""
    M, K, N = 300, 8192, 256
    A, Bm = inputs.gemm_inputs(M, K, N, seed=4)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    full = B.gemm(c8, Ad, Bd)
    rows = torch.tensor([0, 127, 128, 255, 256, 299])
    check_row_tolerance(full[rows.to(DEV)], oracle.gemm_root(bits(A[rows]), bits(Bm), 8))
    for R in (2, 4):
        Kl = K // R
        S = torch.stack([B.gemm_leaf_partial(c8, r, R, Ad[:, r * Kl:(r + 1) * Kl].contiguous(),
                                             Bd[r * Kl:(r + 1) * Kl]) for r in range(R)])
        assert same_bits(B.tree_combine(c8, S), full), R


@pytest.mark.parametrize("M,N,K,L", [(1, 4096, 4096, 8), (7, 136, 2048, 4), (64, 4096, 4096, 8),
                                     (128, 12288, 4096, 8), (100, 1024, 8192, 8), (33, 512, 1024, 2)])
def test_gemm_ws_leaf_groups_match_single_pass_bitwise(M, N, K, L):
    """iso_gemm_ws spreads the leaves of one row block over more SMs (groups of L/R leaves,
    fp32 group roots, then the top tree levels); the bits must be iso_gemm's, for every
    split the heuristic picks (including none) and with a workspace too small to split."""
    c = B.Contract(L)
    A, Bm = inputs.gemm_inputs(M, K, N, seed=M + N)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    ref = B.gemm(c, Ad, Bd)
    assert same_bits(B.gemm_ws(c, Ad, Bd), ref), first_diff(B.gemm_ws(c, Ad, Bd), ref)
    small = torch.empty(M * N * 4, dtype=torch.uint8, device=DEV)  # room for one group: no split
    assert same_bits(B.gemm_ws(c, Ad, Bd, ws=small), ref)
    assert B.last_device_status(c) == B.ISO_OK


def test_gemm_ws_exact_integers_equal_oracle():
    M, N, K = 5, 1024, 4096
    c = B.Contract(8)
    A = inputs.small_int_bf16((M, K), -3, 3, seed=11)
    Bm = inputs.small_int_bf16((K, N), -3, 3, seed=12)
    C = B.gemm_ws(c, A.to(DEV), Bm.to(DEV))
    assert np.array_equal(bits(C), oracle.gemm(bits(A), bits(Bm), 8))


@pytest.mark.slow
def test_config2_full_size_m4096_sampled(c8):
    K, N, M = 4096, 4096, 4096
    A, Bm = inputs.gemm_inputs(M, K, N, seed=1, device=DEV)
    full = B.gemm(c8, A, Bm)
    rows = torch.tensor([0, 1000, 2047, 4095])
    ref = oracle.gemm_root(bits(A[rows.to(DEV)]), bits(Bm), 8)
    check_row_tolerance(full[rows.to(DEV)], ref)
    assert same_bits(B.gemm(c8, A[4000:4001].contiguous(), Bm), full[4000:4001])
    assert same_bits(B.gemm(c8, A[1:65].contiguous(), Bm), full[1:65])


# the three store paths of the bf16 epilogue: 8 warps on one CTA (leaves of 64 k), 4 warps on one
# CTA (16 rows, 256-k leaves, unstaged stores), and CTA pairs (300 rows, 512-k leaves, the second
# CTA of the last pair partly past M)
@pytest.mark.parametrize("M,K", [(70, 512), (16, 2048), (300, 4096)])
def test_canary_guard_bands(c8, M, K):
    """Output written exactly inside its [M x N] window of a wider ldc buffer."""
    N, ldc = 136, 264
    A, Bm = inputs.gemm_inputs(M, K, N, seed=4)
    buf = torch.full((M + 2, ldc), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[1:M + 1]
    Ad, Bd = A.to(DEV), Bm.to(DEV)  # keep the device copies alive until the kernel has run
    st = c8.lib.iso_gemm(c8.handle, B._ptr(Ad), K, B._ptr(Bd), N, B._vp(out.data_ptr()), ldc, M, N, K, B._stream())
    assert st == B.ISO_OK
    torch.cuda.synchronize()
    assert torch.all(buf[0] == 7.0) and torch.all(buf[M + 1] == 7.0) and torch.all(buf[1:M + 1, N:] == 7.0)
    ref = B.gemm(c8, Ad, Bd)
    assert same_bits(out[:, :N], ref)


def test_device_status_clean(c8):
    assert B.last_device_status(c8) == B.ISO_OK


@pytest.mark.parametrize("M,K,N,L", [(1, 4096, 4096, 8), (33, 1024, 392, 8), (128, 2048, 1024, 4), (64, 12288, 4096, 8),
                                     (2, 512, 520, 2)])
def test_cluster_leaf_groups_equal_single_pass(M, K, N, L):
    """One row block with few column tiles runs its leaf groups as thread-block clusters (each
    CTA one group, the top tree levels over distributed shared memory).  Its rows must equal the
    same rows computed inside a 300-row product (single pass, one CTA per tile and all leaves),
    and exact integers must equal the oracle."""
    c = B.Contract(L)
    A, Bm = inputs.gemm_inputs(300, K, N, seed=K + N + M)
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    big = B.gemm(c, Ad, Bd)
    for r0 in (0, 300 - M):
        assert same_bits(B.gemm(c, Ad[r0:r0 + M].contiguous(), Bd), big[r0:r0 + M]), r0
    Ai = inputs.small_int_bf16((M, K), -3, 3, seed=M + 7)
    Bi = inputs.small_int_bf16((K, N), -3, 3, seed=N + 7)
    assert np.array_equal(bits(B.gemm(c, Ai.to(DEV), Bi.to(DEV))), oracle.gemm(bits(Ai), bits(Bi), L))
    assert B.last_device_status(c) == B.ISO_OK
