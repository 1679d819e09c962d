"""GPU parity of iso_mismatch_diagnostics against the float64 oracle (VeXact paper,
Eq. 1, 6, 7; K1 / K3 of §4.1), and the zero-mismatch property of this library's own
logprobs: prefill (packed) and decode (one row per call) give identical values."""
import numpy as np
import pytest
import torch

import oracle
from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _packed(seed):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, 3000, (40,), generator=g).tolist() + [0, 1, 4]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = int(offs[-1])
    ro = -torch.abs(torch.randn(n, generator=g)) * 2
    noise = torch.randn(n, generator=g) * 1e-3
    keep = torch.rand(n, generator=g) < 0.5  # half the tokens agree bit for bit
    tr = torch.where(keep, ro, ro + noise)
    big = torch.rand(n, generator=g) < 0.001
    tr = torch.where(big, tr - 0.8, tr)  # rare large drifts (an argmax flip's size)
    return tr.float(), ro.float(), offs


@pytest.fixture(scope="module")
def c8():
    return B.Contract(8)


def test_diagnostics_vs_oracle(c8):
    tr, ro, offs = _packed(11)
    r = B.mismatch_diagnostics(c8, tr.to(DEV), ro.to(DEV), torch.from_numpy(offs).to(DEV))
    ref = oracle.mismatch(tr.numpy(), ro.numpy(), offs)
    assert np.array_equal(r["delta"].cpu().numpy(), ref["delta"].astype(np.float32))
    w = r["tis_weight"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(w - ref["tis_weight"]) <= np.spacing(np.float32(ref["tis_weight"])) * 1.01)
    assert np.all(w <= 2.0)
    for key in ("seq_k1", "seq_k3", "seq_sum_abs_delta"):
        got = r[key].cpu().numpy()
        want = ref[key] if key != "seq_sum_abs_delta" else np.array(
            [np.abs(ref["delta"][offs[b]:offs[b + 1]]).sum() for b in range(len(offs) - 1)])
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), key
    # the rejection decision is taken in double on both sides; no test sequence sits near tau_seq
    for key, s in (("accept_k1", ref["seq_k1"]), ("accept_k3", ref["seq_k3"])):
        assert np.all(np.abs(s - 0.001) > 1e-9)
        assert np.array_equal(r[key].cpu().numpy(), ref[key]), key
    assert 0 < ref["accept_k3"].sum() < len(ref["accept_k3"])  # both decisions occur
    assert np.array_equal(r["seq_max_abs_delta"].cpu().numpy(), ref["seq_max_abs_delta"].astype(np.float32))
    assert np.array_equal(r["seq_mismatches"].cpu().numpy(), ref["seq_mismatches"])


def test_diagnostics_invariant_to_batch_composition(c8):
    tr, ro, offs = _packed(12)
    full = B.mismatch_diagnostics(c8, tr.to(DEV), ro.to(DEV), torch.from_numpy(offs).to(DEV))
    for b in (0, 7, len(offs) - 2):
        sub = torch.tensor([0, offs[b + 1] - offs[b]], dtype=torch.int32, device=DEV)
        one = B.mismatch_diagnostics(c8, tr[offs[b]:offs[b + 1]].contiguous().to(DEV),
                                     ro[offs[b]:offs[b + 1]].contiguous().to(DEV), sub)
        for key in ("seq_k1", "seq_k3", "seq_sum_abs_delta", "seq_max_abs_delta", "seq_mismatches", "accept_k3"):
            assert torch.equal(one[key][0], full[key][b]), (b, key)


def test_prefill_and_decode_logprobs_show_zero_mismatch(c8):
    """Score 3 sequences once packed (prefill) and token by token (decode, one row per call):
    the library's logprobs agree bit for bit, so every diagnostic reports no mismatch."""
    T, H, V = 96, 512, 2440
    h, W, ids = inputs.logprob_inputs(T, H, V, seed=31, device=DEV)
    prefill = B.selected_logprob(c8, h, W, ids)
    decode = torch.cat([B.selected_logprob(c8, h[t:t + 1].contiguous(), W, ids[t:t + 1].contiguous())
                        for t in range(T)])
    offs = torch.tensor([0, 40, 41, 96], dtype=torch.int32, device=DEV)
    r = B.mismatch_diagnostics(c8, prefill, decode, offs)
    assert torch.all(r["delta"] == 0) and torch.all(r["seq_mismatches"] == 0)
    assert torch.all(r["seq_k1"] == 0) and torch.all(r["seq_k3"] == 0) and torch.all(r["accept_k1"] == 1)
    assert torch.all(r["tis_weight"] == 1.0)


def test_diagnostics_argument_checks(c8):
    x = torch.zeros(4, device=DEV)
    offs = torch.tensor([0, 4], dtype=torch.int32, device=DEV)
    with pytest.raises(B.IsoError):
        B.mismatch_diagnostics(c8, x, x, offs, tau_tok=0.0)
    with pytest.raises(B.IsoError):
        B.mismatch_diagnostics(c8, x, x, offs, tau_seq=-1.0)
