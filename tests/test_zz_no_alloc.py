"""The allocation-free logprob entry point, for callers that cannot allocate
device memory (plugin/callback interfaces that get only input and output
pointers; frameworks that own all device memory).  It must return what the
workspace-taking entry point returns -- within the logprob tolerance of the
other tests, and in fact bit for bit, since the same kernels run -- on two
calls in a row that share its static scratch, and must reject a problem
whose scratch need exceeds the fixed array.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu
SCRATCH_BYTES = 8 << 20


def _static_call(c, h, W, ids):
    T, H = h.shape
    V = W.shape[1]
    out = torch.full((T,), float("nan"), dtype=torch.float32, device=h.device)
    st = c.lib.iso_selected_logprob_static_scratch(c.handle, B._ptr(h), B._ptr(W), B._ptr(ids), B._ptr(out), T, H, V,
                                                   B._stream())
    return st, out


def test_static_scratch_matches_workspace_entry_point_twice():
    c = B.Contract(8)
    cases = [(300, 512, 2440, 21), (1000, 1024, 151936, 22)]  # second call reuses scratch left by the first
    for T, H, V, seed in cases:
        h, W, ids = inputs.logprob_inputs(T, H, V, seed=seed, device="cuda")
        ref = B.selected_logprob(c, h, W, ids)
        st, out = _static_call(c, h, W, ids)
        assert st == B.ISO_OK
        torch.cuda.synchronize()
        diff = (out.double() - ref.double()).abs().max().item()
        assert diff <= 1e-3
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    assert B.last_device_status(c) == B.ISO_OK


def test_static_scratch_rejects_oversize():
    c = B.Contract(8)
    V = 151936
    T = 16513  # one token past what the fixed scratch holds at this vocabulary
    assert c.lib.iso_selected_logprob_min_workspace(c.handle, T - 1, V) <= SCRATCH_BYTES
    assert c.lib.iso_selected_logprob_min_workspace(c.handle, T, V) > SCRATCH_BYTES
    h = torch.zeros(T, 128, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, V, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(T, dtype=torch.int32, device="cuda")
    st, out = _static_call(c, h, W, ids)
    assert st == 7  # ISO_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out).all()  # nothing was launched
