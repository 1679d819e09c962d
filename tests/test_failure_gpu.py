"""Device-side failure detection without a GPU fault: a bounded mbarrier wait
that nothing completes must give up after its limit, report
ISO_ERR_DEVICE_TIMEOUT through the status word, and leave the context usable."""
import time

import pytest
import torch

from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    c = B.Contract(8)
    assert B.last_device_status(c) == B.ISO_OK
    t0 = time.time()
    assert c.lib.iso_selftest_bounded_wait(50_000_000, B._stream()) == B.ISO_OK  # 50 ms
    assert B.last_device_status(c) == 9  # ISO_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 10
    assert B.last_device_status(c) == B.ISO_OK
    A, Bm = inputs.gemm_inputs(16, 256, 128, seed=0)
    C = B.gemm(c, A.cuda(), Bm.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(C.float()).all()
