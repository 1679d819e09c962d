"""Host threads calling the library at once, from a cold start: each thread runs its own
entry points on its own stream, and every result has the bits of the same call made alone.
The calls run in a fresh process, so the threads race on the per-device first-call setup
(kernel attributes, resident-CTA counts, the status word's address)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading, torch
sys.path.insert(0, sys.argv[1])
from parallelism_invariant_logprob_gb300 import binding as B, inputs
dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
c = B.Contract(8)
A, W = inputs.gemm_inputs(300, 4096, 1024, seed=1, device=dev)          # CTA pairs
a1 = A[:1].contiguous()                                                # cluster leaf groups
x, g = inputs.rmsnorm_inputs(64, 1024, seed=2, device=dev)
h, Wl, ids = inputs.logprob_inputs(40, 512, 2440, seed=3, device=dev)
Q, K, V, qs, ks, p0 = inputs.attention_inputs([130, 9], [0, 20], 4, 2, 128, seed=4, device=dev)
torch.cuda.synchronize()  # the inputs exist before any worker stream reads them
def run(kind, stream):
    with torch.cuda.stream(stream):
        if kind == 0:
            return B.gemm(c, A, W, stream=stream)
        if kind == 1:
            return B.gemm(c, a1, W, stream=stream)
        if kind == 2:
            return B.rmsnorm(c, x, g, 1e-6, stream=stream)
        if kind == 3:
            return B.selected_logprob(c, h, Wl, ids, stream=stream)
        return B.attention(c, Q, K, V, qs, ks, p0, 128 ** -0.5, stream=stream)[0]
results = {}
errors = []
def worker(t):
    try:
        s = torch.cuda.Stream(device=dev)
        outs = [run((t + i) % 5, s) for i in range(10)]
        s.synchronize()
        results[t] = outs
    except Exception as e:  # reported by the parent
        errors.append(repr(e))
threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
for th in threads:
    th.start()
for th in threads:
    th.join()
assert not errors, errors
torch.cuda.synchronize()
alone = [run(k, torch.cuda.current_stream()) for k in range(5)]
torch.cuda.synchronize()
for t, outs in results.items():
    for i, o in enumerate(outs):
        ref = alone[(t + i) % 5]
        assert torch.equal(o.view(torch.uint8), ref.view(torch.uint8)), (t, i)
assert B.last_device_status(c) == B.ISO_OK
print("threads ok")
"""


def test_concurrent_host_threads_cold_start():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
