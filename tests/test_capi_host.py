"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point ``include/iso.h`` declares, the contract digest is the
FIPS 180-4 SHA-256 of the canonical serialization, and invalid calls are
rejected on the host with the documented status before anything launches."""
import ctypes
import hashlib
import json
import os
import re

import pytest

from parallelism_invariant_logprob_gb300 import binding as B
from parallelism_invariant_logprob_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return B.load(build_if_missing=False)


def declared_functions():
    src = open(os.path.join(ROOT, "include", "iso.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(iso_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib.lib, n)]
    assert not missing, missing
    assert set(names) == set(B._SIGNATURES), set(names) ^ set(B._SIGNATURES)


@pytest.mark.parametrize("n", [0, 1, 55, 56, 63, 64, 65, 119, 120, 1000])
def test_sha256_matches_hashlib(lib, n):
    data = bytes((i * 37 + 11) & 0xFF for i in range(n))
    out = ctypes.create_string_buffer(32)
    assert lib.iso_sha256(data, n, out) == B.ISO_OK
    assert out.raw == hashlib.sha256(data).digest()


def test_contract_digest_is_sha256_of_serialization(lib):
    digests = {}
    for L in (1, 2, 4, 8):
        c = B.Contract(L, lib)
        s = c.serialize()
        obj = json.loads(s)  # canonical form is valid JSON
        assert obj["gemm"]["leaves"] == L
        assert obj["claims"]["topology"]["simulated_ranks"] == [r for r in (1, 2, 4, 8) if r <= L]
        assert c.digest == hashlib.sha256(s.encode()).digest()
        assert c.check_peer(c.digest) == B.ISO_OK
        digests[L] = c.digest
    assert len(set(digests.values())) == 4
    c8 = B.Contract(8, lib)
    assert c8.check_peer(digests[4]) == 6  # ISO_ERR_CONTRACT_MISMATCH
    assert B.Contract(8, lib).digest == digests[8]  # deterministic


def test_contract_init_rejects(lib):
    h = ctypes.c_void_p()
    assert lib.iso_contract_init(3, 0, B.ISO_F32, B.ISO_BF16, ctypes.byref(h), None) == 1
    assert lib.iso_contract_init(16, 0, B.ISO_F32, B.ISO_BF16, ctypes.byref(h), None) == 5
    assert lib.iso_contract_init(8, 0, B.ISO_BF16, B.ISO_BF16, ctypes.byref(h), None) == 5
    assert lib.iso_contract_init(8, 1, B.ISO_F32, B.ISO_BF16, ctypes.byref(h), None) == 5
    assert lib.iso_contract_init(8, 0, B.ISO_F32, B.ISO_BF16, None, None) == 1


def test_topology_claim(lib):
    c = B.Contract(8, lib)
    for R in (1, 2, 4, 8):
        assert c.check_topology(R) == B.ISO_OK
    for R in (0, 3, 6, 16, -2):
        assert c.check_topology(R) == 4


def test_host_validation_launches_nothing(lib):
    c = B.Contract(8, lib)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every case below fails validation first
    s0 = ctypes.c_void_p(0)
    # K not a multiple of 16 L
    assert lib.iso_gemm(c.handle, fake, 1000, fake, 512, fake, 512, 4, 512, 1000, s0) == 2
    # N not a multiple of 8
    assert lib.iso_gemm(c.handle, fake, 1024, fake, 516, fake, 516, 4, 514, 1024, s0) == 2
    # misaligned pointer
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert lib.iso_gemm(c.handle, odd, 1024, fake, 512, fake, 512, 4, 512, 1024, s0) == 3
    # null contract / negative M
    assert lib.iso_gemm(None, fake, 1024, fake, 512, fake, 512, 4, 512, 1024, s0) == 1
    assert lib.iso_gemm(c.handle, fake, 1024, fake, 512, fake, 512, -1, 512, 1024, s0) == 1
    # M == 0 is a no-op
    assert lib.iso_gemm(c.handle, fake, 1024, fake, 512, fake, 512, 0, 512, 1024, s0) == B.ISO_OK
    # unproven topologies
    assert lib.iso_gemm_leaf_partial(c.handle, 0, 3, fake, 1024, fake, 512, fake, 512, 4, 512, 1024, s0) == 4
    assert lib.iso_gemm_leaf_partial(c.handle, 0, 16, fake, 1024, fake, 512, fake, 512, 4, 512, 1024, s0) == 4
    assert lib.iso_gemm_leaf_partial(c.handle, 2, 2, fake, 1024, fake, 512, fake, 512, 4, 512, 1024, s0) == 1
    assert lib.iso_tree_combine(c.handle, 3, fake, 512, 4 * 512, fake, 512, 4, 512, s0) == 4
    # logprob: workspace too small, V not a multiple of 8, H not a multiple of 16 L
    need = lib.iso_selected_logprob_min_workspace(c.handle, 4, 2440)
    assert 0 < need < lib.iso_selected_logprob_workspace(c.handle, 4, 2440)
    assert lib.iso_selected_logprob(c.handle, fake, fake, fake, fake, 4, 512, 2440, fake, need - 1, s0) == 7
    assert lib.iso_selected_logprob_min_workspace(None, 4, 2440) == 0
    assert lib.iso_selected_logprob(c.handle, fake, fake, fake, fake, 4, 512, 2441, fake, need, s0) == 2
    assert lib.iso_selected_logprob(c.handle, fake, fake, fake, fake, 4, 520, 2440, fake, need, s0) == 2
    # rmsnorm: H not a multiple of 8
    assert lib.iso_rmsnorm(c.handle, fake, fake, ctypes.c_float(1e-6), fake, 4, 100, s0) == 2
    # moe: k not a power of two for the combine; E too large for routing
    assert lib.iso_moe_combine(c.handle, fake, fake, fake, 4, 3, 256, s0) == 5
    assert lib.iso_moe_route(c.handle, fake, 4, 512, 8, fake, fake, s0) == 5
    # expert layer: the one-rank partial needs the layer's workspace minus the slot rows
    # (T k H bf16, here 16*8*256*2 bytes, 256-byte aligned); shape, alignment, workspace and
    # missing-mask errors come from the host checks
    full = lib.iso_grouped_gemm_moe_workspace(c.handle, 16, 8, 8, 256, 128)
    part = lib.iso_moe_experts_partial_workspace(c.handle, 16, 8, 8, 256, 128)
    assert full - part == 16 * 8 * 256 * 2
    assert lib.iso_moe_experts_partial(c.handle, fake, fake, fake, fake, None, fake, 16, 8, 8, 256, 128, fake, part,
                                       s0) == 1
    mask = (ctypes.c_uint8 * 8)(*([1] * 8))
    mk = ctypes.cast(mask, ctypes.c_void_p)
    assert lib.iso_moe_experts_partial(c.handle, fake, fake, fake, fake, mk, fake, 16, 8, 8, 264, 128, fake, part,
                                       s0) == 2
    assert lib.iso_moe_experts_partial(c.handle, fake, fake, fake, fake, mk, odd, 16, 8, 8, 256, 128, fake, part,
                                       s0) == 3
    assert lib.iso_moe_experts_partial(c.handle, fake, fake, fake, fake, mk, fake, 16, 8, 8, 256, 128, fake,
                                       part - 1, s0) == 7
    assert lib.iso_moe_experts_partial(c.handle, fake, fake, fake, fake, mk, fake, 0, 8, 8, 256, 128, fake, part,
                                       s0) == B.ISO_OK
    # bounded-wait self test: limit out of range
    assert lib.iso_selftest_bounded_wait(0, s0) == 1


def test_status_strings(lib):
    for s in range(12):
        assert lib.iso_status_string(s)
