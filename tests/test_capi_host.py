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
    for L in (1, 2, 4, 8, 16):
        c = B.Contract(L, lib)
        s = c.serialize()
        obj = json.loads(s)  # canonical form is valid JSON
        assert obj["gemm"]["leaves"] == L
        assert obj["claims"]["topology"]["simulated_ranks"] == [r for r in (1, 2, 4, 8, 16) if r <= L]
        assert c.digest == hashlib.sha256(s.encode()).digest()
        assert c.check_peer(c.digest) == B.ISO_OK
        digests[L] = c.digest
    assert len(set(digests.values())) == 5
    c8 = B.Contract(8, lib)
    assert c8.check_peer(digests[4]) == 6  # ISO_ERR_CONTRACT_MISMATCH
    assert B.Contract(8, lib).digest == digests[8]  # deterministic


def _leaves(obj, path=()):
    if isinstance(obj, dict):
        for k, v in obj.items():
            yield from _leaves(v, path + (k,))
    elif isinstance(obj, list) and obj and not all(isinstance(v, int) for v in obj):
        for i, v in enumerate(obj):
            yield from _leaves(v, path + (i,))
    else:
        yield path, obj


def _set(obj, path, value):
    for k in path[:-1]:
        obj = obj[k]
    obj[path[-1]] = value


def _header_constant(name):
    src = open(os.path.join(ROOT, "parallelism_invariant_logprob_gb300", "csrc", "iso_internal.h")).read()
    m = re.search(r"constexpr (?:int|float) " + name + r" = ([0-9.]+)f?;", src)
    assert m, name
    return float(m.group(1))


def test_contract_serialization_names_the_executed_numerics(lib):
    """Each kernel family has its block, the block's constants are the ones the kernels are
    compiled with, the stated arithmetic is the one in the kernel source (the fast SiLU
    intrinsics, attention's base-2 approximate exponent), and every value is covered by the
    digest (IsoExec blog, "Unified execution contract": equal identities mean equal numerics)."""
    c = B.Contract(8, lib)
    s = c.serialize()
    obj = json.loads(s)
    for block in ("impl", "gemm", "claims", "logprob", "rmsnorm", "moe", "attention", "math"):
        assert block in obj, block
    assert obj["gemm"]["leaf_chain"]["n"] == 128 and obj["gemm"]["leaf_chain"]["k"] == 16
    assert obj["logprob"]["tile_cols"] == 128
    assert obj["logprob"]["chunk_tiles"] == _header_constant("LP_CHUNK_TILES")
    assert obj["attention"]["chunk_keys"] == _header_constant("ATT_CHUNK_KEYS")
    assert obj["attention"]["lazy_log2"] == _header_constant("ATT_LAZY_LOG2")
    assert "fast_math" not in obj["math"]
    # the SiLU and the attention exponent as the kernel sources write them
    csrc = os.path.join(ROOT, "parallelism_invariant_logprob_gb300", "csrc")
    gemm_src = open(os.path.join(csrc, "gemm_tcgen05.cu")).read()
    assert "__fdividef(g, __fadd_rn(1.0f, __expf(-g)))" in gemm_src
    assert "h=bf16_rn(__fmul_rn(__fdividef(g,__fadd_rn(1,__expf(-g))),u))" in obj["moe"]["stages"]
    att_src = open(os.path.join(csrc, "attention_tcgen05.cu")).read()
    assert "ex2.approx.ftz.f32" in att_src and "__fmaf_rn(u2f(v[j]), c2, neg_m)" in att_src
    assert obj["attention"]["p"] == "ex2.approx.ftz(__fmaf_rn(S,c2,-m))"
    assert "__frcp_rn(l)" in att_src and "__frcp_rn(l)" in obj["attention"]["out"]
    # the serialization is canonical JSON, and changing any one value changes the digest
    assert json.dumps(obj, separators=(",", ":")) == s
    assert hashlib.sha256(s.encode()).digest() == c.digest
    n = 0
    for path, v in _leaves(obj):
        mutated = json.loads(s)
        _set(mutated, path, v + 1 if isinstance(v, (int, float)) and not isinstance(v, bool) else str(v) + "'")
        assert hashlib.sha256(json.dumps(mutated, separators=(",", ":")).encode()).digest() != c.digest, path
        n += 1
    assert n >= 50


def test_contract_init_rejects(lib):
    h = ctypes.c_void_p()
    assert lib.iso_contract_init(3, 0, B.ISO_F32, B.ISO_BF16, ctypes.byref(h), None) == 1
    assert lib.iso_contract_init(32, 0, B.ISO_F32, B.ISO_BF16, ctypes.byref(h), None) == 5
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


def test_static_scratch_limit_on_host(lib):
    """The allocation-free logprob entry point accepts exactly the problems whose minimum
    workspace fits its fixed 8 MiB array (16,512 tokens at V = 151936) and rejects the next
    size on the host, before any device call (so this runs without a GPU)."""
    c = B.Contract(8, lib)
    V, cap = 151936, 8 << 20
    mw = lambda T: int(lib.iso_selected_logprob_min_workspace(c.handle, T, V))
    assert mw(16512) <= cap < mw(16513)
    al = lambda x: (x + 255) // 256 * 256
    assert mw(16512) == al(16512 * 63 * 8) + al(16512 * 4)  # 63 chunks of (m, s) pairs + z_sel
    assert int(lib.iso_selected_logprob_workspace(c.handle, 820, V)) <= cap
    assert int(lib.iso_selected_logprob_workspace(c.handle, 840, V)) > cap
    st = lib.iso_selected_logprob_static_scratch(c.handle, None, None, None, None, 16513, 128, V, None)
    assert st == 7  # ISO_ERR_WORKSPACE
