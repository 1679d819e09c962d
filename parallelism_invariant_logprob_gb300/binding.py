"""Thin ctypes binding over ``libiso.so`` (declared in ``include/iso.h``).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors are PyTorch CUDA tensors (PyTorch is used for
device memory and streams); bf16 tensors are passed as raw pointers.  There
is no fallback of any kind: if the library is missing or a call fails, an
exception is raised.

The function names are those of the C ABI.  The tensor-level helpers at the
end (``gemm``, ``selected_logprob`` ...) allocate outputs and workspaces with
torch and then call the same entry points.
"""
from __future__ import annotations

import ctypes
import os

from .build_lib import library_path

ISO_OK = 0
STATUS_NAMES = {
    0: "ISO_OK", 1: "ISO_ERR_INVALID_ARG", 2: "ISO_ERR_SHAPE", 3: "ISO_ERR_ALIGNMENT",
    4: "ISO_ERR_UNPROVEN_TOPOLOGY", 5: "ISO_ERR_UNSUPPORTED", 6: "ISO_ERR_CONTRACT_MISMATCH",
    7: "ISO_ERR_WORKSPACE", 8: "ISO_ERR_CUDA", 9: "ISO_ERR_DEVICE_TIMEOUT", 10: "ISO_ERR_NOT_IMPLEMENTED",
    11: "ISO_ERR_BAD_TOKEN_ID", 12: "ISO_ERR_DEVICE_CHECK",
}
for _code, _name in STATUS_NAMES.items():
    globals()[_name] = _code
ISO_TREE_BALANCED_BINARY = 0
ISO_F32, ISO_BF16 = 0, 1


class IsoError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_sz = ctypes.c_size_t
_u64 = ctypes.c_uint64

_SIGNATURES = {
    "iso_contract_init": (_int, [_int, _int, _int, _int, ctypes.POINTER(_vp), ctypes.c_char_p]),
    "iso_contract_destroy": (None, [_vp]),
    "iso_contract_serialize": (_int, [_vp, ctypes.c_char_p, _sz, ctypes.POINTER(_sz)]),
    "iso_contract_digest": (_int, [_vp, ctypes.c_char_p]),
    "iso_contract_check_peer": (_int, [_vp, ctypes.c_char_p]),
    "iso_contract_check_topology": (_int, [_vp, _int]),
    "iso_contract_leaf_count": (_int, [_vp]),
    "iso_sha256": (_int, [ctypes.c_char_p, _sz, ctypes.c_char_p]),
    "iso_status_string": (ctypes.c_char_p, [_int]),
    "iso_last_device_status": (_int, [_vp]),
    "iso_gemm": (_int, [_vp, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int, _int, _vp]),
    "iso_gemm_leaf_partial": (_int, [_vp, _int, _int, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int, _int, _vp]),
    "iso_tree_combine": (_int, [_vp, _int, _vp, _i64, _i64, _vp, _i64, _int, _int, _vp]),
    "iso_rmsnorm": (_int, [_vp, _vp, _vp, ctypes.c_float, _vp, _int, _int, _vp]),
    "iso_selected_logprob_workspace": (_sz, [_vp, _int, _int]),
    "iso_selected_logprob": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _vp, _sz, _vp]),
    "iso_moe_route": (_int, [_vp, _vp, _int, _int, _int, _vp, _vp, _vp]),
    "iso_moe_permute_workspace": (_sz, [_int, _int, _int]),
    "iso_gemm_workspace": (_sz, [_vp, _int, _int, _int]),
    "iso_mismatch_diagnostics": (_int, [_vp, _vp, _vp, _vp, _int, _int, ctypes.c_double, ctypes.c_double, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "iso_selected_logprob_partial_workspace": (_sz, [_vp, _int, _int]),
    "iso_selected_logprob_partial": (_int, [_vp, _vp, _vp, _i64, _vp, _int, _int, _int, _int, _int, _vp, _vp, _vp,
                                            _sz, _vp]),
    "iso_selected_logprob_combine": (_int, [_vp, _int, _vp, _vp, _vp, _vp, _vp, _int, _int, _vp]),
    "iso_gemm_ws": (_int, [_vp, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int, _int, _vp, _sz, _vp]),
    "iso_selected_logprob_min_workspace": (_sz, [_vp, _int, _int]),
    "iso_moe_permute": (_int, [_vp, _vp, _int, _int, _int, _vp, _int, _vp, _vp, _vp, _vp]),
    "iso_moe_combine": (_int, [_vp, _vp, _vp, _vp, _int, _int, _int, _vp]),
    "iso_grouped_gemm_moe_workspace": (_sz, [_vp, _int, _int, _int, _int, _int]),
    "iso_grouped_gemm_moe": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _vp, _int, _int, _int, _int, _int,
                                    _vp, _sz, _vp]),
    "iso_moe_experts_partial_workspace": (_sz, [_vp, _int, _int, _int, _int, _int]),
    "iso_moe_experts_partial": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _vp, _sz,
                                       _vp]),
    "iso_selftest_bounded_wait": (_int, [_u64, _vp]),
    "iso_selected_logprob_static_scratch": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _vp]),
    "iso_rmsnorm_gemm_workspace": (_sz, [_vp, _int]),
    "iso_rmsnorm_gemm": (_int, [_vp, _vp, _vp, ctypes.c_float, _vp, _i64, _vp, _i64, _int, _int, _int, _vp, _sz, _vp]),
    "iso_rmsnorm_selected_logprob_workspace": (_sz, [_vp, _int, _int]),
    "iso_rmsnorm_selected_logprob": (_int, [_vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _int, _int, _int, _vp, _sz,
                                            _vp]),
    "iso_attention": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _int,
                             ctypes.c_float, _vp, _vp, _vp]),
}


class Library:
    """The loaded ``libiso.so`` with typed entry points."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(self.lib, name)
            f.restype = res
            f.argtypes = args
            setattr(self, name, f)

    def check(self, status: int, what: str):
        if status != ISO_OK:
            raise IsoError(status, what)


_LIB = {}


def load(build_if_missing: bool = True, debug: bool = False) -> Library:
    """Load the CUDA library (``debug``: the bounds-checked build ``libiso_debug.so``); builds it
    in-tree if absent.  Raises if neither works."""
    if debug in _LIB:
        return _LIB[debug]
    path = library_path(debug)
    if not os.path.exists(path):
        if not build_if_missing:
            raise FileNotFoundError(f"CUDA library not built: {path}")
        from .build_lib import build
        build(debug=debug)
    _LIB[debug] = Library(path)
    return _LIB[debug]


# ------------------------------------------------------------------ contract
class Contract:
    """Host-side numerical contract (owns an ``iso_contract*``)."""

    def __init__(self, leaf_count: int = 8, lib: Library | None = None):
        self.lib = lib or load()
        h = _vp()
        dig = ctypes.create_string_buffer(32)
        st = self.lib.iso_contract_init(leaf_count, ISO_TREE_BALANCED_BINARY, ISO_F32, ISO_BF16, ctypes.byref(h), dig)
        self.lib.check(st, "iso_contract_init")
        self.handle = h
        self.digest = dig.raw
        self.leaf_count = leaf_count

    def serialize(self) -> str:
        n = _sz()
        self.lib.check(self.lib.iso_contract_serialize(self.handle, None, 0, ctypes.byref(n)), "serialize")
        buf = ctypes.create_string_buffer(n.value + 1)
        self.lib.check(self.lib.iso_contract_serialize(self.handle, buf, n.value + 1, ctypes.byref(n)), "serialize")
        return buf.value.decode()

    def check_peer(self, digest: bytes) -> int:
        return self.lib.iso_contract_check_peer(self.handle, digest)

    def check_topology(self, R: int) -> int:
        return self.lib.iso_contract_check_topology(self.handle, R)

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                self.lib.iso_contract_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


# ------------------------------------------------------- tensor-level helpers
def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return _vp(s.cuda_stream)


def gemm_workspace(c: Contract, M: int, N: int, K: int) -> int:
    return int(c.lib.iso_gemm_workspace(c.handle, M, N, K))


def gemm_ws(c: Contract, A, B, out=None, ws=None, stream=None):
    """iso_gemm_ws: iso_gemm's bits, with leaf groups spread over more SMs for small M."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    if ws is None:
        ws = torch.empty(max(gemm_workspace(c, M, N, K), 16), dtype=torch.uint8, device=A.device)
    st = c.lib.iso_gemm_ws(c.handle, _ptr(A), A.stride(0), _ptr(B), B.stride(0), _ptr(out), out.stride(0), M, N, K,
                           _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    c.lib.check(st, "iso_gemm_ws")
    return out


def gemm(c: Contract, A, B, out=None, stream=None):
    import torch
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    st = c.lib.iso_gemm(c.handle, _ptr(A), A.stride(0), _ptr(B), B.stride(0), _ptr(out), out.stride(0), M, N, K,
                        _stream(stream))
    c.lib.check(st, "iso_gemm")
    return out


def gemm_leaf_partial(c: Contract, rank: int, R: int, A_r, B_r, out=None, stream=None):
    import torch
    M, Kl = A_r.shape
    N = B_r.shape[1]
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=A_r.device)
    st = c.lib.iso_gemm_leaf_partial(c.handle, rank, R, _ptr(A_r), A_r.stride(0), _ptr(B_r), B_r.stride(0),
                                     _ptr(out), out.stride(0), M, N, Kl, _stream(stream))
    c.lib.check(st, "iso_gemm_leaf_partial")
    return out


def tree_combine(c: Contract, S, out=None, stream=None):
    """S: fp32 [R, M, N] (contiguous per rank)."""
    import torch
    R, M, N = S.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=S.device)
    st = c.lib.iso_tree_combine(c.handle, R, _ptr(S), S.stride(1), S.stride(0), _ptr(out), out.stride(0), M, N,
                                _stream(stream))
    c.lib.check(st, "iso_tree_combine")
    return out


def rmsnorm(c: Contract, x, gamma, eps: float, out=None, stream=None):
    import torch
    T, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    st = c.lib.iso_rmsnorm(c.handle, _ptr(x), _ptr(gamma), float(eps), _ptr(out), T, H, _stream(stream))
    c.lib.check(st, "iso_rmsnorm")
    return out


def selected_logprob_workspace(c: Contract, T: int, V: int) -> int:
    return int(c.lib.iso_selected_logprob_workspace(c.handle, T, V))


LP_CHUNK_COLS = 128 * 19  # vocabulary columns per statistics chunk


def selected_logprob_partial(c: Contract, h, W_r, ids, V: int, v0: int, stats_r=None, zsel_r=None, ws=None,
                             stream=None):
    """One vocab shard's chunk statistics [C_r x T x 2] and its selected logits [T]."""
    import torch
    T, H = h.shape
    V_r = W_r.shape[1]
    C_r = ((V_r + 127) // 128 + 18) // 19
    if stats_r is None:
        stats_r = torch.empty(C_r, T, 2, dtype=torch.float32, device=h.device)
    if zsel_r is None:
        zsel_r = torch.zeros(T, dtype=torch.float32, device=h.device)
    if ws is None:
        ws = torch.empty(max(int(c.lib.iso_selected_logprob_partial_workspace(c.handle, T, V_r)), 16),
                         dtype=torch.uint8, device=h.device)
    st = c.lib.iso_selected_logprob_partial(c.handle, _ptr(h), _ptr(W_r), W_r.stride(0), _ptr(ids), T, H, V, v0, V_r,
                                            _ptr(stats_r), _ptr(zsel_r), _ptr(ws), ws.numel() * ws.element_size(),
                                            _stream(stream))
    c.lib.check(st, "iso_selected_logprob_partial")
    return stats_r, zsel_r


def selected_logprob_combine(c: Contract, shard_v0, stats, zsel, ids, V: int, out=None, stream=None):
    """Chunk tree over the gathered shard statistics [C x T x 2]; zsel [num_shards x T]."""
    import torch
    T = ids.shape[0]
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=ids.device)
    v0 = (ctypes.c_int * len(shard_v0))(*shard_v0)
    st = c.lib.iso_selected_logprob_combine(c.handle, len(shard_v0), v0, _ptr(stats), _ptr(zsel), _ptr(ids), _ptr(out),
                                            T, V, _stream(stream))
    c.lib.check(st, "iso_selected_logprob_combine")
    return out


def mismatch_diagnostics(c: Contract, logp_train, logp_rollout, offsets, tau_tok=2.0, tau_seq=0.001, stream=None,
                         out=None):
    """Per token delta and min(r_corr, tau_tok); per sequence sums of K1 / K3, rejection masks,
    max and sum of |delta| and the count of differing tokens (all device tensors).  `out`: a
    dict returned by an earlier call of the same sizes, reused as the output buffers."""
    import torch
    N = logp_train.numel()
    B = offsets.numel() - 1
    dev = logp_train.device
    r = out if out is not None else dict(delta=torch.empty(N, dtype=torch.float32, device=dev),
             tis_weight=torch.empty(N, dtype=torch.float32, device=dev),
             seq_k1=torch.empty(B, dtype=torch.float64, device=dev), seq_k3=torch.empty(B, dtype=torch.float64, device=dev),
             accept_k1=torch.empty(B, dtype=torch.uint8, device=dev), accept_k3=torch.empty(B, dtype=torch.uint8, device=dev),
             seq_max_abs_delta=torch.empty(B, dtype=torch.float32, device=dev),
             seq_sum_abs_delta=torch.empty(B, dtype=torch.float64, device=dev),
             seq_mismatches=torch.empty(B, dtype=torch.int32, device=dev))
    st = c.lib.iso_mismatch_diagnostics(c.handle, _ptr(logp_train), _ptr(logp_rollout), _ptr(offsets), B, N, tau_tok,
                                        tau_seq, _ptr(r["delta"]), _ptr(r["tis_weight"]), _ptr(r["seq_k1"]),
                                        _ptr(r["seq_k3"]), _ptr(r["accept_k1"]), _ptr(r["accept_k3"]),
                                        _ptr(r["seq_max_abs_delta"]), _ptr(r["seq_sum_abs_delta"]),
                                        _ptr(r["seq_mismatches"]), _stream(stream))
    c.lib.check(st, "iso_mismatch_diagnostics")
    return r


def attention(c: Contract, Q, K, V, q_start, k_start, pos0, scale: float, max_q_rows: int | None = None,
              out=None, lse=None, want_lse: bool = True, stream=None):
    """Causal attention over packed sequences.  Q [Tq, Hq, d], K and V [Tk, Hkv, d] bf16;
    q_start, k_start [B+1] and pos0 [B] int32 device tensors.  Returns (out, lse); lse is
    None when want_lse is False.  max_q_rows defaults to the largest q_start difference
    (read back from the device)."""
    import torch
    Tq, Hq, d = Q.shape
    Tk, Hkv = K.shape[0], K.shape[1]
    B = q_start.numel() - 1
    if max_q_rows is None:
        max_q_rows = int((q_start[1:] - q_start[:-1]).max().item()) if B > 0 else 0
    if out is None:
        out = torch.empty(Tq, Hq, d, dtype=torch.bfloat16, device=Q.device)
    if lse is None and want_lse:
        lse = torch.empty(Tq, Hq, dtype=torch.float32, device=Q.device)
    st = c.lib.iso_attention(c.handle, _ptr(Q), _ptr(K), _ptr(V), _ptr(q_start), _ptr(k_start), _ptr(pos0), B, Tq,
                             Tk, Hq, Hkv, d, max_q_rows, float(scale), _ptr(out), _ptr(lse) if lse is not None else None,
                             _stream(stream))
    c.lib.check(st, "iso_attention")
    return out, lse


def rmsnorm_gemm_workspace(c: Contract, M: int) -> int:
    return int(c.lib.iso_rmsnorm_gemm_workspace(c.handle, M))


def rmsnorm_selected_logprob_workspace(c: Contract, T: int, V: int) -> int:
    return int(c.lib.iso_rmsnorm_selected_logprob_workspace(c.handle, T, V))


def rmsnorm_gemm(c: Contract, x, gamma, eps: float, B, out=None, ws=None, stream=None):
    """iso_gemm(iso_rmsnorm(x, gamma, eps), B) with the normalisation fused into the A prologue."""
    import torch
    M, K = x.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = torch.empty(max(int(c.lib.iso_rmsnorm_gemm_workspace(c.handle, M)), 16), dtype=torch.uint8,
                         device=x.device)
    st = c.lib.iso_rmsnorm_gemm(c.handle, _ptr(x), _ptr(gamma), float(eps), _ptr(B), B.stride(0), _ptr(out),
                                out.stride(0), M, N, K, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    c.lib.check(st, "iso_rmsnorm_gemm")
    return out


def rmsnorm_selected_logprob(c: Contract, x, gamma, eps: float, W, ids, out=None, ws=None, stream=None):
    """iso_selected_logprob(iso_rmsnorm(x, gamma, eps), W, ids) with the normalisation fused."""
    import torch
    T, H = x.shape
    V = W.shape[1]
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=x.device)
    if ws is None:
        ws = torch.empty(max(int(c.lib.iso_rmsnorm_selected_logprob_workspace(c.handle, T, V)), 16),
                         dtype=torch.uint8, device=x.device)
    st = c.lib.iso_rmsnorm_selected_logprob(c.handle, _ptr(x), _ptr(gamma), float(eps), _ptr(W), _ptr(ids), _ptr(out),
                                            T, H, V, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    c.lib.check(st, "iso_rmsnorm_selected_logprob")
    return out


def selected_logprob_min_workspace(c: Contract, T: int, V: int) -> int:
    return int(c.lib.iso_selected_logprob_min_workspace(c.handle, T, V))


def selected_logprob(c: Contract, h, W, ids, out=None, ws=None, stream=None):
    import torch
    T, H = h.shape
    V = W.shape[1]
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=h.device)
    need = selected_logprob_workspace(c, T, V)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=h.device)
    st = c.lib.iso_selected_logprob(c.handle, _ptr(h), _ptr(W), _ptr(ids), _ptr(out), T, H, V, _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream))
    c.lib.check(st, "iso_selected_logprob")
    return out


def moe_route(c: Contract, logits, k: int, stream=None):
    import torch
    T, E = logits.shape
    ids = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    st = c.lib.iso_moe_route(c.handle, _ptr(logits), T, E, k, _ptr(ids), _ptr(w), _stream(stream))
    c.lib.check(st, "iso_moe_route")
    return ids, w


def moe_permute(c: Contract, ids, E: int, expert_partition=None, partition: int = 0, stream=None):
    import torch
    T, k = ids.shape
    perm = torch.empty(T * k, dtype=torch.int32, device=ids.device)
    offs = torch.empty(E + 1, dtype=torch.int32, device=ids.device)
    cnt = torch.empty(int(c.lib.iso_moe_permute_workspace(T, E, k)) // 4, dtype=torch.int32, device=ids.device)
    st = c.lib.iso_moe_permute(c.handle, _ptr(ids), T, E, k, _ptr(expert_partition), partition, _ptr(perm),
                               _ptr(offs), _ptr(cnt), _stream(stream))
    c.lib.check(st, "iso_moe_permute")
    return perm, offs


def moe_combine(c: Contract, y_slots, w, out=None, stream=None):
    import torch
    T, k, H = y_slots.shape
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y_slots.device)
    st = c.lib.iso_moe_combine(c.handle, _ptr(y_slots), _ptr(w), _ptr(out), T, k, H, _stream(stream))
    c.lib.check(st, "iso_moe_combine")
    return out


def grouped_gemm_moe_workspace(c: Contract, T, E, k, H, F) -> int:
    return int(c.lib.iso_grouped_gemm_moe_workspace(c.handle, T, E, k, H, F))


def grouped_gemm_moe(c: Contract, x, ids, w, W1, W2, expert_partition=None, out=None, ws=None, stream=None):
    """expert_partition: None or a host sequence of E partition ids."""
    import torch
    T, H = x.shape
    E, _, F2 = W1.shape
    F = F2 // 2
    k = ids.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    need = grouped_gemm_moe_workspace(c, T, E, k, H, F)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    part_arr, nparts = None, 0
    if expert_partition is not None:
        vals = [int(v) for v in expert_partition]
        part_arr = (ctypes.c_int32 * E)(*vals)
        nparts = max(vals) + 1
    st = c.lib.iso_grouped_gemm_moe(c.handle, _ptr(x), _ptr(ids), _ptr(w), _ptr(W1), _ptr(W2),
                                    ctypes.cast(part_arr, _vp) if part_arr is not None else None, nparts, _ptr(out),
                                    T, E, k, H, F, _ptr(ws), ws.numel(), _stream(stream))
    c.lib.check(st, "iso_grouped_gemm_moe")
    return out


def moe_experts_partial_workspace(c: Contract, T, E, k, H, F) -> int:
    return int(c.lib.iso_moe_experts_partial_workspace(c.handle, T, E, k, H, F))


def moe_experts_partial(c: Contract, x, ids, W1, W2, expert_mask, y_slots=None, ws=None, stream=None):
    """The slot rows [T*k, H] of the experts with expert_mask[e] set (a host sequence of E
    flags); other rows of y_slots are left as they were (uninitialised when y_slots is None)."""
    import torch
    T, H = x.shape
    E, _, F2 = W1.shape
    F = F2 // 2
    k = ids.shape[1]
    if y_slots is None:
        y_slots = torch.empty(T * k, H, dtype=torch.bfloat16, device=x.device)
    need = moe_experts_partial_workspace(c, T, E, k, H, F)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    mask = (ctypes.c_uint8 * E)(*[1 if v else 0 for v in expert_mask])
    st = c.lib.iso_moe_experts_partial(c.handle, _ptr(x), _ptr(ids), _ptr(W1), _ptr(W2), ctypes.cast(mask, _vp),
                                       _ptr(y_slots), T, E, k, H, F, _ptr(ws), ws.numel(), _stream(stream))
    c.lib.check(st, "iso_moe_experts_partial")
    return y_slots


def last_device_status(c: Contract, stream=None) -> int:
    return c.lib.iso_last_device_status(_stream(stream))
