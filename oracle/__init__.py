"""Float64 CPU oracle for the invariant GEMM, RMSNorm, selected-token logprob
and MoE expert layer.

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library under
``parallelism_invariant_logprob_gb300`` never does, and this package never
imports it.  The arithmetic lives in ``iso_oracle.c`` (plain C, double
precision, compiled with ``-ffp-contract=off``); this module only marshals
numpy arrays into it.

bf16 tensors cross this boundary as ``numpy.uint16`` bit patterns.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):
  gemm_root / leaf_partial / tree_combine : pinned (exact rational brute force,
      exact-integer inputs, identity/permutation B, tree-shape fixture,
      textbook matmul for one leaf, partial+combine == single pass)
  rmsnorm        : pinned (exact brute force, constant-row closed form)
  selected_logprob : pinned (brute-force log-softmax, identities: logprob <= 0,
      logsumexp of the full distribution = 0, chunked == direct LSE, W = 0)
  lse_merge      : pinned (closed form log(e^a + e^b))
  moe_route / moe_permute : pinned (library sort with the stated tie rule)
  moe_layer / moe_combine : pinned (k = 1 dense-FFN reduction against textbook
      matmul + SwiGLU, one-hot gates, equal gates)
  delta          : pinned (worked examples printed in the VeXact paper, Table 1,
      and the RL-Kernel blog, §1 "Minimal Example")
  attention      : pinned (numpy softmax(QK^T)V brute force per head with the GQA
      map, one visible key -> that value row, equal scores -> mean of the visible
      values, causality: keys past a row's position do not change it)
  mismatch       : pinned (Table 1 deltas and mismatch count, identical inputs,
      closed forms of r_corr, K1, K3 and the tau_tok truncation, math.fsum
      brute-force sequence sums, both sides of the tau_seq rejection, the
      small-delta expansion of K3)
"""
from __future__ import annotations

import ctypes
import os
import numpy as np

from .build_oracle import build as _build, library_path

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        _build()
    lib = ctypes.CDLL(path)
    lib.iso_oracle_bf16_to_double.restype = ctypes.c_double
    lib.iso_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.iso_oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.iso_oracle_double_to_bf16.argtypes = [ctypes.c_double]
    lib.iso_oracle_round_bf16.argtypes = [_f64p, _i64, _u16p]
    lib.iso_oracle_gemm_root.argtypes = [_u16p, _i64, _u16p, _i64, _int, _int, _int, _int, _int, _int,
                                         _f64p, _i64, _int]
    lib.iso_oracle_gemm_leaf_partial.argtypes = [_u16p, _i64, _u16p, _i64, _int, _int, _int, _int, _int,
                                                 _f64p, _i64, _int]
    lib.iso_oracle_tree_combine.argtypes = [_f64p, _int, _i64, _int, _int, _i64, _f64p, _i64]
    lib.iso_oracle_rmsnorm.argtypes = [_u16p, _u16p, ctypes.c_double, _int, _int, _u16p, _f64p, _int]
    lib.iso_oracle_lse_merge.argtypes = [ctypes.c_double] * 4 + [_f64p, _f64p]
    lib.iso_oracle_logprob_num_chunks.argtypes = [_int, _int, _int]
    lib.iso_oracle_selected_logprob.argtypes = [_u16p, _u16p, _i32p, _int, _int, _int, _int, _int, _int,
                                                _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _int]
    lib.iso_oracle_moe_route.argtypes = [_f32p, _int, _int, _int, _i32p, _f64p]
    lib.iso_oracle_moe_permute.argtypes = [_i32p, _int, _int, _int, _u8p, _i32p, _i32p]
    lib.iso_oracle_moe_layer.argtypes = [_u16p, _i32p, _f64p, _u16p, _u16p, _int, _int, _int, _int, _int,
                                         _int, _u16p, _u16p, _f64p, _int]
    lib.iso_oracle_moe_combine.argtypes = [_u16p, _f64p, _int, _int, _int, _u16p, _f64p]
    lib.iso_oracle_delta.argtypes = [_f64p, _f64p, _i64, _f64p]
    lib.iso_oracle_attention.argtypes = [_u16p, _u16p, _u16p, _i32p, _i32p, _i32p, _int, _int, _int, _int,
                                         ctypes.c_double, _f64p, _u16p, _f64p]
    lib.iso_oracle_mismatch.argtypes = [_f32p, _f32p, _i32p, _int, ctypes.c_double, ctypes.c_double, _f64p, _f64p,
                                        _f64p, _f64p, _u8p, _u8p, _f64p, _i32p]
    _lib = lib
    return lib


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a, ptype):
    if a is None:
        return ctypes.cast(None, ptype)
    return a.ctypes.data_as(ptype)


def _check(rc, what):
    if rc < 0:
        raise ValueError(f"oracle {what}: invalid arguments (status {rc})")


# ---------------------------------------------------------------- bf16 bits
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact float64 values (numpy, no library call)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 (ties to even), as uint16 bits."""
    lib = _load()
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.iso_oracle_round_bf16(_p(x, _f64p), x.size, _p(out, _u16p))
    return out


# --------------------------------------------------------------------- GEMM
def gemm_root(A, B, L, leaf_lo=0, leaf_hi=None, nthreads=None):
    """Root (float64, unrounded) of the balanced tree over K-leaves
    [leaf_lo, leaf_hi) of A[M,K] @ B[K,N] (bf16 bits in, float64 out)."""
    lib = _load()
    A = _c(A, np.uint16)
    B = _c(B, np.uint16)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    if leaf_hi is None:
        leaf_hi = L
    root = np.empty((M, N), dtype=np.float64)
    rc = lib.iso_oracle_gemm_root(_p(A, _u16p), K, _p(B, _u16p), N, M, N, K, L, leaf_lo, leaf_hi,
                                  _p(root, _f64p), N, _threads(nthreads))
    _check(rc, "gemm_root")
    return root


def gemm(A, B, L, nthreads=None):
    """C = bf16(tree root): the invariant GEMM's defined result (uint16 bits)."""
    return round_bf16(gemm_root(A, B, L, nthreads=nthreads))


def gemm_leaf_partial(A_r, B_r, L, R, nthreads=None):
    """Subtree root of one simulated rank: its K_local = K/R slice holds L/R leaves."""
    lib = _load()
    A_r = _c(A_r, np.uint16)
    B_r = _c(B_r, np.uint16)
    M, Kl = A_r.shape
    N = B_r.shape[1]
    S = np.empty((M, N), dtype=np.float64)
    rc = lib.iso_oracle_gemm_leaf_partial(_p(A_r, _u16p), Kl, _p(B_r, _u16p), N, M, N, Kl, L, R,
                                          _p(S, _f64p), N, _threads(nthreads))
    _check(rc, "gemm_leaf_partial")
    return S


def tree_combine(S):
    """Top log2(R) tree levels over S[R, M, N] (float64) -> float64 root."""
    lib = _load()
    S = _c(S, np.float64)
    R, M, N = S.shape
    root = np.empty((M, N), dtype=np.float64)
    rc = lib.iso_oracle_tree_combine(_p(S, _f64p), R, M * N, M, N, N, _p(root, _f64p), N)
    _check(rc, "tree_combine")
    return root


# ------------------------------------------------------------------ RMSNorm
def rmsnorm(x, gamma, eps, nthreads=None, exact=False):
    lib = _load()
    x = _c(x, np.uint16)
    gamma = _c(gamma, np.uint16)
    T, H = x.shape
    y = np.empty((T, H), dtype=np.uint16)
    ye = np.empty((T, H), dtype=np.float64) if exact else None
    rc = lib.iso_oracle_rmsnorm(_p(x, _u16p), _p(gamma, _u16p), float(eps), T, H, _p(y, _u16p),
                                _p(ye, _f64p), _threads(nthreads))
    _check(rc, "rmsnorm")
    return (y, ye) if exact else y


# ------------------------------------------------------------------ logprob
def lse_merge(m1, s1, m2, s2):
    lib = _load()
    m = ctypes.c_double()
    s = ctypes.c_double()
    lib.iso_oracle_lse_merge(m1, s1, m2, s2, ctypes.byref(m), ctypes.byref(s))
    return m.value, s.value


def num_chunks(V, tile_cols=128, chunk_tiles=19):
    return _load().iso_oracle_logprob_num_chunks(V, tile_cols, chunk_tiles)


def selected_logprob(h, W, ids, L, tile_cols=128, chunk_tiles=19, nthreads=None, chunk_stats=False):
    """Returns dict(out, lse, lse_direct, z_sel[, chunk_m, chunk_s]) in float64."""
    lib = _load()
    h = _c(h, np.uint16)
    W = _c(W, np.uint16)
    ids = _c(ids, np.int32)
    T, H = h.shape
    H2, V = W.shape
    assert H == H2 and ids.shape == (T,)
    out = np.empty(T, np.float64)
    lse = np.empty(T, np.float64)
    lsed = np.empty(T, np.float64)
    zs = np.empty(T, np.float64)
    C = num_chunks(V, tile_cols, chunk_tiles)
    cm = np.empty((T, C), np.float64) if chunk_stats else None
    cs = np.empty((T, C), np.float64) if chunk_stats else None
    rc = lib.iso_oracle_selected_logprob(_p(h, _u16p), _p(W, _u16p), _p(ids, _i32p), T, H, V, L,
                                         tile_cols, chunk_tiles, _p(out, _f64p), _p(lse, _f64p),
                                         _p(lsed, _f64p), _p(zs, _f64p), _p(cm, _f64p), _p(cs, _f64p),
                                         _threads(nthreads))
    _check(rc, "selected_logprob")
    r = dict(out=out, lse=lse, lse_direct=lsed, z_sel=zs)
    if chunk_stats:
        r.update(chunk_m=cm, chunk_s=cs)
    return r


# ---------------------------------------------------------------------- MoE
def moe_route(logits, k):
    lib = _load()
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = lib.iso_oracle_moe_route(_p(logits, _f32p), T, E, k, _p(ids, _i32p), _p(w, _f64p))
    _check(rc, "moe_route")
    return ids, w


def moe_permute(ids, E, mask=None):
    lib = _load()
    ids = _c(ids, np.int32)
    T, k = ids.shape
    perm = np.empty(T * k, np.int32)
    offs = np.empty(E + 1, np.int32)
    m = None if mask is None else _c(mask, np.uint8)
    n = lib.iso_oracle_moe_permute(_p(ids, _i32p), T, E, k, _p(m, _u8p), _p(perm, _i32p), _p(offs, _i32p))
    _check(n, "moe_permute")
    return perm[:n].copy(), offs


def moe_layer(x, ids, w, W1, W2, L, nthreads=None, with_slots=False, exact=False):
    lib = _load()
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    T, H = x.shape
    E, H2, F2 = W1.shape
    F = F2 // 2
    k = ids.shape[1]
    assert H == H2 and W2.shape == (E, F, H)
    out = np.empty((T, H), np.uint16)
    ys = np.empty((T, k, H), np.uint16) if with_slots else None
    oe = np.empty((T, H), np.float64) if exact else None
    rc = lib.iso_oracle_moe_layer(_p(x, _u16p), _p(ids, _i32p), _p(w, _f64p), _p(W1, _u16p), _p(W2, _u16p),
                                  T, E, k, H, F, L, _p(ys, _u16p), _p(out, _u16p), _p(oe, _f64p),
                                  _threads(nthreads))
    _check(rc, "moe_layer")
    res = dict(out=out)
    if with_slots:
        res["y_slots"] = ys
    if exact:
        res["out_exact"] = oe
    return res


def moe_combine(y_slots, w, exact=False):
    lib = _load()
    y_slots = _c(y_slots, np.uint16)
    w = _c(w, np.float64)
    T, k, H = y_slots.shape
    out = np.empty((T, H), np.uint16)
    oe = np.empty((T, H), np.float64) if exact else None
    rc = lib.iso_oracle_moe_combine(_p(y_slots, _u16p), _p(w, _f64p), T, k, H, _p(out, _u16p), _p(oe, _f64p))
    _check(rc, "moe_combine")
    return (out, oe) if exact else out


# ----------------------------------------------------------------- delta_t
def attention(Q, K, V, q_start, k_start, pos0, scale):
    """Causal attention over packed sequences (plain definition in double).  Q [Tq, Hq, d],
    K and V [Tk, Hkv, d] as bf16 bit patterns; returns dict(out (bf16 bits), out_exact, lse)."""
    lib = _load()
    Q = _c(Q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    qs = _c(q_start, np.int32)
    ks = _c(k_start, np.int32)
    p0 = _c(pos0, np.int32)
    Tq, Hq, d = Q.shape
    Hkv = K.shape[1]
    B = qs.size - 1
    oe = np.empty((Tq, Hq, d), np.float64)
    o = np.empty((Tq, Hq, d), np.uint16)
    lse = np.empty((Tq, Hq), np.float64)
    rc = lib.iso_oracle_attention(_p(Q, _u16p), _p(K, _u16p), _p(V, _u16p), _p(qs, _i32p), _p(ks, _i32p),
                                  _p(p0, _i32p), B, Hq, Hkv, d, float(scale), _p(oe, _f64p), _p(o, _u16p),
                                  _p(lse, _f64p))
    _check(rc, "attention")
    return dict(out=o, out_exact=oe, lse=lse)


def mismatch(logp_train, logp_rollout, offsets, tau_tok=2.0, tau_seq=0.001):
    """Mismatch diagnostics over packed sequences (VeXact paper, Eq. 1, 6, 7; K1/K3 of §4.1):
    per token delta, min(r_corr, tau_tok); per sequence sum K1, sum K3, the rejection
    masks S <= tau_seq, max |delta| and the count of tokens whose logprobs differ."""
    lib = _load()
    a = _c(logp_train, np.float32)
    b = _c(logp_rollout, np.float32)
    off = _c(offsets, np.int32)
    B = off.size - 1
    N = a.size
    d = np.empty(N, np.float64)
    w = np.empty(N, np.float64)
    k1 = np.empty(B, np.float64)
    k3 = np.empty(B, np.float64)
    a1 = np.empty(B, np.uint8)
    a3 = np.empty(B, np.uint8)
    mx = np.empty(B, np.float64)
    nm = np.empty(B, np.int32)
    rc = lib.iso_oracle_mismatch(_p(a, _f32p), _p(b, _f32p), _p(off, _i32p), B, tau_tok, tau_seq, _p(d, _f64p),
                                 _p(w, _f64p), _p(k1, _f64p), _p(k3, _f64p), _p(a1, _u8p), _p(a3, _u8p),
                                 _p(mx, _f64p), _p(nm, _i32p))
    _check(rc, "mismatch")
    return dict(delta=d, tis_weight=w, seq_k1=k1, seq_k3=k3, accept_k1=a1, accept_k3=a3, seq_max_abs_delta=mx,
                seq_mismatches=nm)


def delta(logp_train, logp_rollout):
    lib = _load()
    a = _c(logp_train, np.float64)
    b = _c(logp_rollout, np.float64)
    d = np.empty(a.shape, np.float64)
    lib.iso_oracle_delta(_p(a, _f64p), _p(b, _f64p), a.size, _p(d, _f64p))
    return d
