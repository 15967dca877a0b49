"""numpy front end of the fp64 CPU oracle (oracle/spec_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg.  The product package never imports it.

Inputs are numpy arrays (or CPU torch tensors converted by the caller):
f32 logits as float32, bf16 logits as their raw uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
STOCHASTIC, GREEDY = 0, 1

_lib = None


def lib(path=None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _bind(L):
    P = ctypes.c_void_p
    i32, f32, f64 = ctypes.c_int, ctypes.c_float, ctypes.c_double
    L.so_verify_chain.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, f32,
                                  P, P, P, P, P, P, P, P, P, P, i32]
    L.so_verify_chain.restype = None
    L.so_verify_chain_trunc.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, f32, P, P,
                                        P, P, P, P, P, P, P, P, P, P, i32]
    L.so_verify_chain_trunc.restype = None
    L.so_verify_tree.argtypes = [i32, i32, i32, i32, P, P, P, P, f32, P, P, P, P, P, i32]
    L.so_verify_tree.restype = None
    L.so_rollback_lengths.argtypes = [i32, i32, P, P, P, P, ctypes.c_int32, P, P, P]
    L.so_rollback_lengths.restype = None
    L.so_expected_tokens.argtypes = [f64, i32]
    L.so_expected_tokens.restype = f64
    L.so_speedup.argtypes = [f64, i32, f64, f64]
    L.so_speedup.restype = f64
    ll = ctypes.c_longlong
    L.so_kv_compact_tree.argtypes = [i32, i32, i32, ll, ll, P, ll, ll, ll, P, P, P, P]
    L.so_kv_compact_tree.restype = None
    L.so_adaptive_policy.argtypes = [i32, f64, f64, P, P, P, f64, i32, P, P, P, P, P, P]
    L.so_adaptive_policy.restype = None
    L.so_drift_residuals.argtypes = [i32, i32, i32, i32, P, P, P, i32, P, P, P, i32]
    L.so_drift_residuals.restype = None
    L.so_max_threads.argtypes = []
    L.so_max_threads.restype = i32
    return L


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """Return (contiguous array, dtype code) for f32 or bf16-as-uint16 logits."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


def verify_chain(target, draft, draft_tokens, temperature=None, u_accept=None,
                 u_sample=None, mode=STOCHASTIC, kappa=0.0, nthreads=0, L=None,
                 top_k=None, top_p=None):
    """Run the oracle chain verifier.  Returns a dict of numpy outputs.
    top_k [B] int32 / top_p [B] float32 (optional) truncate p and q."""
    L = L or lib()
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    if draft is not None:
        draft, dt2 = _logits(draft)
        assert dt2 == dt and draft.shape == (B, K, V)
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, K)
    temp = None if temperature is None else np.ascontiguousarray(temperature, dtype=np.float32)
    if mode == STOCHASTIC:
        ua = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, K)
        us = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B, K + 1)
    else:
        ua = us = None
    out = dict(
        accepted_len=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, K + 1), np.int32),
        num_emitted=np.zeros(B, np.int32),
        row_status=np.zeros(B, np.int32),
        p_at_draft=np.zeros((B, K)),
        q_at_draft=np.zeros((B, K)),
        ratio=np.zeros((B, K)),
        resid_mass=np.zeros((B, K)),
        accept_margin=np.zeros((B, K)),
        row_margin=np.zeros(B),
    )
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32).reshape(B)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32).reshape(B)
    L.so_verify_chain_trunc(B, K, V, dt, mode, _ptr(target), _ptr(draft), _ptr(toks), _ptr(temp),
                      _ptr(ua), _ptr(us), float(kappa), _ptr(tk), _ptr(tp),
                      _ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
                      _ptr(out["num_emitted"]), _ptr(out["row_status"]),
                      _ptr(out["p_at_draft"]), _ptr(out["q_at_draft"]), _ptr(out["ratio"]),
                      _ptr(out["resid_mass"]), _ptr(out["accept_margin"]),
                      _ptr(out["row_margin"]), int(nthreads))
    return out


def verify_tree(target, parent, node_tokens, temperature=None, kappa=0.0, nthreads=0, L=None):
    """Run the oracle tree verifier.  Returns a dict of numpy outputs."""
    L = L or lib()
    target, dt = _logits(target)
    B, N, V = target.shape
    par = np.ascontiguousarray(parent, dtype=np.int32).reshape(B, N)
    toks = np.ascontiguousarray(node_tokens, dtype=np.int32).reshape(B, N)
    temp = None if temperature is None else np.ascontiguousarray(temperature, dtype=np.float32)
    out = dict(
        accepted_len=np.zeros(B, np.int32),
        path_nodes=np.zeros((B, N), np.int32),
        out_tokens=np.zeros((B, N), np.int32),
        num_emitted=np.zeros(B, np.int32),
        row_status=np.zeros(B, np.int32),
    )
    L.so_verify_tree(B, N, V, dt, _ptr(target), _ptr(par), _ptr(toks), _ptr(temp), float(kappa),
                     _ptr(out["accepted_len"]), _ptr(out["path_nodes"]), _ptr(out["out_tokens"]),
                     _ptr(out["num_emitted"]), _ptr(out["row_status"]), int(nthreads))
    return out


def rollback_lengths(kv_len_in, accepted_len, num_emitted, out_tokens, eos_id=-1,
                     max_len=None, L=None):
    """Run the oracle KV-length rollback.  Returns (committed_kv_len, num_emitted_out)."""
    L = L or lib()
    kv = np.ascontiguousarray(kv_len_in, dtype=np.int32)
    acc = np.ascontiguousarray(accepted_len, dtype=np.int32)
    ne = np.ascontiguousarray(num_emitted, dtype=np.int32)
    toks = np.ascontiguousarray(out_tokens, dtype=np.int32)
    B, max_emit = toks.shape
    ml = None if max_len is None else np.ascontiguousarray(max_len, dtype=np.int32)
    committed = np.zeros(B, np.int32)
    ne_out = np.zeros(B, np.int32)
    L.so_rollback_lengths(B, max_emit, _ptr(kv), _ptr(acc), _ptr(ne), _ptr(toks), int(eos_id),
                          _ptr(ml), _ptr(committed), _ptr(ne_out))
    return committed, ne_out


def expected_tokens(alpha, gamma, L=None):
    return (L or lib()).so_expected_tokens(float(alpha), int(gamma))


def speedup(alpha, gamma, c, g=1.0, L=None):
    return (L or lib()).so_speedup(float(alpha), int(gamma), float(c), float(g))


def max_threads(L=None):
    return (L or lib()).so_max_threads()


def kv_compact_tree(kv, kv_len_in, accepted_len, path_nodes, L=None):
    """Compact the accepted tree path of each row in a copy of `kv`.

    kv: uint8 array [planes, B, S_max, E] (C order); path_nodes: [B, N] int32.
    Returns (new_kv, row_status)."""
    kv = np.array(kv, dtype=np.uint8, order="C", copy=True)
    P_, B, S_max, E = kv.shape
    path = np.ascontiguousarray(path_nodes, dtype=np.int32)
    N = path.shape[1]
    kvl = np.ascontiguousarray(kv_len_in, dtype=np.int32)
    acc = np.ascontiguousarray(accepted_len, dtype=np.int32)
    st = np.zeros(B, dtype=np.int32)
    (L or lib()).so_kv_compact_tree(B, N, P_, S_max, E, _ptr(kv), B * S_max * E, S_max * E, E,
                                    _ptr(kvl), _ptr(acc), _ptr(path), _ptr(st))
    return kv, st


SHALLOW, DEEP = (3, 4, 4), (7, 1, 8)


def adaptive_policy(accepted_len, depth, draft_top1, ema, zero_run, alpha=0.3, divisor=1.0,
                    lo=SHALLOW, hi=DEEP, start=SHALLOW, ema0=0.0, breaker=5, L=None):
    """One policy step.  Returns (shape [B,3] int32, new ema, new zero_run)."""
    acc = np.ascontiguousarray(accepted_len, dtype=np.int32)
    B = acc.shape[0]
    dep = np.ascontiguousarray(depth, dtype=np.int32)
    p1 = np.ascontiguousarray(draft_top1, dtype=np.float32)
    e = np.array(ema, dtype=np.float64, copy=True)
    z = np.array(zero_run, dtype=np.int32, copy=True)
    shape = np.zeros((B, 3), dtype=np.int32)
    lo_, hi_, st_ = (np.ascontiguousarray(x, dtype=np.int32) for x in (lo, hi, start))
    (L or lib()).so_adaptive_policy(B, float(alpha), float(divisor), _ptr(lo_), _ptr(hi_),
                                    _ptr(st_), float(ema0), int(breaker), _ptr(acc), _ptr(dep),
                                    _ptr(p1), _ptr(e), _ptr(z), _ptr(shape))
    return shape, e, z


def drift_residuals(target, draft, temperature=None, m=32, nthreads=0, L=None):
    """Top-m target support and log p - log q on it at every drafted position.

    target [B,K+1,V], draft [B,K,V] (float32, or bf16 as uint16 bits).
    Returns (support [B,K,m] int32, residual [B,K,m] float32, row_status [B])."""
    t, dt = _logits(target)
    d, _ = _logits(draft)
    B, K1, V = t.shape
    K = K1 - 1
    temp = None if temperature is None else np.ascontiguousarray(temperature, dtype=np.float32)
    sup = np.zeros((B, K, m), dtype=np.int32)
    res = np.zeros((B, K, m), dtype=np.float32)
    st = np.zeros(B, dtype=np.int32)
    (L or lib()).so_drift_residuals(B, K, V, dt, _ptr(t), _ptr(d), _ptr(temp), int(m), _ptr(sup),
                                    _ptr(res), _ptr(st), int(nthreads))
    return sup, res, st
