"""ctypes binding of libspecverify.so: argument marshalling only.

Takes torch CUDA tensors, passes their device pointers, the current CUDA
stream and a cached workspace to the C ABI declared in
include/specverify.h, and returns the output tensors.  Every step of the
computation runs in the library's kernels; there is no other code path.
"""
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_F32, SPEC_BF16 = 0, 1
SPEC_STOCHASTIC, SPEC_GREEDY = 0, 1
ROW_STATUS = {0: "OK", 1: "NONFINITE", 2: "BAD_TOKEN", 3: "BAD_UNIFORM", 4: "BAD_PARENT",
              5: "EMPTY", 6: "TIMEOUT", 7: "BAD_TEMPERATURE"}

_c = ctypes
_P = _c.c_void_p


class SpecChainArgs(_c.Structure):
    _fields_ = [("B", _c.c_int32), ("K", _c.c_int32), ("V", _c.c_int32), ("dtype", _c.c_int32),
                ("mode", _c.c_int32), ("margin_kappa", _c.c_float),
                ("target_logits", _P), ("draft_logits", _P), ("draft_tokens", _P),
                ("temperature", _P), ("u_accept", _P), ("u_sample", _P)]


class SpecChainOut(_c.Structure):
    _fields_ = [("accepted_len", _P), ("out_tokens", _P), ("num_emitted", _P),
                ("row_status", _P), ("p_at_draft", _P), ("q_at_draft", _P), ("resid_mass", _P)]


class SpecTreeArgs(_c.Structure):
    _fields_ = [("B", _c.c_int32), ("N", _c.c_int32), ("V", _c.c_int32), ("dtype", _c.c_int32),
                ("margin_kappa", _c.c_float), ("target_logits", _P), ("parent", _P),
                ("node_tokens", _P), ("temperature", _P)]


class SpecTreeOut(_c.Structure):
    _fields_ = [("accepted_len", _P), ("path_nodes", _P), ("out_tokens", _P),
                ("num_emitted", _P), ("row_status", _P)]


class SpecTruncation(_c.Structure):
    _fields_ = [("top_k", _P), ("top_p", _P)]


class SpecKvCompactArgs(_c.Structure):
    _fields_ = [("B", _c.c_int32), ("N", _c.c_int32), ("planes", _c.c_int32), ("pad", _c.c_int32),
                ("S_max", _c.c_int64), ("entry_bytes", _c.c_int64), ("plane_stride", _c.c_int64),
                ("row_stride", _c.c_int64), ("tok_stride", _c.c_int64), ("kv", _P),
                ("kv_len_in", _P), ("accepted_len", _P), ("path_nodes", _P)]


class SpecAdaptiveParams(_c.Structure):
    _fields_ = [("alpha", _c.c_double), ("divisor", _c.c_double), ("ema0", _c.c_double),
                ("shallow", _c.c_int32 * 3), ("deep", _c.c_int32 * 3), ("start", _c.c_int32 * 3),
                ("breaker", _c.c_int32)]


class SpecError(RuntimeError):
    """A spec_* entry point returned a non-zero spec_status."""

    def __init__(self, code, msg):
        super().__init__(msg)
        self.code = code


_lib = None
_lib_lock = threading.Lock()


def lib(path=None):
    """The loaded C library (raises if it was never built)."""
    global _lib
    if path is not None:
        return _bind(_c.CDLL(path))
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            _lib = _bind(_c.CDLL(LIB_PATH))
    return _lib


def _bind(L):
    i32, u64, sz = _c.c_int32, _c.c_uint64, _c.c_size_t
    L.spec_verify_chain_workspace_size.argtypes = [i32, i32, i32]
    L.spec_verify_chain_workspace_size.restype = sz
    L.spec_verify_chain_truncated_workspace_size.argtypes = [i32, i32, i32]
    L.spec_verify_chain_truncated_workspace_size.restype = sz
    L.spec_verify_tree_workspace_size.argtypes = [i32, i32, i32]
    L.spec_verify_tree_workspace_size.restype = sz
    L.spec_verify_chain.argtypes = [_c.POINTER(SpecChainArgs), _c.POINTER(SpecChainOut), _P, sz, _P]
    L.spec_verify_chain.restype = _c.c_int
    L.spec_verify_chain_static.argtypes = [_c.POINTER(SpecChainArgs), _c.POINTER(SpecChainOut), _P]
    L.spec_verify_chain_static.restype = _c.c_int
    L.spec_verify_tree.argtypes = [_c.POINTER(SpecTreeArgs), _c.POINTER(SpecTreeOut), _P, sz, _P]
    L.spec_verify_tree.restype = _c.c_int
    L.spec_verify_chain_truncated.argtypes = [_c.POINTER(SpecChainArgs), _c.POINTER(SpecTruncation),
                                              _c.POINTER(SpecChainOut), _P, sz, _P]
    L.spec_verify_chain_truncated.restype = _c.c_int
    L.spec_drift_residuals.argtypes = [_c.POINTER(SpecChainArgs), i32, _P, _P, _P, _P, sz, _P]
    L.spec_drift_residuals.restype = _c.c_int
    L.spec_kv_compact_tree.argtypes = [_c.POINTER(SpecKvCompactArgs), _P, _P]
    L.spec_kv_compact_tree.restype = _c.c_int
    L.spec_adaptive_tree_policy.argtypes = [_c.POINTER(SpecAdaptiveParams), i32, _P, _P, _P, _P,
                                            _P, _P, _P]
    L.spec_adaptive_tree_policy.restype = _c.c_int
    L.spec_rollback_lengths.argtypes = [i32, i32, _P, _P, _P, _P, i32, _P, _P, _P, _P]
    L.spec_rollback_lengths.restype = _c.c_int
    L.spec_workspace_init.argtypes = [_P, sz, _P]
    L.spec_workspace_init.restype = _c.c_int
    L.spec_status_string.argtypes = [_c.c_int]
    L.spec_status_string.restype = _c.c_char_p
    L.spec_set_wait_timeout_ns.argtypes = [u64]
    L.spec_set_wait_timeout_ns.restype = None
    L.spec_get_wait_timeout_ns.argtypes = []
    L.spec_get_wait_timeout_ns.restype = u64
    L.spec_debug_force_wait_timeout.argtypes = [_c.c_int]
    L.spec_debug_force_wait_timeout.restype = None
    return L


def _check(code):
    if code != 0:
        raise SpecError(code, lib().spec_status_string(code).decode())


def _ptr(t):
    return None if t is None else _P(t.data_ptr())


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _req(t, name, device, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a tensor on {device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# Workspaces: one buffer per (device, stream), grown on demand.  The library
# needs no particular contents; it keeps a small header at the buffer's end
# between calls, so the same buffer is always passed with its full size.
_ws = {}
_ws_lock = threading.Lock()


def workspace(device, nbytes, stream):
    key = (device, stream)
    with _ws_lock:
        buf = _ws.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws[key] = buf
    return buf


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s, _P(s.cuda_stream)


def spec_verify_chain(target_logits, draft_logits, draft_tokens, temperature=None,
                      u_accept=None, u_sample=None, mode="stochastic", margin_kappa=0.0,
                      diagnostics=False, out=None, stream=None, top_k=None, top_p=None):
    """Verify B draft chains (see spec_verify_chain in include/specverify.h).

    target_logits [B,K+1,V] and draft_logits [B,K,V] (bf16 or fp32, CUDA),
    draft_tokens [B,K] int32, temperature [B] fp32 or None, u_accept [B,K] and
    u_sample [B,K+1] fp32 (stochastic mode).  mode: "stochastic" | "greedy".
    Returns a dict of CUDA tensors: accepted_len, out_tokens, num_emitted,
    row_status (+ p_at_draft, q_at_draft, resid_mass with diagnostics=True).
    top_k [B] int32 / top_p [B] float32 (stochastic mode, optional) truncate
    p and q (spec_verify_chain_truncated).
    """
    dev = target_logits.device
    greedy = mode == "greedy"
    _req(target_logits, "target_logits", dev)
    B, K1, V = target_logits.shape
    K = K1 - 1
    dt = _dtype_code(target_logits)
    if not greedy or draft_logits is not None:
        _req(draft_logits, "draft_logits", dev, target_logits.dtype)
    _req(draft_tokens, "draft_tokens", dev, torch.int32)
    _req(temperature, "temperature", dev, torch.float32)
    _req(u_accept, "u_accept", dev, torch.float32)
    _req(u_sample, "u_sample", dev, torch.float32)
    if out is None:
        out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                   num_emitted=torch.empty(B, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
        if diagnostics and not greedy:
            for k in ("p_at_draft", "q_at_draft", "resid_mass"):
                out[k] = torch.empty(B, K, dtype=torch.float32, device=dev)
    args = SpecChainArgs(B, K, V, dt, SPEC_GREEDY if greedy else SPEC_STOCHASTIC,
                         float(margin_kappa), _ptr(target_logits),
                         None if greedy else _ptr(draft_logits), _ptr(draft_tokens),
                         _ptr(temperature), None if greedy else _ptr(u_accept),
                         None if greedy else _ptr(u_sample))
    o = SpecChainOut(_ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
                     _ptr(out["num_emitted"]), _ptr(out["row_status"]),
                     _ptr(out.get("p_at_draft")), _ptr(out.get("q_at_draft")),
                     _ptr(out.get("resid_mass")))
    L = lib()
    truncated = top_k is not None or top_p is not None
    nbytes = (L.spec_verify_chain_truncated_workspace_size if truncated
              else L.spec_verify_chain_workspace_size)(B, K, V)
    s, sp = _stream(dev, stream)
    ws = workspace(dev, nbytes, s.cuda_stream)
    if not truncated:
        _check(L.spec_verify_chain(_c.byref(args), _c.byref(o), _ptr(ws), ws.numel(), sp))
    else:
        if greedy:
            raise ValueError("top_k / top_p apply to mode='stochastic' only")
        _req(top_k, "top_k", dev, torch.int32)
        _req(top_p, "top_p", dev, torch.float32)
        t = SpecTruncation(_ptr(top_k), _ptr(top_p))
        _check(L.spec_verify_chain_truncated(_c.byref(args), _c.byref(t), _c.byref(o), _ptr(ws),
                                             ws.numel(), sp))
    return out


def spec_verify_tree(target_logits, parent, node_tokens, temperature=None, margin_kappa=0.0,
                     out=None, stream=None):
    """Verify one draft tree per row (see spec_verify_tree in include/specverify.h).

    target_logits [B,N,V] (bf16 or fp32), parent [B,N] int32, node_tokens
    [B,N] int32.  Returns accepted_len, path_nodes, out_tokens, num_emitted,
    row_status.
    """
    dev = target_logits.device
    _req(target_logits, "target_logits", dev)
    B, N, V = target_logits.shape
    dt = _dtype_code(target_logits)
    _req(parent, "parent", dev, torch.int32)
    _req(node_tokens, "node_tokens", dev, torch.int32)
    _req(temperature, "temperature", dev, torch.float32)
    if out is None:
        out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
                   path_nodes=torch.empty(B, N, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty(B, N, dtype=torch.int32, device=dev),
                   num_emitted=torch.empty(B, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
    args = SpecTreeArgs(B, N, V, dt, float(margin_kappa), _ptr(target_logits), _ptr(parent),
                        _ptr(node_tokens), _ptr(temperature))
    o = SpecTreeOut(_ptr(out["accepted_len"]), _ptr(out["path_nodes"]), _ptr(out["out_tokens"]),
                    _ptr(out["num_emitted"]), _ptr(out["row_status"]))
    L = lib()
    nbytes = L.spec_verify_tree_workspace_size(B, N, V)
    s, sp = _stream(dev, stream)
    ws = workspace(dev, nbytes, s.cuda_stream)
    _check(L.spec_verify_tree(_c.byref(args), _c.byref(o), _ptr(ws), ws.numel(), sp))
    return out


def spec_rollback_lengths(kv_len_in, accepted_len, num_emitted, out_tokens, eos_id=-1,
                          max_len=None, stream=None):
    """Committed KV lengths (see spec_rollback_lengths in include/specverify.h).

    Returns (committed_kv_len [B], num_emitted_out [B]) int32 CUDA tensors.
    """
    dev = out_tokens.device
    for t, n in ((kv_len_in, "kv_len_in"), (accepted_len, "accepted_len"),
                 (num_emitted, "num_emitted"), (out_tokens, "out_tokens"), (max_len, "max_len")):
        _req(t, n, dev, torch.int32)
    B, max_emit = out_tokens.shape
    committed = torch.empty(B, dtype=torch.int32, device=dev)
    n_out = torch.empty(B, dtype=torch.int32, device=dev)
    _, sp = _stream(dev, stream)
    _check(lib().spec_rollback_lengths(B, max_emit, _ptr(kv_len_in), _ptr(accepted_len),
                                       _ptr(num_emitted), _ptr(out_tokens), int(eos_id),
                                       _ptr(max_len), _ptr(committed), _ptr(n_out), sp))
    return committed, n_out


def spec_drift_residuals(target_logits, draft_logits, temperature=None, m=32, stream=None):
    """Top-m target support and log p - log q on it at every drafted position
    (see spec_drift_residuals in include/specverify.h).  Returns (support
    [B,K,m] int32, residual [B,K,m] float32, row_status [B] int32)."""
    dev = target_logits.device
    _req(target_logits, "target_logits", dev)
    _req(draft_logits, "draft_logits", dev, target_logits.dtype)
    _req(temperature, "temperature", dev, torch.float32)
    B, K1, V = target_logits.shape
    K = K1 - 1
    sup = torch.empty(B, K, m, dtype=torch.int32, device=dev)
    res = torch.empty(B, K, m, dtype=torch.float32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)
    args = SpecChainArgs(B, K, V, _dtype_code(target_logits), SPEC_STOCHASTIC, 0.0,
                         _ptr(target_logits), _ptr(draft_logits), None, _ptr(temperature),
                         None, None)
    L = lib()
    nbytes = L.spec_verify_chain_truncated_workspace_size(B, K, V)
    s, sp = _stream(dev, stream)
    ws = workspace(dev, nbytes, s.cuda_stream)
    _check(L.spec_drift_residuals(_c.byref(args), int(m), _ptr(sup), _ptr(res), _ptr(st),
                                  _ptr(ws), ws.numel(), sp))
    return sup, res, st


def spec_kv_compact_tree(kv, kv_len_in, accepted_len, path_nodes, stream=None):
    """Compact each row's accepted tree path in place (see spec_kv_compact_tree
    in include/specverify.h).

    kv: a CUDA tensor [planes, B, S_max, ...] whose trailing dimensions form
    one token's entry (contiguous, any dtype); path_nodes [B, N] int32.
    Returns row_status [B] int32.
    """
    dev = kv.device
    if not kv.is_contiguous() or kv.dim() < 3:
        raise ValueError("kv must be a contiguous [planes, B, S_max, ...] tensor")
    for t, n in ((kv_len_in, "kv_len_in"), (accepted_len, "accepted_len"),
                 (path_nodes, "path_nodes")):
        _req(t, n, dev, torch.int32)
    planes, B, S_max = kv.shape[:3]
    E = kv[0, 0, 0].numel() * kv.element_size() if kv.numel() else 0
    status = torch.empty(B, dtype=torch.int32, device=dev)
    a = SpecKvCompactArgs(B, path_nodes.shape[1], planes, 0, S_max, E, B * S_max * E, S_max * E, E,
                          _ptr(kv), _ptr(kv_len_in), _ptr(accepted_len), _ptr(path_nodes))
    _, sp = _stream(dev, stream)
    _check(lib().spec_kv_compact_tree(_c.byref(a), _ptr(status), sp))
    return status


def spec_adaptive_tree_policy(accepted_len, depth, draft_top1, ema, zero_run, alpha=0.3,
                              divisor=1.0, shallow=(3, 4, 4), deep=(7, 1, 8), start=(3, 4, 4),
                              ema0=0.0, breaker=5, stream=None):
    """One policy step for B sequences (see spec_adaptive_tree_policy in
    include/specverify.h).  ema (float64) and zero_run (int32) are updated in
    place; returns shape [B, 3] int32 = (nsteps, top-k, ndt)."""
    dev = accepted_len.device
    for t, n, dt in ((accepted_len, "accepted_len", torch.int32), (depth, "depth", torch.int32),
                     (draft_top1, "draft_top1", torch.float32), (ema, "ema", torch.float64),
                     (zero_run, "zero_run", torch.int32)):
        _req(t, n, dev, dt)
    B = accepted_len.shape[0]
    shape = torch.empty(B, 3, dtype=torch.int32, device=dev)
    q = SpecAdaptiveParams(float(alpha), float(divisor), float(ema0), (_c.c_int32 * 3)(*shallow),
                           (_c.c_int32 * 3)(*deep), (_c.c_int32 * 3)(*start), int(breaker))
    _, sp = _stream(dev, stream)
    _check(lib().spec_adaptive_tree_policy(_c.byref(q), B, _ptr(accepted_len), _ptr(depth),
                                           _ptr(draft_top1), _ptr(ema), _ptr(zero_run),
                                           _ptr(shape), sp))
    return shape


def set_wait_timeout_ns(ns):
    lib().spec_set_wait_timeout_ns(int(ns))


def get_wait_timeout_ns():
    return lib().spec_get_wait_timeout_ns()


def debug_force_wait_timeout(on):
    lib().spec_debug_force_wait_timeout(1 if on else 0)
