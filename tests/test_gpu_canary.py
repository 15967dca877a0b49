"""Guard-region (canary) checks of every entry point's writes (needs a GB300).

Every case runs twice: through the library, and through its bounds-check
copy (-DSV_BOUNDS), whose kernels check each computed index before the access
and must record no bad one.

compute-sanitizer is closed on this machine, so out-of-bounds writes are caught
the old way: every buffer a call receives -- inputs, outputs, workspace --
is carved out of a larger allocation whose head and tail are filled with a
sentinel byte.  After each call the sentinels must be intact and the inputs
unchanged.  The shapes are odd on purpose: vocabularies of 1, 3, 4099 and
40000 tokens (rows that are not 16-byte aligned take the element-load paths,
a ragged last slice), 0, 1 and 63 drafts, tiny trees and a tree of 64 nodes.
The arithmetic itself is checked elsewhere; here only the row statuses are
asserted, so that the calls are known to have done their work.
"""
import ctypes

import numpy as np
import pytest

from workloads import synthetic as S

pytestmark = pytest.mark.gpu

GUARD = 4096      # sentinel bytes before and after every buffer
SENTINEL = 0xCD


class Arena:
    """Device buffers, each inside a larger allocation with sentinel guards."""

    def __init__(self):
        import torch
        self.torch = torch
        self.items = []  # (name, whole allocation, nbytes, copy of an input or None)

    def put(self, name, shape, dtype, data=None, writable=False):
        """A buffer of `shape` / `dtype`, holding `data` if given; the content
        of an input (data given, not writable) must survive the call."""
        torch = self.torch
        shape = tuple(int(s) for s in shape)
        item = np.dtype(dtype).itemsize
        nbytes = int(np.prod(shape)) * item if shape else item
        whole = torch.full((GUARD + ((nbytes + 255) // 256) * 256 + GUARD,), SENTINEL,
                           dtype=torch.uint8, device="cuda")
        view = whole[GUARD:GUARD + nbytes]
        keep = None
        if data is not None:
            host = np.ascontiguousarray(data).view(np.uint8).reshape(-1)
            assert host.size == nbytes, (name, host.size, nbytes)
            view.copy_(torch.from_numpy(host.copy()).cuda())
            keep = None if writable else host.copy()
        self.items.append((name, whole, nbytes, keep))
        return view

    @staticmethod
    def ptr(view):
        return None if view is None else ctypes.c_void_p(view.data_ptr())

    def check(self):
        self.torch.cuda.synchronize()
        for name, whole, nbytes, keep in self.items:
            h = whole.cpu().numpy()
            head, tail = h[:GUARD], h[GUARD + nbytes:]
            assert np.all(head == SENTINEL), f"{name}: bytes before the buffer were written"
            assert np.all(tail == SENTINEL), f"{name}: bytes after the buffer were written"
            if keep is not None:
                assert np.array_equal(h[GUARD:GUARD + nbytes], keep), f"input {name} was modified"

    def host(self, view, dtype, shape):
        self.torch.cuda.synchronize()
        return view.cpu().numpy().view(dtype).reshape(shape)


class BoundsChecked:
    """The bounds-check copy of the library (built with -DSV_BOUNDS): after
    every call, the kernels' record of bad indexes must be empty."""

    def __init__(self, lib):
        self._lib = lib
        lib.spec_debug_bounds.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_uint)]
        lib.spec_debug_bounds.restype = ctypes.c_int
        lib.spec_debug_bounds_selftest.argtypes = [ctypes.c_void_p]
        lib.spec_debug_bounds_selftest.restype = ctypes.c_int

    def record(self):
        import torch
        torch.cuda.synchronize()
        count, line = ctypes.c_uint(0), ctypes.c_uint(0)
        assert self._lib.spec_debug_bounds(ctypes.byref(count), ctypes.byref(line)) == 0
        return count.value, line.value

    def __getattr__(self, name):
        fn = getattr(self._lib, name)
        if not name.startswith(("spec_verify", "spec_rollback", "spec_kv", "spec_adaptive", "spec_drift")):
            return fn

        def checked(*args):
            rc = fn(*args)
            count, line = self.record()
            assert count == 0, f"{name}: {count} bad indexes, the first at source line {line}"
            return rc
        return checked


@pytest.fixture(scope="module", params=["default", "bounds"])
def L(request):
    """Each case runs through the library and through its bounds-check copy."""
    import torch
    import speculative_decoding_verification_32_gb300 as sv
    from speculative_decoding_verification_32_gb300 import _binding
    from speculative_decoding_verification_32_gb300 import build as lib_build
    assert torch.cuda.is_available()
    if request.param == "default":
        return sv.lib()
    return BoundsChecked(_binding._bind(ctypes.CDLL(lib_build.build(variant="bounds"))))


def test_bounds_record_sees_a_failed_check():
    """The checker's own check: the self-test kernel tests an index of 5
    against an extent of 3 (touching no memory), which must be recorded."""
    import torch
    from speculative_decoding_verification_32_gb300 import _binding
    from speculative_decoding_verification_32_gb300 import build as lib_build
    B = BoundsChecked(_binding._bind(ctypes.CDLL(lib_build.build(variant="bounds"))))
    B.record()  # clears what earlier calls left
    assert B.spec_debug_bounds_selftest(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    count, line = B.record()
    assert count == 1 and line > 0
    assert B.record() == (0, 0)  # read and cleared


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _logit_dtype(a):
    return np.uint16 if a.dtype == np.uint16 else np.float32


def _chain_case(L, A, inp, mode, static=False, trunc=None):
    from speculative_decoding_verification_32_gb300._binding import (
        SPEC_BF16, SPEC_F32, SpecChainArgs, SpecChainOut, SpecTruncation)
    B, K1, V = inp["target"].shape
    K = K1 - 1
    greedy = mode == 1
    dt = SPEC_BF16 if inp["target"].dtype == np.uint16 else SPEC_F32
    ldt = _logit_dtype(inp["target"])
    tgt = A.put("target", (B, K1, V), ldt, inp["target"])
    drf = None if greedy else A.put("draft", (B, K, V), ldt, inp["draft"])
    tok = A.put("draft_tokens", (B, K), np.int32, inp["draft_tokens"])
    tmp = A.put("temperature", (B,), np.float32, inp["temperature"])
    ua = None if greedy else A.put("u_accept", (B, K), np.float32, inp["u_accept"])
    us = None if greedy else A.put("u_sample", (B, K1), np.float32, inp["u_sample"])
    acc = A.put("accepted_len", (B,), np.int32)
    out = A.put("out_tokens", (B, K1), np.int32)
    nem = A.put("num_emitted", (B,), np.int32)
    st = A.put("row_status", (B,), np.int32)
    diag = [None, None, None] if greedy else [A.put(n, (B, K), np.float32)
                                              for n in ("p_at_draft", "q_at_draft", "resid_mass")]
    p = A.ptr
    a = SpecChainArgs(B, K, V, dt, mode, 0.3 if greedy else 0.0, p(tgt), p(drf), p(tok), p(tmp),
                      p(ua), p(us))
    o = SpecChainOut(p(acc), p(out), p(nem), p(st), *[p(x) for x in diag])
    if static:
        rc = L.spec_verify_chain_static(ctypes.byref(a), ctypes.byref(o), _stream())
    else:
        nb = (L.spec_verify_chain_workspace_size if trunc is None
              else L.spec_verify_chain_truncated_workspace_size)(B, K, V)
        ws = A.put("workspace", (nb,), np.uint8)
        if trunc is not None:
            tk = A.put("top_k", (B,), np.int32, trunc[0])
            tp = A.put("top_p", (B,), np.float32, trunc[1])
            t = SpecTruncation(p(tk), p(tp))
            rc = L.spec_verify_chain_truncated(ctypes.byref(a), ctypes.byref(t), ctypes.byref(o),
                                               p(ws), nb, _stream())
        else:
            rc = L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), p(ws), nb, _stream())
    assert rc == 0, L.spec_status_string(rc)
    A.check()
    status = A.host(st, np.int32, (B,))
    assert np.all(status == 0), status
    return A.host(acc, np.int32, (B,)), A.host(out, np.int32, (B, K1))


CHAIN_SHAPES = [(V, K) for V in (1, 3, 4099, 40000) for K in (0, 1, 63)]


@pytest.mark.parametrize("V,K", CHAIN_SHAPES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chain_writes_stay_in_bounds(L, V, K, dtype):
    inp = S.chain_inputs(B=3, K=K, V=V, dtype=dtype, sigma=2.0, seed=7 * V + K,
                         temperature=(0.5, 1.5))
    for mode in (0, 1):
        _chain_case(L, Arena(), inp, mode)
    if V > 1:  # top-k / top-p need a vocabulary to cut
        trunc = (np.array([2, 0, V], np.int32), np.array([0.9, 0.5, 1.0], np.float32))
        _chain_case(L, Arena(), inp, 0, trunc=trunc)


@pytest.mark.parametrize("V,K", [(4099, 1), (40000, 63), (3, 0)])
def test_static_entry_point_writes_stay_in_bounds(L, V, K):
    inp = S.chain_inputs(B=3, K=K, V=V, dtype="bf16", sigma=2.0, seed=V + K, temperature=(0.5, 1.5))
    _chain_case(L, Arena(), inp, 0, static=True)


@pytest.mark.parametrize("N,V", [(1, 3), (2, 2), (7, 4099), (64, 40000)])
def test_tree_and_kv_compaction_write_in_bounds(L, N, V):
    from speculative_decoding_verification_32_gb300._binding import (
        SPEC_BF16, SpecKvCompactArgs, SpecTreeArgs, SpecTreeOut)
    inp = S.tree_inputs(B=3, N=N, V=V, dtype="bf16", max_depth=min(6, max(1, N - 1)),
                        branch=(1, 3), seed=N * 131 + V)
    A = Arena()
    B = 3
    tgt = A.put("target", (B, N, V), np.uint16, inp["target"])
    par = A.put("parent", (B, N), np.int32, inp["parent"])
    tok = A.put("node_tokens", (B, N), np.int32, inp["node_tokens"])
    acc = A.put("accepted_len", (B,), np.int32)
    path = A.put("path_nodes", (B, N), np.int32)
    out = A.put("out_tokens", (B, N), np.int32)
    nem = A.put("num_emitted", (B,), np.int32)
    st = A.put("row_status", (B,), np.int32)
    nb = L.spec_verify_tree_workspace_size(B, N, V)
    ws = A.put("workspace", (nb,), np.uint8)
    p = A.ptr
    a = SpecTreeArgs(B, N, V, SPEC_BF16, 0.3, p(tgt), p(par), p(tok), None)
    o = SpecTreeOut(p(acc), p(path), p(out), p(nem), p(st))
    rc = L.spec_verify_tree(ctypes.byref(a), ctypes.byref(o), p(ws), nb, _stream())
    assert rc == 0, L.spec_status_string(rc)
    A.check()
    assert np.all(A.host(st, np.int32, (B,)) == 0)
    # compact a small cache along the verified paths: 2 planes, 48-byte entries
    S_max, E, planes = N + 5, 48, 2
    kvl = A.put("kv_len_in", (B,), np.int32, np.array([0, 3, 5], np.int32))
    rng = np.random.default_rng(N)
    cache = A.put("kv", (planes, B, S_max, E), np.uint8,
                  rng.integers(0, 255, (planes, B, S_max, E), dtype=np.uint8), writable=True)
    st2 = A.put("kv_row_status", (B,), np.int32)
    k = SpecKvCompactArgs(B, N, planes, 0, S_max, E, B * S_max * E, S_max * E, E, p(cache),
                          p(kvl), p(acc), p(path))
    rc = L.spec_kv_compact_tree(ctypes.byref(k), p(st2), _stream())
    assert rc == 0, L.spec_status_string(rc)
    A.check()
    assert np.all(A.host(st2, np.int32, (B,)) == 0)


def test_rollback_and_policy_write_in_bounds(L):
    from speculative_decoding_verification_32_gb300._binding import SpecAdaptiveParams
    A = Arena()
    B, E = 5, 4
    rng = np.random.default_rng(1)
    acc_h = rng.integers(0, E, B).astype(np.int32)
    p = A.ptr
    kvl = A.put("kv_len_in", (B,), np.int32, rng.integers(10, 50, B).astype(np.int32))
    acc = A.put("accepted_len", (B,), np.int32, acc_h)
    nin = A.put("num_emitted_in", (B,), np.int32, acc_h + 1)
    toks = A.put("out_tokens", (B, E), np.int32, rng.integers(0, 9, (B, E)).astype(np.int32))
    mlen = A.put("max_len", (B,), np.int32, np.full(B, 60, np.int32))
    com = A.put("committed", (B,), np.int32)
    nout = A.put("num_emitted_out", (B,), np.int32)
    rc = L.spec_rollback_lengths(B, E, p(kvl), p(acc), p(nin), p(toks), 2, p(mlen), p(com), p(nout),
                                 _stream())
    assert rc == 0
    A.check()
    dep = A.put("depth", (B,), np.int32, np.full(B, E - 1, np.int32))
    top1 = A.put("draft_top1", (B,), np.float32, rng.random(B).astype(np.float32))
    ema = A.put("ema", (B,), np.float64, np.zeros(B), writable=True)
    zero = A.put("zero_run", (B,), np.int32, np.zeros(B, np.int32), writable=True)
    shape = A.put("shape", (B, 3), np.int32)
    q = SpecAdaptiveParams(0.3, 1.0, 0.5, (ctypes.c_int32 * 3)(3, 4, 4), (ctypes.c_int32 * 3)(7, 1, 8),
                           (ctypes.c_int32 * 3)(3, 4, 4), 5)
    rc = L.spec_adaptive_tree_policy(ctypes.byref(q), B, p(acc), p(dep), p(top1), p(ema), p(zero),
                                     p(shape), _stream())
    assert rc == 0
    A.check()


@pytest.mark.parametrize("V,K,m", [(3, 1, 3), (4099, 1, 32), (40000, 63, 64), (1, 2, 1)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_drift_writes_stay_in_bounds(L, V, K, m, dtype):
    from speculative_decoding_verification_32_gb300._binding import (SPEC_BF16, SPEC_F32,
                                                                      SpecChainArgs)
    inp = S.chain_inputs(B=3, K=K, V=V, dtype=dtype, sigma=2.0, seed=V * 3 + K, temperature=(0.5, 1.5))
    A = Arena()
    B = 3
    ldt = _logit_dtype(inp["target"])
    tgt = A.put("target", (B, K + 1, V), ldt, inp["target"])
    drf = A.put("draft", (B, K, V), ldt, inp["draft"])
    tmp = A.put("temperature", (B,), np.float32, inp["temperature"])
    sup = A.put("support", (B, K, m), np.int32)
    res = A.put("residual", (B, K, m), np.float32)
    st = A.put("row_status", (B,), np.int32)
    nb = L.spec_verify_chain_truncated_workspace_size(B, K, V)
    ws = A.put("workspace", (nb,), np.uint8)
    p = A.ptr
    dt = SPEC_BF16 if dtype == "bf16" else SPEC_F32
    a = SpecChainArgs(B, K, V, dt, 0, 0.0, p(tgt), p(drf), None, p(tmp), None, None)
    rc = L.spec_drift_residuals(ctypes.byref(a), m, p(sup), p(res), p(st), p(ws), nb, _stream())
    assert rc == 0, L.spec_status_string(rc)
    A.check()
    assert np.all(A.host(st, np.int32, (B,)) == 0)
