"""spec_verify_chain_static -- the chain verifier with the library's built-in
scratch buffer -- against spec_verify_chain with a caller workspace, both
called through the C ABI.

The file name sorts last so that, in a full run, these calls come after every
other test of the process; the GPU test must also pass alone in a fresh
process, where its first call does the per-device set-up.
"""
import ctypes

import numpy as np
import pytest

from tests.gpu_util import PROB_ATOL, cuda
from workloads import synthetic as S

SPEC_ERR_NULL, SPEC_ERR_SHAPE, SPEC_ERR_STATIC_LIMIT = 1, 2, 8
INT_OUT = ("accepted_len", "out_tokens", "num_emitted", "row_status")
F32_OUT = ("p_at_draft", "q_at_draft", "resid_mass")


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verification_32_gb300 import _binding
    from speculative_decoding_verification_32_gb300 import build as lib_build

    lib_build.build()
    return _binding.lib()


# ------------------------------------------------------------- host checks
def test_static_rejects_on_host(L):
    """Bad or oversized problems are refused before any CUDA call."""
    from speculative_decoding_verification_32_gb300._binding import SpecChainArgs, SpecChainOut
    p = ctypes.c_void_p(0x10000000)
    o = SpecChainOut(p, p, p, p, None, None, None)
    assert L.spec_verify_chain_static(None, ctypes.byref(o), None) == SPEC_ERR_NULL
    a = SpecChainArgs(4, 5, 0, 1, 0, 0.0, p, p, p, None, p, p)
    assert L.spec_verify_chain_static(ctypes.byref(a), ctypes.byref(o), None) == SPEC_ERR_SHAPE
    # B = 4096 chains of 8 drafts over 128256 tokens need far more than 4 MiB
    a = SpecChainArgs(4096, 8, 128256, 1, 0, 0.0, p, p, p, None, p, p)
    assert L.spec_verify_chain_workspace_size(4096, 8, 128256) > 4 << 20
    assert L.spec_verify_chain_static(ctypes.byref(a), ctypes.byref(o), None) == SPEC_ERR_STATIC_LIMIT
    assert L.spec_status_string(SPEC_ERR_STATIC_LIMIT).decode().startswith("SPEC_ERR_STATIC_LIMIT")
    # the stated example fits
    assert L.spec_verify_chain_workspace_size(256, 8, 128256) <= 4 << 20


# ------------------------------------------------------------ GPU parity
def _marshal(inp, greedy, dev):
    import torch
    from speculative_decoding_verification_32_gb300._binding import (SPEC_BF16, SPEC_F32,
                                                                      SPEC_GREEDY, SPEC_STOCHASTIC,
                                                                      SpecChainArgs, SpecChainOut)
    B, K1, V = inp["target"].shape
    K = K1 - 1
    t = {k: cuda(inp.get(k)) for k in ("target", "draft", "draft_tokens", "temperature",
                                       "u_accept", "u_sample")}
    dt = SPEC_BF16 if inp["target"].dtype == np.uint16 else SPEC_F32

    def ptr(x):
        return None if x is None else ctypes.c_void_p(x.data_ptr())

    def outputs():
        out = {k: torch.full((B,) if k != "out_tokens" else (B, K1), -7, dtype=torch.int32,
                             device=dev) for k in INT_OUT}
        if not greedy:
            for k in F32_OUT:
                out[k] = torch.full((B, K), -7.0, dtype=torch.float32, device=dev)
        o = SpecChainOut(*(ptr(out.get(k)) for k in INT_OUT + F32_OUT))
        return out, o

    args = SpecChainArgs(B, K, V, dt, SPEC_GREEDY if greedy else SPEC_STOCHASTIC,
                         0.3 if greedy else 0.0, ptr(t["target"]),
                         None if greedy else ptr(t["draft"]), ptr(t["draft_tokens"]),
                         ptr(t["temperature"]), None if greedy else ptr(t["u_accept"]),
                         None if greedy else ptr(t["u_sample"]))
    return t, args, outputs


def _host(out):
    import torch
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.gpu
def test_static_matches_workspace_entry_point(L):
    import torch
    assert torch.cuda.is_available()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    # two stochastic calls in a row (the second reuses scratch the first
    # wrote, at a larger size), then a greedy call with the margin rule
    cases = [("c2", False), ("c3", False), ("c2", True)]
    for name, greedy in cases:
        inp = S.make(name, greedy=greedy) if greedy else S.make(name)
        keep, args, outputs = _marshal(inp, greedy, dev)
        B, K1, V = inp["target"].shape
        nbytes = L.spec_verify_chain_workspace_size(B, K1 - 1, V)
        assert 0 < nbytes <= 4 << 20
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        ref, o_ref = outputs()
        rc = L.spec_verify_chain(ctypes.byref(args), ctypes.byref(o_ref),
                                 ctypes.c_void_p(ws.data_ptr()), nbytes, stream)
        assert rc == 0, L.spec_status_string(rc)
        got, o_got = outputs()
        rc = L.spec_verify_chain_static(ctypes.byref(args), ctypes.byref(o_got), stream)
        assert rc == 0, L.spec_status_string(rc)
        r, g = _host(ref), _host(got)
        for k in INT_OUT:
            assert np.array_equal(g[k], r[k]), (name, greedy, k)
        assert np.all(g["num_emitted"] >= 1), (name, greedy)
        if not greedy:
            for k in F32_OUT:
                np.testing.assert_allclose(g[k], r[k], atol=PROB_ATOL, rtol=0,
                                           err_msg=f"{name} {k}")
        del keep


@pytest.mark.gpu
def test_static_oversize_launches_nothing(L):
    import torch
    from speculative_decoding_verification_32_gb300._binding import SpecChainArgs, SpecChainOut
    dev = torch.device("cuda", torch.cuda.current_device())
    sentinel = torch.full((8,), -7, dtype=torch.int32, device=dev)
    p = ctypes.c_void_p(sentinel.data_ptr())
    a = SpecChainArgs(4096, 8, 128256, 1, 0, 0.0, p, p, p, None, p, p)
    o = SpecChainOut(p, p, p, p, None, None, None)
    rc = L.spec_verify_chain_static(ctypes.byref(a), ctypes.byref(o),
                                    ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert rc == SPEC_ERR_STATIC_LIMIT
    torch.cuda.synchronize()
    assert torch.all(sentinel == -7).item()
