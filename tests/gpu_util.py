"""Helpers of the GPU parity tests: numpy <-> CUDA marshalling and the band rule."""
import numpy as np
import torch

BAND = 1e-5  # decision margin below which fp32 and fp64 may legitimately disagree
PROB_ATOL = 1e-5


def cuda(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def host(d):
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in d.items()}


def run_chain(sv, inp, mode="stochastic", kappa=0.0, diagnostics=True, draft=True):
    g = sv.spec_verify_chain(cuda(inp["target"]), cuda(inp["draft"]) if draft else None,
                             cuda(inp["draft_tokens"]), cuda(inp.get("temperature")),
                             cuda(inp.get("u_accept")), cuda(inp.get("u_sample")), mode=mode,
                             margin_kappa=kappa, diagnostics=diagnostics)
    return host(g)


def compare_stochastic(g, o, band=BAND):
    """Per-sample parity under the band rule.  Returns the number of rows whose
    outputs differ while the oracle's smallest decision margin is below band;
    fails on any difference outside the band."""
    assert np.array_equal(g["row_status"], o["row_status"]), (g["row_status"], o["row_status"])
    ok = o["row_status"] == 0
    same = (g["accepted_len"] == o["accepted_len"]) & np.all(g["out_tokens"] == o["out_tokens"], axis=1)
    mism = ~same & ok
    outside = mism & (o["row_margin"] >= band)
    if outside.any():
        b = int(np.nonzero(outside)[0][0])
        raise AssertionError(
            f"{int(outside.sum())} rows differ outside the band; row {b}: gpu len "
            f"{g['accepted_len'][b]} toks {g['out_tokens'][b]} vs oracle len "
            f"{o['accepted_len'][b]} toks {o['out_tokens'][b]} margin {o['row_margin'][b]}")
    bad = ~ok
    assert np.all(g["accepted_len"][bad] == -1) and np.all(g["num_emitted"][bad] == 0)
    assert np.all(g["out_tokens"][bad] == -1)
    assert np.array_equal(g["num_emitted"][ok], g["accepted_len"][ok] + 1)
    if "p_at_draft" in g and g["p_at_draft"].size:
        np.testing.assert_allclose(g["p_at_draft"][ok], o["p_at_draft"][ok], atol=PROB_ATOL, rtol=0)
        np.testing.assert_allclose(g["q_at_draft"][ok], o["q_at_draft"][ok], atol=PROB_ATOL, rtol=0)
        # residual mass (reported at the stopping position) of rows that agree
        rows = same & ok
        np.testing.assert_allclose(g["resid_mass"][rows], o["resid_mass"][rows],
                                   atol=PROB_ATOL, rtol=0)
    return int(mism.sum())


def chain_via_abi(L, inp, ws, nbytes=None, diagnostics=True):
    """spec_verify_chain (stochastic) through the C ABI with the caller's
    workspace tensor `ws` (uint8, CUDA); returns host arrays."""
    import ctypes
    from speculative_decoding_verification_32_gb300._binding import (SPEC_BF16, SPEC_F32,
                                                                      SPEC_STOCHASTIC,
                                                                      SpecChainArgs, SpecChainOut)
    B, K1, V = inp["target"].shape
    K = K1 - 1
    dev = ws.device
    t = {k: cuda(inp.get(k)) for k in ("target", "draft", "draft_tokens", "temperature",
                                       "u_accept", "u_sample")}
    out = {k: torch.empty(B, dtype=torch.int32, device=dev)
           for k in ("accepted_len", "num_emitted", "row_status")}
    out["out_tokens"] = torch.empty(B, K1, dtype=torch.int32, device=dev)
    if diagnostics:
        for k in ("p_at_draft", "q_at_draft", "resid_mass"):
            out[k] = torch.empty(B, K, dtype=torch.float32, device=dev)

    def ptr(x):
        return None if x is None else ctypes.c_void_p(x.data_ptr())
    dt = SPEC_BF16 if inp["target"].dtype == np.uint16 else SPEC_F32
    a = SpecChainArgs(B, K, V, dt, SPEC_STOCHASTIC, 0.0, ptr(t["target"]), ptr(t["draft"]),
                      ptr(t["draft_tokens"]), ptr(t["temperature"]), ptr(t["u_accept"]),
                      ptr(t["u_sample"]))
    o = SpecChainOut(ptr(out["accepted_len"]), ptr(out["out_tokens"]), ptr(out["num_emitted"]),
                     ptr(out["row_status"]), ptr(out.get("p_at_draft")),
                     ptr(out.get("q_at_draft")), ptr(out.get("resid_mass")))
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ptr(ws),
                             ws.numel() if nbytes is None else nbytes, stream)
    assert rc == 0, L.spec_status_string(rc)
    return host(out)
