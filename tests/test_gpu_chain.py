"""GPU parity of spec_verify_chain against the fp64 oracle (needs a GB300).

Greedy and margin outputs must match bit for bit.  Stochastic outputs may
differ only in rows where the oracle's decision margin (|u - min(1, ratio)| or
the inverse-CDF boundary gap) is below 1e-5; p(y), q(y) and the residual mass
must agree within 1e-5 absolute.
"""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import chain_via_abi, compare_stochastic, cuda, host, run_chain
from tests.util import grid_chain_inputs, log_probs, within_sigma
from workloads import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch
    import speculative_decoding_verification_32_gb300 as m
    assert torch.cuda.is_available()
    return m


def oracle_chain(inp, mode=O.STOCHASTIC, kappa=0.0):
    return O.verify_chain(inp["target"], inp["draft"] if mode == O.STOCHASTIC else None,
                          inp["draft_tokens"], inp.get("temperature"), inp.get("u_accept"),
                          inp.get("u_sample"), mode=mode, kappa=kappa)


# ------------------------------------------------------------- workloads
@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c5"])
def test_stochastic_workloads(sv, name):
    inp = S.make(name)
    g = run_chain(sv, inp)
    o = oracle_chain(inp)
    n_band = compare_stochastic(g, o)
    assert n_band <= max(1, inp["draft_tokens"].shape[0] // 100)


@pytest.mark.parametrize("kappa", [0.0, 0.3, 1.0, 1e-30])
def test_greedy_c2(sv, kappa):
    inp = S.make("c2", greedy=True)
    g = run_chain(sv, inp, mode="greedy", kappa=kappa, draft=False)
    o = oracle_chain(inp, O.GREEDY, kappa)
    for k in ("accepted_len", "out_tokens", "num_emitted", "row_status"):
        assert np.array_equal(g[k], o[k]), k


def test_greedy_c3_sizes_with_temperature_margin(sv):
    inp = S.make("c3", greedy=True)
    inp["temperature"] = np.linspace(0.3, 1.5, inp["target"].shape[0]).astype(np.float32)
    g = run_chain(sv, inp, mode="greedy", kappa=0.3, draft=False)
    o = oracle_chain(inp, O.GREEDY, 0.3)
    for k in ("accepted_len", "out_tokens", "num_emitted", "row_status"):
        assert np.array_equal(g[k], o[k]), k


def test_greedy_ties_lowest_index(sv):
    rng = np.random.default_rng(2)
    B, K, V = 16, 3, 5000
    t = rng.integers(-4, 5, size=(B, K + 1, V)).astype(np.float32)  # heavy ties
    inp = dict(target=S.f32_to_bf16_bits(t), draft=None,
               draft_tokens=rng.integers(0, V, size=(B, K)).astype(np.int32))
    tv = S.as_float32(inp["target"])
    # make some drafts the first maximum and some a later tied maximum
    for b in range(B):
        for j in range(K):
            m = np.flatnonzero(tv[b, j] == tv[b, j].max())
            inp["draft_tokens"][b, j] = m[0] if (b + j) % 2 == 0 else m[-1]
    g = run_chain(sv, inp, mode="greedy", draft=False)
    o = oracle_chain(inp, O.GREEDY)
    assert np.array_equal(g["out_tokens"], o["out_tokens"])
    assert np.array_equal(g["accepted_len"], o["accepted_len"])


# ------------------------------------------------------------ page examples
@pytest.mark.parametrize("pq", [([0.6, 0.3, 0.1], [0.2, 0.5, 0.3]),
                                ([0.5, 0.3, 0.2], [0.2, 0.5, 0.3]),
                                ([0.1, 0.5, 0.4], [0.4, 0.3, 0.3])])
def test_exact_law_by_enumeration_on_gpu(sv, pq):
    """Draft, Verify, and Correct -- 'Three possible next tokens' and the
    [CRS] section 2 example: enumerating y and a uniform grid through the GPU
    path reproduces p exactly, and matches the oracle row for row."""
    p, q = pq
    inp, w = grid_chain_inputs([p], [q], p, n=60)
    g = run_chain(sv, inp)
    o = O.verify_chain(**inp)
    assert compare_stochastic(g, o) == 0
    law = np.bincount(g["out_tokens"][:, 0], weights=w, minlength=3)
    np.testing.assert_allclose(law, p, atol=1e-9)


def test_two_position_exact_law_on_gpu(sv):
    p0, q0 = [0.6, 0.3, 0.1], [0.2, 0.5, 0.3]
    p1, q1 = [0.5, 0.3, 0.2], [0.2, 0.5, 0.3]
    inp, w = grid_chain_inputs([p0, p1], [q0, q1], [0.5, 0.3, 0.2], n=30)
    g = run_chain(sv, inp)
    o = O.verify_chain(**inp)
    assert compare_stochastic(g, o) == 0


def test_monte_carlo_200k_on_gpu(sv, golden):
    """[CRS] section 4 protocol through the GPU path."""
    g0 = golden("crs_abc_example.json")
    n = golden("crs_monte_carlo.json")["trials"]
    rng = np.random.default_rng(20260923)
    p, q = g0["p"], g0["q"]
    B = n
    tgt = np.broadcast_to(np.stack([log_probs(p), log_probs(p)]), (B, 2, 3)).astype(np.float32)
    drf = np.broadcast_to(log_probs(q)[None], (B, 1, 3)).astype(np.float32)
    inp = dict(target=tgt, draft=drf, draft_tokens=rng.choice(3, size=(B, 1), p=q).astype(np.int32),
               temperature=np.ones(B, np.float32), u_accept=rng.random((B, 1), dtype=np.float32),
               u_sample=rng.random((B, 2), dtype=np.float32))
    g = run_chain(sv, inp)
    freq = np.bincount(g["out_tokens"][:, 0], minlength=3) / n
    ok, z = within_sigma(freq, p, n)
    assert ok, z
    o = O.verify_chain(**inp)
    assert compare_stochastic(g, o) <= 5


def test_constant_alpha_on_gpu(sv):
    alpha, K, n = 0.7, 4, 200_000
    rng = np.random.default_rng(11)
    target = np.broadcast_to(log_probs([alpha, 1 - alpha]), (n, K + 1, 2)).astype(np.float32)
    draft = np.broadcast_to(log_probs([1.0, 0.0]), (n, K, 2)).astype(np.float32)
    inp = dict(target=target, draft=draft, draft_tokens=np.zeros((n, K), np.int32),
               temperature=None, u_accept=rng.random((n, K), dtype=np.float32),
               u_sample=rng.random((n, K + 1), dtype=np.float32))
    g = run_chain(sv, inp, diagnostics=False)
    L = g["accepted_len"]
    law = np.array([alpha ** i * (1 - alpha) for i in range(K)] + [alpha ** K])
    ok, z = within_sigma(np.bincount(L, minlength=K + 1) / n, law, n)
    assert ok, z
    rej = L < K
    assert np.all(g["out_tokens"][rej, L[rej]] == 1)
    assert abs(g["num_emitted"].mean() - O.expected_tokens(alpha, K)) < \
        3 * g["num_emitted"].std() / np.sqrt(n)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identical_laws_never_reject_on_gpu(sv, dtype):
    """p = q: the ratio is exactly 1, no residual branch is ever taken."""
    inp = S.chain_inputs(B=64, K=4, V=20000, dtype=dtype, seed=5, temperature=(0.3, 1.2))
    inp["draft"] = inp["target"][:, :4].copy()
    inp["u_accept"][:] = np.nextafter(np.float32(1), np.float32(0))
    g = run_chain(sv, inp)
    assert np.all(g["accepted_len"] == 4)
    assert np.all(g["resid_mass"] == 0)


# --------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [3, 37, 1001, 4099, 16384, 40000])
@pytest.mark.parametrize("K", [0, 1, 4])
def test_ragged_and_small_vocabularies(sv, dtype, V, K):
    """Vocabularies that span several slices with a ragged tail, rows that are
    not 16-byte aligned (direct-load path), K = 0 (bonus only)."""
    inp = S.chain_inputs(B=6, K=K, V=V, dtype=dtype, sigma=2.0, seed=V + K, temperature=(0.5, 1.5))
    g = run_chain(sv, inp)
    o = oracle_chain(inp)
    compare_stochastic(g, o)
    gg = run_chain(sv, inp, mode="greedy", kappa=0.2, draft=False)
    og = oracle_chain(inp, O.GREEDY, 0.2)
    assert np.array_equal(gg["out_tokens"], og["out_tokens"])


def test_masked_draft_entries(sv):
    """q = 0 tokens come only through the residual ([DVC] 'Try it')."""
    inp = S.make("c5", B=32, V=30000)
    g = run_chain(sv, inp)
    o = oracle_chain(inp)
    compare_stochastic(g, o)
    dv = S.as_float32(inp["draft"])
    for b in range(32):
        for j in range(g["accepted_len"][b]):
            assert np.isfinite(dv[b, j, g["out_tokens"][b, j]])


def test_row_status_codes_on_gpu(sv):
    inp = S.make("c1")
    B = 8
    r = lambda a: np.repeat(a, B, 0).copy()  # noqa: E731
    inp = dict(target=r(inp["target"]), draft=r(inp["draft"]), draft_tokens=r(inp["draft_tokens"]),
               temperature=np.ones(B, np.float32), u_accept=r(inp["u_accept"]),
               u_sample=r(inp["u_sample"]))
    inp["target"][1, 2, 3] = np.nan
    inp["draft"][2, 0, 5] = np.inf
    inp["draft_tokens"][3, 1] = 32
    inp["u_accept"][4, 0] = 1.0
    inp["temperature"][5] = 0.0
    inp["target"][6, 4, :] = -np.inf
    inp["u_sample"][7, 4] = -0.5
    g = run_chain(sv, inp)
    o = oracle_chain(inp)
    assert list(o["row_status"]) == [0, 1, 1, 2, 3, 7, 5, 3]
    compare_stochastic(g, o)
    gg = run_chain(sv, inp, mode="greedy", draft=False)
    og = oracle_chain(inp, O.GREEDY)
    assert np.array_equal(gg["row_status"], og["row_status"])
    assert np.array_equal(gg["out_tokens"], og["out_tokens"])


def test_empty_batch(sv):
    inp = S.chain_inputs(B=0, K=3, V=100, dtype="bf16", seed=1)
    g = run_chain(sv, inp)
    assert g["accepted_len"].shape == (0,)


def test_workspace_reuse_is_clean(sv):
    """Each call leaves the workspace zero-filled: back-to-back calls agree."""
    inp = S.make("c2")
    a = run_chain(sv, inp)
    b = run_chain(sv, inp)
    for k in ("accepted_len", "out_tokens", "row_status"):
        assert np.array_equal(a[k], b[k])


def test_bounded_wait_gives_up_and_recovers(sv):
    """A wait on a barrier that nothing completes gives up after the limit,
    marks the rows SPEC_ROW_TIMEOUT, and leaves the context usable."""
    inp = S.make("c2")
    old = sv.get_wait_timeout_ns()
    try:
        sv.set_wait_timeout_ns(2_000_000)  # 2 ms
        sv.debug_force_wait_timeout(True)
        g = run_chain(sv, inp)
        assert np.all(g["row_status"] == 6)
        assert np.all(g["accepted_len"] == -1)
        # the truncated chain: the stream gives up the same way and the
        # selection kernel withholds its records
        B = inp["target"].shape[0]
        gt = run_trunc(sv, inp, np.full(B, 20, np.int32), np.full(B, 0.9, np.float32))
        assert np.all(gt["row_status"] == 6)
        # the greedy kernels stream with plain loads: no wait, nothing to give up
        t = S.make("c4", B=2, V=4096)
        gtr = sv.spec_verify_tree(cuda(t["target"]), cuda(t["parent"]), cuda(t["node_tokens"]))
        assert np.all(host(gtr)["row_status"] == 0)
    finally:
        sv.debug_force_wait_timeout(False)
        sv.set_wait_timeout_ns(old)
    g = run_chain(sv, inp)
    compare_stochastic(g, oracle_chain(inp))


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_workspace_first_use_and_reuse(sv, name):
    """Any workspace works, whatever it holds on its first call (zero-filled
    or arbitrary contents, including a generation word about to wrap to 0).
    Each call advances the generation word in the
    header (the second 4-byte word of the last 16 bytes of the size given,
    kept 16-byte aligned when that size is not a multiple of 16) and every
    call matches the oracle."""
    import torch
    from speculative_decoding_verification_32_gb300 import _binding as Bn
    L = Bn.lib()
    inp = S.make(name)
    o = oracle_chain(inp)
    B, K1, V = inp["target"].shape
    need = L.spec_verify_chain_workspace_size(B, K1 - 1, V)
    for fill, extra in ((0, 0), (0xA5, 40), (0xFF, 7)):
        ws = torch.full((need + extra,), fill, dtype=torch.uint8, device="cuda")
        end = (need + extra) // 16 * 16
        gen = int(ws[end - 12:end - 8].cpu().numpy().view(np.uint32)[0])
        for call in range(3):
            g = chain_via_abi(L, inp, ws)
            compare_stochastic(g, o)
            now = int(ws[end - 12:end - 8].cpu().numpy().view(np.uint32)[0])
            # the generation skips 0, so zero-filled memory never carries a
            # current stamp
            assert now == ((gen + 1) % (1 << 32) or 1), (fill, call, gen, now)
            gen = now


def test_workspace_shared_across_shapes(sv):
    """One workspace serves calls of different shapes in turn: their records
    sit at different offsets, and only the generation stamp keeps a call from
    reading what an earlier call of another shape left there."""
    import torch
    from speculative_decoding_verification_32_gb300 import _binding as Bn
    L = Bn.lib()
    shapes = [("c2", {}), ("chain", dict(B=6, K=1, V=4099)), ("c2", dict(B=3)),
              ("chain", dict(B=8, K=3, V=20000)), ("c2", {}), ("chain", dict(B=6, K=1, V=4099))]
    cases = []
    for name, kw in shapes:
        if name == "chain":
            inp = S.chain_inputs(dtype="bf16", sigma=2.0, seed=kw["V"] + kw["K"], temperature=(0.7, 1.3), **kw)
        else:
            inp = S.make(name, **kw)
        cases.append(inp)
    need = max(L.spec_verify_chain_workspace_size(i["target"].shape[0], i["target"].shape[1] - 1,
                                                  i["target"].shape[2]) for i in cases)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    for inp in cases:
        compare_stochastic(chain_via_abi(L, inp, ws), oracle_chain(inp))


def test_truncated_drift_and_plain_share_one_workspace(sv):
    """Truncated, DRIFT and plain calls of different shapes in turn on the
    binding's one cached workspace (the largest shape comes first, so the
    buffer is not reallocated): the truncation kernel's stamped records and
    the DRIFT kernel's position flags sit at shape-dependent offsets, and only
    the generation stamp keeps a call from taking another call's.  K = 0 (a
    bonus-only truncated call) is among them."""
    rng = np.random.default_rng(91)
    shapes = [(8, 3, 20000), (6, 0, 4099), (5, 2, 7000), (8, 3, 20000), (6, 0, 4099)]
    for i, (B, K, V) in enumerate(shapes):
        inp = S.chain_inputs(B=B, K=K, V=V, dtype="bf16", sigma=3.0, seed=V + K, temperature=(0.7, 1.3),
                             peaks=5, peak_boost=6.0)
        k = rng.choice([0, 1, 20, 50, V], B).astype(np.int32)
        p = rng.choice([1.0, 0.5, 0.9], B).astype(np.float32)
        g = run_trunc(sv, inp, k, p)
        o = O.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], inp.get("temperature"),
                           inp["u_accept"], inp["u_sample"], top_k=k, top_p=p)
        assert compare_stochastic(g, o) <= 1
        if K > 0:  # DRIFT on the same shape, then a plain verify
            sup, res, st = (x.cpu().numpy() for x in sv.spec_drift_residuals(
                cuda(inp["target"]), cuda(inp["draft"]), cuda(inp["temperature"]), m=16))
            osup, ores, ost = O.drift_residuals(inp["target"], inp["draft"], inp["temperature"], m=16)
            assert np.array_equal(st, ost)
            assert np.array_equal(sup, osup)
            np.testing.assert_allclose(res, ores, rtol=0, atol=2e-4)
            compare_stochastic(run_chain(sv, inp), oracle_chain(inp))


# ------------------------------------------------------ top-k / top-p truncation
def _trunc_params(rng, B, V):
    k = rng.choice([0, 1, 2, 20, 50, 1000, V], B).astype(np.int32)
    p = rng.choice([1.0, 0.5, 0.8, 0.9, 0.99], B).astype(np.float32)
    return k, p


def run_trunc(sv, inp, k, p):
    g = sv.spec_verify_chain(cuda(inp["target"]), cuda(inp["draft"]), cuda(inp["draft_tokens"]),
                             cuda(inp.get("temperature")), cuda(inp.get("u_accept")),
                             cuda(inp.get("u_sample")), diagnostics=True, top_k=cuda(k),
                             top_p=cuda(p))
    return host(g)


@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
def test_truncated_workloads(sv, name):
    inp = S.make(name, B=48) if name == "c5" else S.make(name)
    B, _, V = inp["target"].shape
    k, p = _trunc_params(np.random.default_rng(len(name) + B), B, V)
    # draft tokens drawn from the untruncated q may fall outside q's kept set:
    # both sides then take q'(y) = 0 (accept iff p'(y) > 0)
    g = run_trunc(sv, inp, k, p)
    o = O.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], inp.get("temperature"),
                       inp["u_accept"], inp["u_sample"], top_k=k, top_p=p)
    n_band = compare_stochastic(g, o)
    assert n_band <= max(1, B // 50)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_truncated_flat_rows_ties_and_fp32(sv, dtype):
    """Flat rows (the nucleus spans most of the vocabulary: the whole-row
    search), rows of ties at the top-k boundary, and small vocabularies."""
    rng = np.random.default_rng(21)
    B, K, V = 12, 3, 3000
    t = rng.normal(0, 0.05, (B, K + 1, V)).astype(np.float32)   # nearly flat
    t[:4] = rng.normal(0, 3, (4, K + 1, V)).astype(np.float32)  # peaked rows
    t[4:6, :, :40] = 2.0                                        # 40-way ties at the top
    d = (t[:, :K] + rng.normal(0, 0.5, (B, K, V))).astype(np.float32)
    if dtype == "bf16":
        t, d = S.f32_to_bf16_bits(t), S.f32_to_bf16_bits(d)
    toks = rng.integers(0, V, (B, K)).astype(np.int32)
    inp = dict(target=t, draft=d, draft_tokens=toks,
               temperature=np.full(B, 0.9, np.float32),
               u_accept=rng.random((B, K), dtype=np.float32),
               u_sample=rng.random((B, K + 1), dtype=np.float32))
    k = np.array([0, 5, 50, 0, 20, 41, 0, 10, 0, 2999, 1, 0], np.int32)
    p = np.array([0.9, 1, 0.7, 0.3, 1, 0.95, 0.9, 0.5, 0.99, 0.8, 1, 0.6], np.float32)
    g = run_trunc(sv, inp, k, p)
    o = O.verify_chain(t, d, toks, inp["temperature"], inp["u_accept"], inp["u_sample"],
                       top_k=k, top_p=p)
    assert compare_stochastic(g, o) <= 1


def test_back_to_back_calls_of_every_mode_without_a_sync(sv):
    """Plain, DRIFT, truncated, greedy, tree and plain calls enqueued on one
    stream with no host synchronisation between them, then checked against
    the oracle.  Each call's first kernel may be scheduled while the previous
    call's last one still runs (programmatic dependent launch), so this is
    where a call could read its inputs, the workspace's generation or another
    call's records too early."""
    import torch
    rng = np.random.default_rng(2027)
    plain = S.make("c2")
    deep = S.chain_inputs(B=12, K=4, V=30000, dtype="bf16", sigma=3.0, seed=77, temperature=(0.7, 1.3))
    tree = S.make("c4", B=4, V=4096)
    k, p = _trunc_params(rng, 12, 30000)
    dev_inp = {n: {key: cuda(v) for key, v in d.items() if isinstance(v, np.ndarray)}
               for n, d in (("plain", plain), ("deep", deep), ("tree", tree))}
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        a, d = dev_inp["plain"], dev_inp["deep"]
        outs = []
        for _ in range(2):
            outs.append(("plain", sv.spec_verify_chain(a["target"], a["draft"], a["draft_tokens"],
                                                       a["temperature"], a["u_accept"], a["u_sample"],
                                                       stream=s)))
            outs.append(("drift", sv.spec_drift_residuals(d["target"], d["draft"], d["temperature"],
                                                          m=16, stream=s)))
            outs.append(("trunc", sv.spec_verify_chain(d["target"], d["draft"], d["draft_tokens"],
                                                       d["temperature"], d["u_accept"], d["u_sample"],
                                                       top_k=cuda(k), top_p=cuda(p), stream=s)))
            outs.append(("greedy", sv.spec_verify_chain(a["target"], None, a["draft_tokens"],
                                                        mode="greedy", margin_kappa=0.3, stream=s)))
            t = dev_inp["tree"]
            outs.append(("tree", sv.spec_verify_tree(t["target"], t["parent"], t["node_tokens"],
                                                     margin_kappa=tree["kappa"], stream=s)))
            outs.append(("deep", sv.spec_verify_chain(d["target"], d["draft"], d["draft_tokens"],
                                                      d["temperature"], d["u_accept"], d["u_sample"],
                                                      stream=s)))
    s.synchronize()
    want = {
        "plain": oracle_chain(plain),
        "deep": oracle_chain(deep),
        "greedy": O.verify_chain(plain["target"], None, plain["draft_tokens"], mode=O.GREEDY, kappa=0.3),
        "trunc": O.verify_chain(deep["target"], deep["draft"], deep["draft_tokens"], deep["temperature"],
                                deep["u_accept"], deep["u_sample"], top_k=k, top_p=p),
        "drift": O.drift_residuals(deep["target"], deep["draft"], deep["temperature"], m=16),
        "tree": O.verify_tree(tree["target"], tree["parent"], tree["node_tokens"], kappa=tree["kappa"]),
    }
    for name, g in outs:
        o = want[name]
        if name == "drift":
            sup, res, st = (x.cpu().numpy() for x in g)
            assert np.array_equal(st, o[2]) and np.array_equal(sup, o[0])
            np.testing.assert_allclose(res, o[1], rtol=0, atol=2e-4)
        elif name == "tree":
            h = host(g)
            assert np.array_equal(h["path_nodes"], o["path_nodes"])
            assert np.array_equal(h["out_tokens"], o["out_tokens"])
        elif name == "greedy":
            h = host(g)
            assert np.array_equal(h["out_tokens"], o["out_tokens"])
            assert np.array_equal(h["accepted_len"], o["accepted_len"])
        else:
            assert compare_stochastic(host(g), o) <= 1
