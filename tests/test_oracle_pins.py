"""Pins of the fp64 oracle to facts the pages and the mathematics fix (no GPU).

Each test names the page section it follows.  Worked-example numbers live in
tests/golden/*.json with their citation.
"""
import numpy as np
import pytest

from oracle import oracle as O
from tests.util import (grid_chain_inputs, log_probs, softmax64, within_sigma)
from workloads import synthetic as S


def _law_first_token(out, weights, V):
    return np.bincount(out["out_tokens"][:, 0], weights=weights, minlength=V)


def _single_position(p, q, y, u_acc, u_smp, p_bonus=None, T=1.0):
    """K = 1 inputs for rows with draft tokens y and uniforms u_acc, u_smp."""
    B = len(y)
    pb = p if p_bonus is None else p_bonus
    tgt = np.stack([log_probs(p) * np.float32(T), log_probs(pb) * np.float32(T)])
    drf = (log_probs(q) * np.float32(T))[None]
    return dict(target=np.broadcast_to(tgt, (B, 2, len(p))).astype(np.float32),
                draft=np.broadcast_to(drf, (B, 1, len(p))).astype(np.float32),
                draft_tokens=np.asarray(y, np.int32).reshape(B, 1),
                temperature=np.full(B, T, np.float32),
                u_accept=np.asarray(u_acc, np.float32).reshape(B, 1),
                u_sample=np.repeat(np.asarray(u_smp, np.float32).reshape(B, 1), 2, axis=1))


# --------------------------------------------------------------------- P1 / P2
@pytest.mark.parametrize("fixture", ["dvc_three_tokens.json", "crs_abc_example.json"])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_worked_example_acceptance_and_residual(golden, fixture, T):
    """Draft, Verify, and Correct -- 'Three possible next tokens'; why correcting a
    rejection is not resampling -- section 2: acceptance probabilities, accepted mass,
    rejection mass and the residual direction."""
    g = golden(fixture)
    p, q = np.array(g["p"]), np.array(g["q"])
    if "acceptance_probability" in g:
        acc_prob = g["acceptance_probability"]
    else:  # [CRS]: A always accepted, B in 60% of proposals, C with 2/3
        acc_prob = np.array(g["accepted_contribution"]) / q
    # one row per draft token, u_accept = 0.999999 forces the rejection branch
    # whenever min(1, ratio) < 1
    inp = _single_position(p, q, [0, 1, 2], [0.999999] * 3, [0.5] * 3, T=T)
    out = O.verify_chain(**inp)
    ratio = out["ratio"][:, 0]
    np.testing.assert_allclose(np.minimum(1.0, ratio), acc_prob, atol=1e-6)
    np.testing.assert_allclose(out["p_at_draft"][:, 0], p, atol=1e-6)
    np.testing.assert_allclose(out["q_at_draft"][:, 0], q, atol=1e-6)
    accepted_mass = q * np.minimum(1.0, ratio)
    total = g.get("accepted_total")
    np.testing.assert_allclose(accepted_mass.sum(), total, atol=1e-6)
    Z = g["rejection_mass_Z"] if "rejection_mass_Z" in g else 1.0 - total
    rejecting = ratio < 1
    np.testing.assert_allclose(out["resid_mass"][rejecting, 0], Z, atol=1e-6)
    assert np.all(out["resid_mass"][~rejecting, 0] == 0)
    # residual (1, 0, 0): every correction is token 0, whatever u_sample
    for s in [0.0, 0.3, 0.999]:
        inp = _single_position(p, q, [1, 2], [0.999999] * 2, [s] * 2, T=T)
        out = O.verify_chain(**inp)
        assert list(out["accepted_len"]) == [0, 0]
        assert list(out["out_tokens"][:, 0]) == [int(np.argmax(g["residual_normalised"]))] * 2


@pytest.mark.parametrize("fixture", ["dvc_three_tokens.json", "crs_abc_example.json"])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_worked_example_exact_law_by_enumeration(golden, fixture, T):
    """Why the correction recovers the target: accepted mass + Z * residual = p.
    Enumerating y and a midpoint grid of both uniforms (breakpoints 0.6, 1/3, 2/3
    are multiples of 1/30) gives the exact law of the emitted token."""
    g = golden(fixture)
    inp, w = grid_chain_inputs([g["p"]], [g["q"]], g["p"], n=30, temperature=T)
    out = O.verify_chain(**inp)
    law = _law_first_token(out, w, 3)
    np.testing.assert_allclose(law, g["p"], atol=1e-12)
    if "recovered_law" in g:
        np.testing.assert_allclose(law, g["recovered_law"], atol=1e-12)
    # probability that the draft survives = sum min(p, q)
    p_acc = w[out["accepted_len"] == 1].sum()
    np.testing.assert_allclose(p_acc, np.minimum(g["p"], g["q"]).sum(), atol=1e-12)
    # the same example with the token order reversed (residual mass on the last token)
    inp, w = grid_chain_inputs([g["p"][::-1]], [g["q"][::-1]], g["p"][::-1], n=30, temperature=T)
    law = _law_first_token(O.verify_chain(**inp), w, 3)
    np.testing.assert_allclose(law, g["p"][::-1], atol=1e-12)


def test_split_residual_exact_law():
    """Why the correction recovers the target, with the residual spread over two
    tokens: p = (0.1, 0.5, 0.4), q = (0.4, 0.3, 0.3), [p - q]_+ = (0, 0.2, 0.1).
    Breakpoints 0.25, 2/3 are multiples of 1/60, so the enumeration is exact."""
    p, q = [0.1, 0.5, 0.4], [0.4, 0.3, 0.3]
    inp, w = grid_chain_inputs([p], [q], p, n=60)
    out = O.verify_chain(**inp)
    np.testing.assert_allclose(_law_first_token(out, w, 3), p, atol=1e-12)
    rej = out["accepted_len"] == 0
    corr = np.bincount(out["out_tokens"][rej, 0], weights=w[rej], minlength=3) / w[rej].sum()
    np.testing.assert_allclose(corr, [0.0, 2 / 3, 1 / 3], atol=1e-12)


# ------------------------------------------------------------------------- P3
@pytest.mark.parametrize("fixture", ["dvc_three_tokens.json", "crs_abc_example.json"])
def test_monte_carlo_200k(golden, fixture):
    """Why correcting a rejection is not resampling -- section 4: 200,000 trials,
    every frequency within three standard errors of p."""
    mc = golden("crs_monte_carlo.json")
    g = golden(fixture)
    n = mc["trials"]
    rng = np.random.default_rng(20260923)
    y = rng.choice(3, size=n, p=g["q"])
    inp = _single_position(g["p"], g["q"], y, rng.random(n, dtype=np.float32),
                           rng.random(n, dtype=np.float32))
    out = O.verify_chain(**inp)
    freq = np.bincount(out["out_tokens"][:, 0], minlength=3) / n
    ok, z = within_sigma(freq, g["p"], n)
    assert ok, z
    # the page's standard-error scale for A: sqrt(0.5 * 0.5 / 200000) = 0.00112
    assert abs(np.sqrt(0.25 / n) - mc["page_reported_standard_error_for_A"]) < 5e-6


def test_monte_carlo_c1_vocabulary():
    """Monte Carlo on the V = 32 fp32 workload: the first emitted token follows the
    target law of position 0 (drafts redrawn from q for each trial)."""
    base = S.make("c1")
    n = 200_000
    rng = np.random.default_rng(7)
    V = base["target"].shape[-1]
    K = base["draft"].shape[1]
    tgt = np.broadcast_to(base["target"], (n,) + base["target"].shape[1:]).copy()
    drf = np.broadcast_to(base["draft"], (n,) + base["draft"].shape[1:]).copy()
    y = S.gumbel_max_tokens(drf.astype(np.float32), np.float32(1.0), rng)
    out = O.verify_chain(tgt, drf, y, np.ones(n, np.float32),
                         rng.random((n, K), dtype=np.float32),
                         rng.random((n, K + 1), dtype=np.float32))
    p0 = softmax64(base["target"][0, 0])
    freq = np.bincount(out["out_tokens"][:, 0], minlength=V) / n
    ok, z = within_sigma(freq, p0, n, k=4.0)  # 32 cells: 4 sigma keeps the family-wise rate low
    assert ok, z.max()


# ------------------------------------------------------------------------- P4
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identical_laws_never_reject(dtype):
    """Draft, Verify, and Correct -- 'Name the two distributions': if p = q
    acceptance is certain and the residual branch is never needed."""
    inp = S.chain_inputs(B=64, K=4, V=1000, dtype=dtype, sigma=3.0, seed=5,
                         temperature=(0.3, 1.2))
    out = O.verify_chain(inp["target"], inp["target"][:, :4].copy(), inp["draft_tokens"],
                         inp["temperature"], np.nextafter(np.float32(1), np.float32(0)) *
                         np.ones((64, 4), np.float32), inp["u_sample"])
    assert np.all(out["ratio"] == 1.0)
    assert np.all(out["accepted_len"] == 4)
    assert np.all(out["resid_mass"] == 0.0)


# ------------------------------------------------------------------------- P5
def test_constant_alpha_geometric_law():
    """Expected committed tokens 1 + a + ... + a^k (Draft, Verify, and Correct --
    'When is drafting worth it?'; why correcting ... -- section 6).  V = 2,
    q = (1, 0), p = (alpha, 1 - alpha) makes every acceptance independent with
    rate alpha; every rejection must emit token 1, which q never proposes."""
    alpha, K, n = 0.7, 4, 200_000
    rng = np.random.default_rng(11)
    tgt_row = log_probs([alpha, 1 - alpha])
    drf_row = log_probs([1.0, 0.0])
    target = np.broadcast_to(tgt_row, (n, K + 1, 2)).astype(np.float32)
    draft = np.broadcast_to(drf_row, (n, K, 2)).astype(np.float32)
    out = O.verify_chain(target, draft, np.zeros((n, K), np.int32), None,
                         rng.random((n, K), dtype=np.float32),
                         rng.random((n, K + 1), dtype=np.float32))
    L = out["accepted_len"]
    law = np.array([alpha ** i * (1 - alpha) for i in range(K)] + [alpha ** K])
    ok, z = within_sigma(np.bincount(L, minlength=K + 1) / n, law, n)
    assert ok, z
    E = O.expected_tokens(alpha, K)
    assert abs(E - (1 - alpha ** (K + 1)) / (1 - alpha)) < 1e-12
    sd = out["num_emitted"].std()
    assert abs(out["num_emitted"].mean() - E) < 3 * sd / np.sqrt(n)
    rejected = L < K
    assert np.all(out["out_tokens"][rejected, L[rejected]] == 1)


# ------------------------------------------------------------------------- P6
def test_cost_model_page_numbers(golden):
    """Why correcting a rejection is not resampling -- sections 6 and 7: the grid
    maximum at alpha = 0.7 and the g = 3 ratio."""
    g = golden("crs_cost_model.json")
    a = 0.7
    assert round(O.expected_tokens(a, 6), 6) == g["alpha_0.7_c_0.05"]["E"]
    for key, c in [("alpha_0.7_c_0.05", 0.05), ("alpha_0.7_c_0.20", 0.20)]:
        S_vals = [O.speedup(a, gm, c) for gm in range(1, 17)]
        best = int(np.argmax(S_vals)) + 1
        assert best == g[key]["best_gamma"]
        assert round(max(S_vals), 3) == g[key]["S"]
    assert round(O.speedup(a, 6, 0.05, g=3.0), 3) == g["alpha_0.7_gamma_6_c_0.05_g_3"]["S"]


# ------------------------------------------------------------------------- P7
@pytest.mark.parametrize("name,kw", [("c1", {}), ("c2", dict(B=8, V=3000)),
                                     ("c5", dict(B=16, V=2000))])
def test_stochastic_invariants(name, kw):
    """Every correction token has p > q; 1..K+1 tokens per cycle (why correcting
    ... -- section 5); masked draft entries (q = 0) are only reachable through the
    residual (Draft, Verify, and Correct -- 'Try it')."""
    inp = S.make(name, **kw)
    out = O.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], inp["temperature"],
                         inp["u_accept"], inp["u_sample"])
    B, K = inp["draft_tokens"].shape
    assert np.all(out["row_status"] == 0)
    assert np.all((out["num_emitted"] >= 1) & (out["num_emitted"] <= K + 1))
    assert np.all(out["num_emitted"] == out["accepted_len"] + 1)
    tv = S.as_float32(inp["target"])
    dv = S.as_float32(inp["draft"])
    for b in range(B):
        a = out["accepted_len"][b]
        assert list(out["out_tokens"][b, :a]) == list(inp["draft_tokens"][b, :a])
        assert np.all(out["out_tokens"][b, a + 1:] == -1)
        tok = out["out_tokens"][b, a]
        if a < K:
            T = inp["temperature"][b]
            p = softmax64(tv[b, a], T)
            q = softmax64(dv[b, a], T)
            assert p[tok] > q[tok]
        for j in range(a):
            assert np.isfinite(dv[b, j, out["out_tokens"][b, j]])


# ------------------------------------------------------------------------- P8
def test_greedy_is_argmax_walk():
    """How a Small Model Speeds Up a Big One -- 'The Guarantee Behind Rejection
    Sampling': greedy keeps a draft iff it is the target argmax (np.argmax: first
    maximum), and at the first mismatch emits the argmax."""
    inp = S.make("c2", greedy=True, V=4000)
    t = S.as_float32(inp["target"]).copy()
    # plant exact ties at the maximum to exercise the lowest-index rule
    t[0, 0, 10] = t[0, 0, 20] = t[0, 0].max() + 1
    inp["target"] = S.f32_to_bf16_bits(t)
    tv = S.as_float32(inp["target"])
    toks = inp["draft_tokens"].copy()
    toks[0, 0] = 10
    out = O.verify_chain(inp["target"], None, toks, mode=O.GREEDY)
    B, K = toks.shape
    for b in range(B):
        top = np.argmax(tv[b], axis=-1)
        a = next((j for j in range(K) if toks[b, j] != top[j]), K)
        assert out["accepted_len"][b] == a
        assert out["out_tokens"][b, a] == top[a]
    assert out["accepted_len"][0] >= 1


def test_margin_hand_example(golden):
    g = golden("margin_hand_example.json")
    for c in g["cases"]:
        B = 1
        target = np.array([[g["logits"], g["logits"]]], np.float32)
        out = O.verify_chain(target, None, np.array([[c["draft"]]], np.int32),
                             np.array([c["temperature"]], np.float32), mode=O.GREEDY,
                             kappa=g["kappa"])
        assert (out["accepted_len"][0] == 1) == c["promoted"], c
        # the ratio the rule compares, from the definition with fp64 softmax
        p = softmax64(g["logits"], c["temperature"])
        assert abs(p[c["draft"]] / p.max() - c["ratio"]) < 1e-12


def test_margin_special_cases():
    """kappa >= 1 reduces the margin rule to strict greedy; a tiny kappa promotes
    every finite draft (Margins, Not Windows -- section 3)."""
    inp = S.make("c2", V=4000)
    args = (inp["target"], None, inp["draft_tokens"], inp["temperature"])
    strict = O.verify_chain(*args, mode=O.GREEDY)
    for k in [1.0, 1.5]:
        o = O.verify_chain(*args, mode=O.GREEDY, kappa=k)
        assert np.array_equal(o["out_tokens"], strict["out_tokens"])
    o = O.verify_chain(*args, mode=O.GREEDY, kappa=1e-30)
    assert np.all(o["accepted_len"] == inp["draft_tokens"].shape[1])
    o = O.verify_chain(*args, mode=O.GREEDY, kappa=0.3)
    assert np.all(o["accepted_len"] >= strict["accepted_len"])


@pytest.mark.parametrize("kappa", [0.0, 0.3])
def test_tree_with_chain_parents_equals_chain(kappa):
    inp = S.make("c2", greedy=True, V=3000)
    B, K = inp["draft_tokens"].shape
    chain = O.verify_chain(inp["target"], None, inp["draft_tokens"], mode=O.GREEDY, kappa=kappa)
    parent = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    toks = np.concatenate([np.zeros((B, 1), np.int32), inp["draft_tokens"]], axis=1)
    tree = O.verify_tree(inp["target"], parent, toks, kappa=kappa)
    assert np.array_equal(tree["accepted_len"], chain["accepted_len"])
    assert np.array_equal(tree["out_tokens"], chain["out_tokens"])
    a = tree["accepted_len"]
    for b in range(B):
        assert list(tree["path_nodes"][b, :a[b]]) == list(range(1, a[b] + 1))


@pytest.mark.parametrize("kappa", [0.0, 0.05])
def test_tree_brute_force(kappa):
    """Brute force over root paths on small random trees: a node counts iff every
    node of its root path passes the argmax / margin test; the kept branch is the
    deepest such node, lowest index on ties."""
    rng = np.random.default_rng(3)
    B, N, V = 40, 12, 6
    target = rng.integers(-3, 3, size=(B, N, V)).astype(np.float32)  # many ties
    parent = np.zeros((B, N), np.int32)
    toks = np.zeros((B, N), np.int32)
    for b in range(B):
        parent[b], _ = S.random_tree(N, 4, (1, 3), rng)
        toks[b] = rng.integers(0, V, size=N)
        toks[b, 0] = 0
    out = O.verify_tree(target, parent, toks, kappa=kappa)
    for b in range(B):
        top = np.argmax(target[b], axis=-1)

        def passes(i):
            pa = parent[b, i]
            t = toks[b, i]
            if t == top[pa]:
                return True
            p = softmax64(target[b, pa])
            return kappa > 0 and p[t] / p[top[pa]] > kappa

        def path(i):
            nodes = []
            while i != 0:
                nodes.append(i)
                i = parent[b, i]
            return nodes[::-1]
        ok = [i for i in range(N) if all(passes(n) for n in path(i))]
        best = max(ok, key=lambda i: (len(path(i)), -i))
        d = len(path(best))
        assert out["accepted_len"][b] == d
        assert list(out["path_nodes"][b, :d]) == path(best)
        assert list(out["out_tokens"][b, :d]) == [toks[b, n] for n in path(best)]
        assert out["out_tokens"][b, d] == top[best]
        assert np.all(out["path_nodes"][b, d:] == -1)


# ------------------------------------------------------------------------- P9
def test_two_position_exact_law():
    """Verify several proposed tokens in one target pass: walking the positions in
    order preserves each position's target law given the accepted prefix.  K = 2,
    V = 3, enumerated exactly (grid breakpoints are multiples of 1/30)."""
    p0, q0 = [0.6, 0.3, 0.1], [0.2, 0.5, 0.3]
    p1, q1 = [0.5, 0.3, 0.2], [0.2, 0.5, 0.3]
    p2 = [0.5, 0.3, 0.2]
    inp, w = grid_chain_inputs([p0, p1], [q0, q1], p2, n=30)
    out = O.verify_chain(**inp)
    L = out["accepted_len"]
    t = out["out_tokens"]
    np.testing.assert_allclose(np.bincount(t[:, 0], weights=w, minlength=3), p0, atol=1e-12)
    m1 = L >= 1
    np.testing.assert_allclose(w[m1].sum(), np.minimum(p0, q0).sum(), atol=1e-12)
    np.testing.assert_allclose(np.bincount(t[m1, 1], weights=w[m1], minlength=3) / w[m1].sum(),
                               p1, atol=1e-12)
    m2 = L == 2
    np.testing.assert_allclose(np.bincount(t[m2, 2], weights=w[m2], minlength=3) / w[m2].sum(),
                               p2, atol=1e-12)


# ------------------------------------------------------------------ rollback
def test_rollback_lengths_cases():
    """Speculation needs cache rollback: cache lengths, returned tokens and stopping
    conditions agree."""
    kv = np.array([100, 100, 100, 100, 100, 50], np.int32)
    acc = np.array([3, 3, 3, 0, -1, 4], np.int32)
    ne = np.array([4, 4, 4, 1, 0, 5], np.int32)
    toks = np.array([[5, 6, 7, 8, -1],
                     [5, 2, 7, 8, -1],    # EOS (2) at index 1 -> keep 2 tokens
                     [5, 6, 7, 2, -1],    # EOS is the correction token
                     [2, -1, -1, -1, -1],
                     [-1] * 5,
                     [1, 1, 1, 1, 1]], np.int32)
    c, n = O.rollback_lengths(kv, acc, ne, toks, eos_id=2)
    assert list(n) == [4, 2, 4, 1, 0, 5]
    assert list(c) == [104, 103, 104, 101, 100, 55]
    max_len = np.array([102, 1000, 1000, 1000, 1000, 51], np.int32)
    c, n = O.rollback_lengths(kv, acc, ne, toks, eos_id=-1, max_len=max_len)
    assert list(n) == [1, 4, 4, 1, 0, 0]
    assert list(c) == [102, 104, 104, 101, 100, 51]


# ------------------------------------------------------------- row statuses
def test_row_status_codes():
    inp = S.make("c1")
    B = 7
    tgt = np.repeat(inp["target"], B, 0)
    drf = np.repeat(inp["draft"], B, 0)
    toks = np.repeat(inp["draft_tokens"], B, 0)
    temp = np.ones(B, np.float32)
    ua = np.repeat(inp["u_accept"], B, 0)
    us = np.repeat(inp["u_sample"], B, 0)
    tgt[1, 2, 3] = np.nan
    drf[2, 0, 5] = np.inf
    toks[3, 1] = 32
    ua[4, 0] = 1.0
    temp[5] = 0.0
    tgt[6, 4, :] = -np.inf
    out = O.verify_chain(tgt, drf, toks, temp, ua, us)
    assert list(out["row_status"]) == [0, 1, 1, 2, 3, 7, 5]
    assert np.all(out["accepted_len"][1:] == -1)
    assert np.all(out["num_emitted"][1:] == 0)
    assert np.all(out["out_tokens"][1:] == -1)
    # tree: bad parent
    par = np.array([[-1, 0, 1, 3]], np.int32)
    t = np.zeros((1, 4, 8), np.float32)
    o = O.verify_tree(t, par, np.zeros((1, 4), np.int32))
    assert o["row_status"][0] == 4


# ------------------------------------------------------- band bookkeeping pins
# The parity tests forgive a GPU/oracle disagreement only where the oracle's
# decision margin (row_margin) is below 1e-5, so these margins are pinned to
# hand-computed values.  Inputs are log-probabilities in fp32, which moves
# each probability by at most a few 1e-8; the uniforms are exact in fp32.

def test_accept_margin_worked_example():
    """Draft, Verify, and Correct -- 'Three possible next tokens': with
    p = (.6, .3, .1) and q = (.2, .5, .3) the acceptance probabilities are
    min(1, p/q) = (1, .6, 1/3).  The accept margin is |u - min(1, p/q)|,
    worked out by hand for each (token, u) below."""
    p, q = [0.6, 0.3, 0.1], [0.2, 0.5, 0.3]
    #          y, u_accept, hand margin, accepted?
    cases = [(0, 0.75, 0.25, True),      # ratio 3: min(1, 3) = 1
             (0, 0.0, 1.0, True),
             (1, 0.25, 0.35, True),      # ratio .6
             (1, 0.875, 0.275, False),
             (2, 0.5, 0.5 - 1 / 3, False),  # ratio 1/3
             (2, 0.125, 1 / 3 - 0.125, True)]
    y = [c[0] for c in cases]
    ua = [c[1] for c in cases]
    out = O.verify_chain(**_single_position(p, q, y, ua, [0.5] * len(cases)))
    np.testing.assert_allclose(out["accept_margin"][:, 0], [c[2] for c in cases], atol=1e-7)
    np.testing.assert_array_equal(out["accepted_len"] >= 1, [c[3] for c in cases])


# residual spread over two tokens: p = (.1, .5, .4), q = (.4, .3, .3) gives
# [p - q]+ = (0, .2, .1) with Z = .3 and running sums (0, .2, .3)
SPLIT_P, SPLIT_Q = [0.1, 0.5, 0.4], [0.4, 0.3, 0.3]


@pytest.mark.parametrize("u_smp,token,gap", [
    # t = u * Z; the gap is the distance of t to the nearer end of the chosen
    # token's interval, divided by Z
    (0.5, 1, 0.05 / 0.3),     # t = .15 in (0, .2]: ends .15 and .05 away
    (0.625, 1, 0.0125 / 0.3),  # t = .1875: .0125 below .2
    (0.25, 1, 0.075 / 0.3),    # t = .075: .075 above 0
    (0.75, 2, 0.025 / 0.3),    # t = .225 in (.2, .3]: .025 above .2
    (0.875, 2, 0.0375 / 0.3),  # t = .2625: .0375 below .3
])
def test_residual_gap_split_example(u_smp, token, gap):
    """Draft, Verify, and Correct -- 'Why the correction recovers the target';
    why correcting a rejection is not resampling, section 2: the correction is
    the inverse CDF of the residual at u * Z.  Position 0 rejects (y = 0,
    ratio .25, u_accept .5: accept margin .25), so row_margin is the smaller of
    .25 and the residual gap, both by hand."""
    out = O.verify_chain(**_single_position(SPLIT_P, SPLIT_Q, [0], [0.5], [u_smp]))
    assert out["accepted_len"][0] == 0
    assert out["out_tokens"][0, 0] == token
    np.testing.assert_allclose(out["resid_mass"][0, 0], 0.3, atol=1e-7)
    np.testing.assert_allclose(out["accept_margin"][0, 0], 0.25, atol=1e-7)
    np.testing.assert_allclose(out["row_margin"][0], min(0.25, gap), atol=1e-7)


@pytest.mark.parametrize("delta,token", [(2e-7, 1), (-2e-7, 0), (6e-7, 1), (-6e-7, 0)])
def test_bonus_draw_at_a_cdf_boundary(delta, token):
    """A bonus draw (K = 0) from p = (.6, .3, .1) at u = .6 + delta lands
    |delta| away from the boundary between tokens 0 and 1 (up to the fp32
    rounding of the inputs, a few 1e-8), so row_margin is about |delta|: below
    1e-6 here, inside the band that forgives a disagreement."""
    p = [0.6, 0.3, 0.1]
    tgt = log_probs(p)[None, None, :]
    us = np.array([[0.6 + delta]], np.float32)
    out = O.verify_chain(tgt, np.zeros((1, 0, 3), np.float32), np.zeros((1, 0), np.int32),
                         u_accept=np.zeros((1, 0), np.float32), u_sample=us)
    assert out["accepted_len"][0] == 0 and out["out_tokens"][0, 0] == token
    assert abs(out["row_margin"][0] - abs(delta)) < 1e-7
    assert out["row_margin"][0] < 1e-6


def test_row_margin_is_the_smallest_margin_of_the_walk():
    """Verify several proposed tokens in one target pass: the walk reads the
    accept test of positions 0..stop and the draw at the stop; row_margin is
    the least of those margins and ignores positions after the stop.
    Position 0 (DVC example, y = 1, u = .5) accepts with margin .1; position 1
    (split example, y = 0, u = .5) rejects with margin .25 and draws at u = .5
    (gap 1/6); position 2 (y = 1, ratio .6, u = .59) would have margin .01 but
    is never read."""
    p0, q0 = [0.6, 0.3, 0.1], [0.2, 0.5, 0.3]
    tgt = np.stack([log_probs(p0), log_probs(SPLIT_P), log_probs(p0), log_probs(p0)])[None]
    drf = np.stack([log_probs(q0), log_probs(SPLIT_Q), log_probs(q0)])[None]
    out = O.verify_chain(tgt, drf, np.array([[1, 0, 1]], np.int32),
                         u_accept=np.array([[0.5, 0.5, 0.59]], np.float32),
                         u_sample=np.full((1, 4), 0.5, np.float32))
    assert out["accepted_len"][0] == 1 and list(out["out_tokens"][0, :2]) == [1, 1]
    np.testing.assert_allclose(out["accept_margin"][0], [0.1, 0.25, 0.01], atol=1e-7)
    np.testing.assert_allclose(out["row_margin"][0], 0.1, atol=1e-7)
    # with position 0 at u = .3 (margin .3) the draw's gap 1/6 is the least
    out = O.verify_chain(tgt, drf, np.array([[1, 0, 1]], np.int32),
                         u_accept=np.array([[0.3, 0.5, 0.59]], np.float32),
                         u_sample=np.full((1, 4), 0.5, np.float32))
    np.testing.assert_allclose(out["row_margin"][0], 0.05 / 0.3, atol=1e-7)


def test_row_margin_of_greedy_rows_is_infinite():
    """Greedy verification takes no floating-point draw, so no band applies."""
    t = log_probs([0.6, 0.3, 0.1])[None, None, :].repeat(2, axis=1)
    out = O.verify_chain(t, None, np.array([[0]], np.int32), mode=O.GREEDY)
    assert np.isinf(out["row_margin"][0])
