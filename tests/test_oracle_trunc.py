"""Pins of the oracle's top-k / top-p truncated verification against facts
outside the oracle: hand-computed truncated laws of the worked example in
"Speculative Decoding: Draft, Verify, and Correct" ('Three possible next
tokens'), the exact law by enumeration over a uniform grid, the reduction of
top-k = 1 to the greedy walk, and the identity when truncation is off."""
import numpy as np
import pytest

from oracle import oracle as O
from workloads import synthetic as S

P3 = np.array([0.6, 0.3, 0.1])
Q3 = np.array([0.2, 0.5, 0.3])


def _example(y, ua, us, **kw):
    t = np.log(np.tile(P3, (len(y), 2, 1))).astype(np.float32)
    d = np.log(np.tile(Q3, (len(y), 1, 1))).astype(np.float32)
    return O.verify_chain(t, d, np.array(y, np.int32).reshape(-1, 1), None,
                          np.array(ua, np.float32).reshape(-1, 1),
                          np.array(us, np.float32).reshape(-1, 2), **kw)


@pytest.mark.parametrize("kw", [dict(top_k=[2] * 4), dict(top_p=[0.7] * 4)])
def test_truncated_worked_example(kw):
    """top-2 (or top-p 0.7, which keeps the same tokens): p' = (2/3, 1/3, 0),
    q' = (0, 0.625, 0.375); the draft token 1 passes with probability
    (1/3)/0.625; token 2 never passes; the residual is all on token 0."""
    o = _example([1, 1, 2, 2], [0.53, 0.54, 0.0, 0.99], [0.5] * 8, **kw)
    assert o["accepted_len"].tolist() == [1, 0, 0, 0]
    assert o["out_tokens"][1:, 0].tolist() == [0, 0, 0]  # the residual's only token
    np.testing.assert_allclose(o["p_at_draft"][:, 0], [1 / 3, 1 / 3, 0, 0], rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(o["q_at_draft"][:, 0], [0.625, 0.625, 0.375, 0.375], rtol=1e-6)
    np.testing.assert_allclose(o["resid_mass"][1:, 0], [2 / 3] * 3, rtol=1e-6)


def test_top_k_then_top_p_on_the_renormalised_law():
    """Top-k first, then top-p on the renormalised top-k law, written out by
    hand.  top-2 of p = (.6, .3, .1) is (2/3, 1/3, 0); its top-0.65 set is
    {0} alone (2/3 >= 0.65), so p'' = (1, 0, 0).  top-2 of q = (.2, .5, .3)
    is (0, .625, .375); .625 < 0.65, so q'' keeps both: (0, .625, .375).
    Draft token 1: p''(1) = 0 rejects it whatever u, and the residual
    (p'' - q'')+ = (1, 0, 0) emits token 0.  (Counting the top-p mass on the
    law before the top-k renormalisation would keep token 1 in p'': .6 <
    0.65.)"""
    o = _example([1, 1], [0.0, 0.99], [0.5] * 4, top_k=[2] * 2, top_p=[0.65] * 2)
    assert o["accepted_len"].tolist() == [0, 0]
    assert o["out_tokens"][:, 0].tolist() == [0, 0]
    np.testing.assert_allclose(o["p_at_draft"][:, 0], [0.0, 0.0], atol=1e-12)
    np.testing.assert_allclose(o["q_at_draft"][:, 0], [0.625, 0.625], rtol=1e-6)
    np.testing.assert_allclose(o["resid_mass"][:, 0], [1.0, 1.0], rtol=1e-6)


def test_truncated_exact_law_by_enumeration():
    """Draft tokens drawn from q' and uniforms on a fine grid: the first
    emitted token follows p' exactly (accepted mass + residual mass)."""
    qp = np.array([0.0, 0.625, 0.375])
    pp = np.array([2 / 3, 1 / 3, 0.0])
    n = 400
    u = (np.arange(n) + 0.5) / n
    law = np.zeros(3)
    for y in (1, 2):
        o = _example([y] * n, u, np.repeat(u[:, None], 2, 1).ravel(), top_k=[2] * n)
        first = o["out_tokens"][:, 0]
        for v in range(3):
            law[v] += qp[y] * np.mean(first == v)
    np.testing.assert_allclose(law, pp, atol=1.5 / n)


def test_top_k_one_is_the_greedy_walk():
    """With top-k = 1 both laws are one-hot: a draft equal to the draft argmax
    passes iff it is the target argmax, and a rejection emits the target
    argmax -- the greedy rule, whatever the uniforms."""
    inp = S.make("c2", greedy=True)
    B, K = inp["draft_tokens"].shape
    rng = np.random.default_rng(8)
    g = O.verify_chain(inp["target"], None, inp["draft_tokens"], mode=O.GREEDY)
    s = O.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], None,
                       rng.random((B, K), dtype=np.float32), rng.random((B, K + 1), dtype=np.float32),
                       top_k=np.ones(B, np.int32))
    assert np.array_equal(s["accepted_len"], g["accepted_len"])
    assert np.array_equal(s["out_tokens"], g["out_tokens"])


def test_top_k_keeps_boundary_ties():
    t = np.log(np.array([[[0.4, 0.2, 0.2, 0.2]] * 2], np.float64)).astype(np.float32)
    d = np.log(np.array([[[0.25] * 4]], np.float64)).astype(np.float32)
    o = O.verify_chain(t, d, np.array([[3]], np.int32), None, np.array([[0.0]], np.float32),
                       np.array([[0.5, 0.5]], np.float32), top_k=[2])
    # target keeps all four (three tied at the 2nd largest); draft keeps all four
    np.testing.assert_allclose(o["p_at_draft"][0, 0], 0.2, rtol=1e-6)
    np.testing.assert_allclose(o["q_at_draft"][0, 0], 0.25, rtol=1e-6)


def test_truncation_off_is_the_plain_verifier():
    inp = S.make("c2")
    B = inp["draft_tokens"].shape[0]
    args = (inp["target"], inp["draft"], inp["draft_tokens"], inp.get("temperature"),
            inp["u_accept"], inp["u_sample"])
    a = O.verify_chain(*args)
    b = O.verify_chain(*args, top_k=np.full(B, 32000, np.int32), top_p=np.ones(B, np.float32))
    c = O.verify_chain(*args, top_k=np.zeros(B, np.int32))
    for k in a:
        assert np.array_equal(a[k], b[k]) and np.array_equal(a[k], c[k]), k


def test_top_p_margin_enters_the_band():
    """The top-p boundary is a floating-point decision: a row whose cumulative
    mass lands next to top_p reports a tiny row margin."""
    t = np.log(np.tile(P3, (1, 2, 1))).astype(np.float32)
    d = np.log(np.tile(Q3, (1, 1, 1))).astype(np.float32)
    o = O.verify_chain(t, d, np.array([[1]], np.int32), None, np.array([[0.99]], np.float32),
                       np.array([[0.5, 0.5]], np.float32), top_p=[0.9 + 1e-9])
    assert o["row_margin"][0] < 1e-6
