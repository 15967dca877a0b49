"""Pins of the oracle's next-row functions against facts that do not come from
the oracle itself: the shape endpoints and breaker count printed in "Margins,
Not Windows" ("Method", dynamic draft tree-shaping), the closed form of an
exponential moving average under a constant input, and byte patterns that
name their own (plane, row, slot) for the KV path compaction."""
import numpy as np
import pytest

from oracle import oracle as O


# ------------------------------------------------------ AdaptiveSpec policy
def test_policy_endpoints_are_the_pages_shapes():
    """DCS = 0 gives the shallow-wide (3, 4, 4); DCS = 1 the deep-narrow
    (7, 1, 8)."""
    # DCS = 0: draft top-1 probability 0
    s, _, _ = O.adaptive_policy([3], [7], [0.0], [0.5], [0])
    assert s.tolist() == [[3, 4, 4]]
    # DCS = 1: full acceptance history and a certain draft
    s, e, _ = O.adaptive_policy([7], [7], [1.0], [1.0], [0])
    assert e[0] == 1.0 and s.tolist() == [[7, 1, 8]]


def test_policy_depth_grows_and_branching_shrinks_with_confidence():
    p1 = np.linspace(0.0, 1.0, 101).astype(np.float32)
    n = p1.size
    s, _, _ = O.adaptive_policy(np.full(n, 7), np.full(n, 7), p1, np.ones(n), np.zeros(n))
    assert np.all(np.diff(s[:, 0]) >= 0) and np.all(np.diff(s[:, 2]) >= 0)  # nsteps, ndt
    assert np.all(np.diff(s[:, 1]) <= 0)  # top-k
    assert s[:, 0].min() == 3 and s[:, 0].max() == 7


def test_policy_ema_closed_form():
    """alpha = 0.3 moving average of a constant acceptance fraction f from e0:
    e_t = f + (e0 - f) * 0.7^t."""
    f, e0 = 3.0 / 7.0, 0.9
    e = np.array([e0])
    z = np.array([0])
    for t in range(1, 41):
        _, e, z = O.adaptive_policy([3], [7], [0.5], e, z, alpha=0.3)
        assert abs(e[0] - (f + (e0 - f) * 0.7 ** t)) < 1e-12


def test_policy_circuit_breaker_after_five_zero_accept_steps():
    start = (6, 4, 5)  # not a shape the interpolation can produce
    e, z = np.array([0.8]), np.array([0])
    for step in range(1, 6):
        s, e, z = O.adaptive_policy([0], [7], [0.9], e, z, start=start, ema0=0.25)
        if step < 5:
            assert z[0] == step and s.tolist() != [list(start)]
        else:  # the fifth consecutive zero-accept step restores the start
            assert s.tolist() == [list(start)] and e[0] == 0.25 and z[0] == 0
    _, _, z = O.adaptive_policy([0], [7], [0.9], [0.5], [4])
    assert z[0] == 0  # the fifth zero: the breaker fired and cleared the count
    _, _, z = O.adaptive_policy([1], [7], [0.9], [0.5], [3])
    assert z[0] == 0  # an accepted token clears it too


def test_policy_divisor_saturates_the_score():
    """DCS = min(1, p1 * ema / d): with d = 0.5, p1 * ema >= 0.5 is already the
    deep-narrow end; with d = 1 it is not."""
    s, _, _ = O.adaptive_policy([7], [7], [0.6], [1.0], [0], divisor=0.5)
    assert s.tolist() == [[7, 1, 8]]
    s, _, _ = O.adaptive_policy([7], [7], [0.6], [1.0], [0], divisor=1.0)
    assert s.tolist() != [[7, 1, 8]]


# ---------------------------------------------------------- KV compaction
def _named_cache(planes, B, S, E):
    """Every entry's bytes spell its own (plane, row, slot)."""
    kv = np.zeros((planes, B, S, E), dtype=np.uint8)
    p, b, s = np.meshgrid(np.arange(planes), np.arange(B), np.arange(S), indexing="ij")
    code = (p * 7919 + b * 131 + s).astype(np.uint32)
    for i in range(E):
        kv[..., i] = ((code >> (8 * (i % 4))) + i) & 0xFF
    return kv


def test_kv_compaction_moves_each_path_entry_to_its_slot():
    rng = np.random.default_rng(7)
    planes, B, N, S, E = 3, 5, 12, 40, 8
    kv = _named_cache(planes, B, S, E)
    kvl = rng.integers(0, S - N, B).astype(np.int32)
    path = np.full((B, N), -1, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        a = int(rng.integers(0, 6))
        path[b, :a] = np.sort(rng.choice(np.arange(1, N), a, replace=False))
        acc[b] = a
    out, st = O.kv_compact_tree(kv, kvl, acc, path)
    assert np.all(st == 0)
    for b in range(B):
        a, base = acc[b], kvl[b]
        moved = set(base + 1 + np.arange(a))
        for k in range(a):  # destination holds the named source entry
            assert np.array_equal(out[:, b, base + 1 + k], kv[:, b, base + path[b, k]])
        for s in range(S):  # every other slot is untouched
            if s not in moved:
                assert np.array_equal(out[:, b, s], kv[:, b, s])


def test_kv_compaction_of_a_chain_is_the_identity():
    """A chain's accepted nodes 1..a already sit in their slots."""
    kv = _named_cache(2, 3, 20, 16)
    path = np.tile(np.arange(1, 10, dtype=np.int32), (3, 1))  # N = 9 nodes per tree
    path[:, -1] = -1
    out, st = O.kv_compact_tree(kv, [0, 4, 11], [8, 3, 0], path)
    assert np.all(st == 0) and np.array_equal(out, kv)


def test_kv_compaction_rejects_bad_paths_and_skips_failed_rows():
    kv = _named_cache(1, 4, 16, 4)
    path = np.array([[2, 2, 0, 0], [0, 1, 0, 0], [1, 5, 0, 0], [3, 1, 0, 0]], np.int32)
    out, st = O.kv_compact_tree(kv, [0, 0, 0, 0], [2, 1, 2, 2], path)
    # not increasing, node 0, node >= N, decreasing
    assert st.tolist() == [4, 4, 4, 4] and np.array_equal(out, kv)
    out, st = O.kv_compact_tree(kv, [14, 0, 0, 0], [1, -1, 0, 0], np.tile([[1, 2, 3, 0]], (4, 1)))
    assert st.tolist() == [4, 0, 0, 0]  # slots past S_max; a < 0 is a no-op
    assert np.array_equal(out, kv)


# ------------------------------------------------------- DRIFT residuals
def _log_softmax(x):
    from scipy.special import logsumexp
    return x - logsumexp(x)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_drift_residual_closed_form(T):
    """Draft logits a * target: log q is log_softmax(a l / T), computed here by
    scipy's logsumexp; the support is the top-m of the target by a stable
    lexsort (ties to the lower index)."""
    rng = np.random.default_rng(3)
    B, K, V, m = 2, 3, 500, 32
    tgt = (rng.normal(0, 3, (B, K + 1, V))).astype(np.float32)
    tgt[0, 0, 10:20] = tgt[0, 0, 7]  # a run of ties inside the support
    tgt[0, 0, 7] = tgt[0, 0].max() + 1.0
    tgt[0, 0, 10:20] = tgt[0, 0, 7] - 0.5
    drf = (0.6 * tgt[:, :K]).astype(np.float32)
    sup, res, st = O.drift_residuals(tgt, drf, np.full(B, T, np.float32), m=m)
    assert np.all(st == 0)
    for b in range(B):
        for j in range(K):
            l = tgt[b, j].astype(np.float64)
            order = np.lexsort((np.arange(V), -l))[:m]
            assert np.array_equal(sup[b, j], order)
            lp = _log_softmax(l / T)
            lq = _log_softmax(drf[b, j].astype(np.float64) / T)
            np.testing.assert_allclose(res[b, j], (lp - lq)[order], rtol=0, atol=1e-5)
    assert sup[0, 0, 0] == 7 and list(sup[0, 0, 1:11]) == list(range(10, 20))


def test_drift_residual_identical_laws_and_masks():
    """draft = target + c: q = p, so the residual is 0; a masked draft logit
    inside the support gives +inf."""
    rng = np.random.default_rng(4)
    tgt = rng.normal(0, 2, (1, 3, 300)).astype(np.float32)
    drf = (tgt[:, :2] + 3.0).astype(np.float32)
    sup, res, _ = O.drift_residuals(tgt, drf, m=16)
    assert np.all(np.abs(res) < 1e-12 + 1e-6)
    drf[0, 1, sup[0, 1, 3]] = -np.inf
    sup2, res2, st = O.drift_residuals(tgt, drf, m=16)
    assert st[0] == 0 and np.array_equal(sup2, sup)
    assert res2[0, 1, 3] == np.inf and np.isfinite(np.delete(res2[0, 1], 3)).all()


def test_drift_residual_bad_rows():
    tgt = np.zeros((2, 2, 40), np.float32)
    drf = np.zeros((2, 1, 40), np.float32)
    tgt[1, 0, 5] = np.nan
    sup, res, st = O.drift_residuals(tgt, drf, np.array([1.0, 1.0], np.float32), m=4)
    assert st.tolist() == [0, 1]
    assert np.all(sup[1] == -1) and np.all(np.isnan(res[1]))
    assert sup[0, 0].tolist() == [0, 1, 2, 3]  # all equal: lowest indices
    _, _, st = O.drift_residuals(tgt, drf, np.array([0.0, 1.0], np.float32), m=4)
    assert st[0] == 7
