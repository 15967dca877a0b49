"""GPU parity at the boundary's size limits: the largest vocabulary
(SPEC_MAX_V = 262144), long chains whose walk spans several 32-position
chunks, the largest tree (SPEC_MAX_TREE_NODES = 1024 nodes) and the largest
DRIFT shapes (64 drafted positions, a support of 64).  Small batches keep the
oracle fast; the sizes that matter are the per-row ones."""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import compare_stochastic, cuda, host, run_chain
from workloads import synthetic as S

pytestmark = pytest.mark.gpu

MAX_V = 262144
MAX_NODES = 1024


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


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_largest_vocabulary_stochastic(sv, dtype):
    """V = 262144: 32 (bf16) or 64 (fp32) stream tiles per logit row and the
    resolve kernel's most vocabulary per cluster CTA."""
    inp = S.chain_inputs(B=3, K=3, V=MAX_V, dtype=dtype, sigma=3.0, seed=71, temperature=(0.6, 1.2),
                         peaks=20, peak_boost=8.0)
    compare_stochastic(run_chain(sv, inp), oracle_chain(inp))


def test_largest_vocabulary_greedy_and_truncated(sv):
    inp = S.chain_inputs(B=3, K=4, V=MAX_V, dtype="bf16", sigma=3.0, seed=72, greedy=True)
    g = run_chain(sv, inp, mode="greedy", kappa=0.3, draft=False)
    o = oracle_chain(inp, O.GREEDY, 0.3)
    assert np.array_equal(g["out_tokens"], o["out_tokens"])
    assert np.array_equal(g["accepted_len"], o["accepted_len"])
    st = S.chain_inputs(B=3, K=3, V=MAX_V, dtype="bf16", sigma=3.0, seed=73, peaks=20, peak_boost=8.0)
    k = np.array([50, 0, 1000], np.int32)
    p = np.array([0.9, 0.95, 1.0], np.float32)
    g = host(sv.spec_verify_chain(cuda(st["target"]), cuda(st["draft"]), cuda(st["draft_tokens"]),
                                  cuda(st.get("temperature")), cuda(st["u_accept"]), cuda(st["u_sample"]),
                                  diagnostics=True, top_k=cuda(k), top_p=cuda(p)))
    o = O.verify_chain(st["target"], st["draft"], st["draft_tokens"], st.get("temperature"),
                       st["u_accept"], st["u_sample"], top_k=k, top_p=p)
    assert compare_stochastic(g, o) <= 1


@pytest.mark.parametrize("K", [63, 200])
def test_long_chains(sv, K):
    """The walk crosses several 32-position chunks; identical target and
    draft laws make long acceptance runs, so later chunks decide the stop."""
    rng = np.random.default_rng(K)
    B, V = 4, 1000
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 0.05, (B, K, V))).astype(np.float32)
    d[1] = t[1, :K]  # row 1: identical laws, every draft passes (bonus)
    temp = np.full(B, 1.0, np.float32)
    # drafts sampled from q (Gumbel-max), uniforms fixed
    y = np.argmax(d / temp[:, None, None] + rng.gumbel(size=d.shape), axis=-1).astype(np.int32)
    inp = dict(target=S.f32_to_bf16_bits(t), draft=S.f32_to_bf16_bits(d), draft_tokens=y,
               temperature=temp, u_accept=rng.random((B, K), dtype=np.float32),
               u_sample=rng.random((B, K + 1), dtype=np.float32))
    g = run_chain(sv, inp)
    o = oracle_chain(inp)
    compare_stochastic(g, o)
    assert g["accepted_len"][1] == K  # identical laws never reject
    assert o["accepted_len"].max() >= 32  # the walk left the first chunk
    gg = run_chain(sv, inp, mode="greedy", kappa=1e-30, draft=False)
    og = oracle_chain(inp, O.GREEDY, 1e-30)
    assert np.array_equal(gg["out_tokens"], og["out_tokens"])


def test_largest_tree(sv):
    """N = 1024 nodes: the walk kernel's combine over every node and its
    root-path AND by pointer jumping over all of them."""
    inp = S.tree_inputs(B=2, N=MAX_NODES, V=512, dtype="bf16", sigma=2.0, max_depth=40,
                        branch=(1, 3), seed=74)
    for kappa in (0.0, 0.3):
        g = host(sv.spec_verify_tree(cuda(inp["target"]), cuda(inp["parent"]),
                                     cuda(inp["node_tokens"]), margin_kappa=kappa))
        o = O.verify_tree(inp["target"], inp["parent"], inp["node_tokens"], kappa=kappa)
        for k in ("accepted_len", "path_nodes", "out_tokens", "num_emitted", "row_status"):
            assert np.array_equal(g[k], o[k]), (kappa, k)


def test_deepest_tree_pointer_jumping(sv):
    """A 1024-node tree that is one chain (parent[i] = i - 1) is 1023 edges
    deep, so the walk's pointer jumping takes its full 10 rounds before the
    links all reach the root.  Row 0 accepts every node; rows 1 and 2 have a
    single mismatch (at node 3 and node 700) that the margin rule cannot
    promote (the token with the smallest logit).  Checked at kappa 0 and 0.3."""
    rng = np.random.default_rng(1023)
    B, N, V = 3, MAX_NODES, 512
    t = S.f32_to_bf16_bits(rng.normal(0.0, 2.0, (B, N, V)).astype(np.float32))
    tv = S.as_float32(t)
    parent = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    toks = np.zeros((B, N), np.int32)
    toks[:, 1:] = np.argmax(tv[:, :-1], axis=-1)  # first index of the maximum
    for b, node in ((1, 3), (2, 700)):
        toks[b, node] = int(np.argmin(tv[b, node - 1]))
    for kappa in (0.0, 0.3):
        g = host(sv.spec_verify_tree(cuda(t), cuda(parent), cuda(toks), margin_kappa=kappa))
        o = O.verify_tree(t, parent, toks, kappa=kappa)
        assert list(o["accepted_len"]) == [N - 1, 2, 699]
        for k in ("accepted_len", "path_nodes", "out_tokens", "num_emitted", "row_status"):
            assert np.array_equal(g[k], o[k]), (kappa, k)


def test_largest_drift_shapes(sv):
    """K = 64 drafted positions with a support of m = 64."""
    inp = S.chain_inputs(B=2, K=64, V=3000, dtype="bf16", sigma=3.0, seed=75, temperature=(0.7, 1.1))
    g = sv.spec_drift_residuals(cuda(inp["target"]), cuda(inp["draft"]), cuda(inp["temperature"]), m=64)
    sup, res, st = (x.cpu().numpy() for x in g)
    osup, ores, ost = O.drift_residuals(inp["target"], inp["draft"], inp["temperature"], m=64)
    assert np.array_equal(st, ost)
    ok = ost == 0
    assert np.array_equal(sup[ok], osup[ok])
    np.testing.assert_allclose(res[ok], ores[ok], rtol=0, atol=2e-4)
