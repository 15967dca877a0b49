"""GPU parity of spec_verify_tree and spec_rollback_lengths (bit exact)."""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import cuda, host
from workloads import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch
    import speculative_decoding_verification_32_gb300 as m
    assert torch.cuda.is_available()
    return m


def run_tree(sv, inp, kappa, temperature=None):
    return host(sv.spec_verify_tree(cuda(inp["target"]), cuda(inp["parent"]),
                                    cuda(inp["node_tokens"]), cuda(temperature),
                                    margin_kappa=kappa))


def check_tree(g, o):
    for k in ("accepted_len", "path_nodes", "out_tokens", "num_emitted", "row_status"):
        assert np.array_equal(g[k], o[k]), k


@pytest.mark.parametrize("kappa", [0.3, 0.0])
def test_c4_full(sv, kappa):
    """B = 32 trees of 60 nodes over V = 151936, margin rule kappa = 0.3."""
    inp = S.make("c4")
    g = run_tree(sv, inp, kappa)
    o = O.verify_tree(inp["target"], inp["parent"], inp["node_tokens"], kappa=kappa)
    check_tree(g, o)
    if kappa:
        assert o["accepted_len"].max() >= 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [5, 300, 4099, 70000])
def test_small_trees_with_ties(sv, dtype, V):
    rng = np.random.default_rng(V)
    B, N = 24, 40
    t = rng.integers(-3, 3, size=(B, N, V)).astype(np.float32)
    parent = np.zeros((B, N), np.int32)
    toks = np.zeros((B, N), np.int32)
    for b in range(B):
        parent[b], _ = S.random_tree(N, 6, (1, 4), rng)
        top = np.argmax(t[b], axis=-1)
        for i in range(1, N):  # mostly the parent's argmax, sometimes a random token
            toks[b, i] = top[parent[b, i]] if rng.random() < 0.7 else rng.integers(0, V)
    target = S.f32_to_bf16_bits(t) if dtype == "bf16" else t
    temp = rng.uniform(0.5, 2.0, B).astype(np.float32)
    inp = dict(target=target, parent=parent, node_tokens=toks)
    for kappa in (0.0, 0.3, 0.9):
        g = run_tree(sv, inp, kappa, temp)
        o = O.verify_tree(target, parent, toks, temperature=temp, kappa=kappa)
        check_tree(g, o)


def test_tree_with_chain_parents_equals_chain(sv):
    inp = S.make("c2", greedy=True)
    B, K = inp["draft_tokens"].shape
    parent = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    toks = np.concatenate([np.zeros((B, 1), np.int32), inp["draft_tokens"]], axis=1)
    for kappa in (0.0, 0.3):
        gt = run_tree(sv, dict(target=inp["target"], parent=parent, node_tokens=toks), kappa)
        gc = host(sv.spec_verify_chain(cuda(inp["target"]), None, cuda(inp["draft_tokens"]),
                                       mode="greedy", margin_kappa=kappa))
        assert np.array_equal(gt["out_tokens"], gc["out_tokens"])
        assert np.array_equal(gt["accepted_len"], gc["accepted_len"])


def test_tree_bad_inputs(sv):
    inp = S.make("c4", B=4, V=1000)
    inp["parent"][1, 5] = 7            # parent after child
    inp["parent"][2, 0] = 0            # root must have parent -1
    inp["node_tokens"][3, 9] = 1000    # token out of range
    g = run_tree(sv, inp, 0.3)
    o = O.verify_tree(inp["target"], inp["parent"], inp["node_tokens"], kappa=0.3)
    assert list(o["row_status"]) == [0, 4, 4, 2]
    check_tree(g, o)


def test_tree_nonfinite_and_cross_slice_ties(sv):
    """The walk kernel's thread-per-node combine (60 nodes): a NaN, a +inf and
    a node with no finite logit flag their rows; equal maxima in the first and
    last vocabulary slices resolve to the lower index."""
    inp = S.make("c4", B=6, V=9000)
    t = S.as_float32(inp["target"]).copy()
    t[1, 7, 4000] = np.nan
    t[2, 3, 8999] = np.inf
    t[3, 11, :] = -np.inf
    t[4, 20, 100] = t[4, 20].max() + 1
    t[4, 20, 8990] = t[4, 20, 100]
    t[5, 0, 9] = t[5, 0].max() + 1  # root: argmax at the first slice's start...
    t[5, 0, 8999] = t[5, 0, 9]      # ...tied at the last slice's end
    target = S.f32_to_bf16_bits(t)
    for kappa in (0.0, 0.3):
        g = run_tree(sv, dict(target=target, parent=inp["parent"], node_tokens=inp["node_tokens"]), kappa)
        o = O.verify_tree(target, inp["parent"], inp["node_tokens"], kappa=kappa)
        assert list(o["row_status"]) == [0, 1, 1, 5, 0, 0]
        check_tree(g, o)


def test_single_node_tree(sv):
    inp = S.make("c4", B=3, N=1, V=2000)
    g = run_tree(sv, inp, 0.3)
    o = O.verify_tree(inp["target"], inp["parent"], inp["node_tokens"], kappa=0.3)
    check_tree(g, o)
    assert np.all(g["accepted_len"] == 0)


def test_rollback_parity(sv):
    rng = np.random.default_rng(9)
    B, E = 300, 9
    acc = rng.integers(-1, E, size=B).astype(np.int32)
    ne = np.where(acc >= 0, acc + 1, 0).astype(np.int32)
    toks = rng.integers(0, 6, size=(B, E)).astype(np.int32)
    kv = rng.integers(0, 500, size=B).astype(np.int32)
    max_len = (kv + rng.integers(-2, 12, size=B)).astype(np.int32)
    for eos, ml in [(-1, None), (3, None), (3, max_len), (-1, max_len)]:
        c, n = sv.spec_rollback_lengths(cuda(kv), cuda(acc), cuda(ne), cuda(toks), eos,
                                        cuda(ml))
        oc, on = O.rollback_lengths(kv, acc, ne, toks, eos, ml)
        assert np.array_equal(c.cpu().numpy(), oc)
        assert np.array_equal(n.cpu().numpy(), on)
