"""GPU parity of the post-verification entry points against the fp64 oracle:
spec_adaptive_tree_policy (bit for bit, state included, over many steps) and
spec_kv_compact_tree (byte for byte, on paths from spec_verify_tree and on
hand-made bad paths)."""
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


@pytest.mark.parametrize("kw", [dict(), dict(divisor=0.5), dict(divisor=2.0, breaker=1),
                                dict(alpha=0.0, start=(6, 4, 5), ema0=0.4),
                                dict(alpha=1.0, shallow=(2, 8, 3), deep=(9, 1, 12))])
def test_policy_matches_oracle_over_steps(sv, kw):
    import torch
    rng = np.random.default_rng(11)
    B = 1000
    ema = rng.random(B)
    zero = rng.integers(0, 6, B).astype(np.int32)
    okw = dict(kw)
    if "shallow" in okw:
        okw["lo"], okw["hi"] = okw.pop("shallow"), okw.pop("deep")
    g_ema, g_zero = cuda(ema.copy()), cuda(zero.copy())
    for step in range(25):
        acc = rng.integers(0, 9, B).astype(np.int32)
        acc[rng.random(B) < 0.3] = 0  # runs of zero-accept steps
        dep = rng.integers(-1, 9, B).astype(np.int32)
        p1 = rng.random(B).astype(np.float32) * 1.2 - 0.1
        p1[::97] = np.nan
        shape_o, ema, zero = O.adaptive_policy(acc, dep, p1, ema, zero, **okw)
        shape_g = sv.spec_adaptive_tree_policy(cuda(acc), cuda(dep), cuda(p1), g_ema, g_zero, **kw)
        h = host(dict(shape=shape_g, ema=g_ema, zero=g_zero))
        assert np.array_equal(h["shape"], shape_o), step
        assert np.array_equal(h["ema"].view(np.uint64), ema.view(np.uint64)), step
        assert np.array_equal(h["zero"], zero), step


def _cache(rng, planes, B, S, E):
    return rng.integers(0, 256, (planes, B, S, E), dtype=np.uint8)


@pytest.mark.parametrize("draft_noise", [2.0, 0.0])
def test_kv_compaction_of_verified_tree_paths(sv, draft_noise):
    """Paths straight from spec_verify_tree on the tree workload (scaled
    down), entries of 2 KB (8 heads x 128 bf16) in 6 planes.  With no draft
    noise the drafts follow the target's own ranking, so most accepted paths
    run to the trees' depth (up to 6 moved entries a row)."""
    import torch
    inp = S.make("c4", B=32, V=4096, draft_noise=draft_noise)
    g = sv.spec_verify_tree(cuda(inp["target"]), cuda(inp["parent"]), cuda(inp["node_tokens"]),
                            margin_kappa=0.3)
    h = host(g)
    B, N = inp["parent"].shape
    rng = np.random.default_rng(5)
    planes, S_max, E = 6, N + 40, 2048
    kv = _cache(rng, planes, B, S_max, E)
    kvl = rng.integers(0, S_max - N + 1, B).astype(np.int32)
    want, st_o = O.kv_compact_tree(kv, kvl, h["accepted_len"], h["path_nodes"])
    kv_g = cuda(kv)
    st = sv.spec_kv_compact_tree(kv_g, cuda(kvl), g["accepted_len"], g["path_nodes"])
    out = host(dict(kv=kv_g, st=st))
    assert np.array_equal(out["st"], st_o)
    assert np.array_equal(out["kv"], want)
    assert (h["accepted_len"] > 1).any()  # some path really moved
    if draft_noise == 0.0:
        assert h["accepted_len"].mean() >= 3  # deep paths


@pytest.mark.parametrize("E", [16, 2048 + 16, 4096])
def test_kv_compaction_random_paths_and_bad_rows(sv, E):
    rng = np.random.default_rng(E)
    planes, B, N, S_max = 3, 40, 30, 64
    kv = _cache(rng, planes, B, S_max, E)
    kvl = rng.integers(0, S_max - N + 1, B).astype(np.int32)
    path = np.full((B, N), -1, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        a = int(rng.integers(0, N))
        path[b, :a] = np.sort(rng.choice(np.arange(1, N), a, replace=False))
        acc[b] = a
    acc[0] = -1                    # failed verify: no-op
    path[1, :3] = [4, 4, 9]        # not increasing
    acc[1] = 3
    path[2, :2] = [1, N]           # node out of range
    acc[2] = 2
    kvl[3] = S_max - N + 1         # slots past the end
    acc[3] = max(acc[3], 1)
    path[3, 0] = 1
    acc[4] = N                     # longer than a tree path can be
    want, st_o = O.kv_compact_tree(kv, kvl, acc, path)
    kv_g = cuda(kv)
    st = sv.spec_kv_compact_tree(kv_g, cuda(kvl), cuda(acc), cuda(path))
    out = host(dict(kv=kv_g, st=st))
    assert st_o[1:5].tolist() == [4, 4, 4, 4] and st_o[0] == 0
    assert np.array_equal(out["st"], st_o)
    assert np.array_equal(out["kv"], want)


# ------------------------------------------------------- DRIFT residuals
DRIFT_ATOL = 2e-4  # nats: fp32 rounding of l*s2 - M*s2 - log2 S at |l*s2| <~ 100


def compare_drift(g, o):
    gs, gr, gst = g
    os_, or_, ost = o
    assert np.array_equal(gst, ost)
    assert np.array_equal(gs, os_)
    fin = np.isfinite(or_)
    assert np.array_equal(np.isfinite(gr), fin)
    assert np.array_equal(np.isnan(gr), np.isnan(or_))
    assert np.array_equal(gr[np.isinf(or_)], or_[np.isinf(or_)])
    np.testing.assert_allclose(gr[fin], or_[fin], atol=DRIFT_ATOL, rtol=0)


def run_drift(sv, inp, m):
    g = sv.spec_drift_residuals(cuda(inp["target"]), cuda(inp["draft"]),
                                cuda(inp.get("temperature")), m=m)
    return tuple(x.cpu().numpy() for x in g)


@pytest.mark.parametrize("name,m", [("c2", 32), ("c3", 32), ("c5", 8), ("c1", 16)])
def test_drift_workloads(sv, name, m):
    inp = S.make(name, B=16) if name == "c5" else S.make(name)
    o = O.drift_residuals(inp["target"], inp["draft"], inp.get("temperature"), m=m)
    compare_drift(run_drift(sv, inp, m), o)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [37, 1001, 40000])
def test_drift_ties_unaligned_and_edges(sv, dtype, V):
    rng = np.random.default_rng(V)
    B, K, m = 6, 3, 24
    t = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 2, (B, K, V))).astype(np.float32)
    # row 0: forty equal logits straddle the support boundary
    t[0, 1, :] = np.minimum(t[0, 1, :], 5.0)
    t[0, 1, rng.choice(V, min(V, 40), replace=False)] = 5.0
    # row 1: all logits equal
    t[1, 2, :] = 1.25
    # row 2: masked draft logits inside the support
    d[2, 0, np.argsort(-t[2, 0])[:5]] = -np.inf
    # row 3: identical laws
    d[3] = t[3, :K]
    # row 4: a NaN; row 5: bad temperature
    t[4, 0, 3] = np.nan
    temp = np.full(B, 0.8, np.float32)
    temp[5] = 0.0
    if dtype == "bf16":
        t, d = S.f32_to_bf16_bits(t), S.f32_to_bf16_bits(d)
    inp = dict(target=t, draft=d, temperature=temp)
    o = O.drift_residuals(t, d, temp, m=min(m, V))
    g = run_drift(sv, inp, min(m, V))
    compare_drift(g, o)
    assert g[2][4] == 1 and g[2][5] == 7
    assert np.all(g[1][3] == 0.0)  # identical laws: exactly zero
    assert np.isinf(g[1][2, 0]).sum() == 5


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_drift_edge_rows_in_the_last_wave(sv, dtype):
    """43 rows x 8 drafted positions over V = 20000 (three ring tiles a row),
    the last rows carrying the edge cases: ties that straddle the support
    boundary in both halves of the row (many chunks share the largest
    maximum), an all-equal row (every chunk ties: the whole-row search),
    identical laws (exactly zero), masked drafts, a NaN and a bad
    temperature."""
    rng = np.random.default_rng(4343)
    B, K, V, m = 43, 8, 20000, 32
    t = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 2, (B, K, V))).astype(np.float32)
    # row 38: forty equal logits in both halves straddle the boundary
    t[38, 1, :] = np.minimum(t[38, 1, :], 5.0)
    t[38, 1, np.r_[rng.choice(V // 2, 20, replace=False), V // 2 + rng.choice(V // 2, 20, replace=False)]] = 5.0
    t[38, 4, :] = 1.25          # all logits equal
    d[39] = t[39, :K]           # identical laws
    d[40, 2, np.argsort(-t[40, 2])[:5]] = -np.inf  # masked drafts in the support
    t[41, 6, 17000] = np.nan    # a NaN in the second half
    temp = np.full(B, 0.8, np.float32)
    temp[42] = -1.0             # bad temperature
    if dtype == "bf16":
        t, d = S.f32_to_bf16_bits(t), S.f32_to_bf16_bits(d)
    inp = dict(target=t, draft=d, temperature=temp)
    o = O.drift_residuals(t, d, temp, m=m)
    g = run_drift(sv, inp, m)
    compare_drift(g, o)
    assert g[2][41] == 1 and g[2][42] == 7
    assert np.all(g[1][39] == 0.0)  # identical laws: exactly zero
    assert np.isinf(g[1][40, 2]).sum() == 5
