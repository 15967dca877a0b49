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


def test_kv_compaction_of_verified_tree_paths(sv):
    """Paths straight from spec_verify_tree on the tree workload (scaled
    down), entries of 2 KB (8 heads x 128 bf16) in 6 planes."""
    import torch
    inp = S.make("c4", B=32, V=4096)
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
