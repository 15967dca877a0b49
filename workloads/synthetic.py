"""Seeded synthetic inputs for the draft-verification sampler.

This module is the ONLY code that both the CUDA path's tests/bench and the
oracle consume.  It holds none of the verification arithmetic: it draws
logits, draft tokens, uniforms and trees, nothing else.  Draft tokens are
drawn from the draft law q = softmax(draft / T) with the Gumbel-max trick
(argmax of draft / T + Gumbel noise), which samples q exactly without ever
forming q.

All randomness comes from numpy's PCG64 with per-row-chunk child seeds, so the
same seed gives the same inputs on any machine and any thread count.

Logits come back as numpy arrays: float32, or bf16 as raw uint16 bit patterns
(round-to-nearest-even from float32).
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# The five workloads (name -> parameters).  "sigma" is the standard deviation
# of the target logits; draft logits are draft_scale * target + N(0, draft_noise).
CONFIGS = {
    # tiny fp32 chain: the oracle runs it instantly
    "c1": dict(kind="chain", B=1, K=4, V=32, dtype="f32", sigma=2.0, draft_scale=1.0,
               draft_noise=1.0, temperature=1.0, seed=1001),
    # small bf16 chain, greedy and stochastic
    "c2": dict(kind="chain", B=8, K=4, V=32000, dtype="bf16", sigma=3.0, draft_scale=0.8,
               draft_noise=1.5, temperature=1.0, seed=1002),
    # headline chain: 64 rows, 5 drafts, 128256-token vocabulary, T = 0.7,
    # 20 boosted "peak" tokens per row
    "c3": dict(kind="chain", B=64, K=5, V=128256, dtype="bf16", sigma=3.0, draft_scale=1.0,
               draft_noise=2.0, temperature=0.7, peaks=20, peak_boost=8.0, seed=1003),
    # parent-indexed draft trees with the margin rule
    "c4": dict(kind="tree", B=32, N=60, V=151936, dtype="bf16", sigma=3.0, draft_noise=2.0,
               max_depth=6, branch=(1, 4), kappa=0.3, seed=1004),
    # chain at scale: per-row temperatures, 10% of draft logits masked to -inf
    "c5": dict(kind="chain", B=256, K=8, V=128256, dtype="bf16", sigma=3.0, draft_scale=1.0,
               draft_noise=2.5, temperature=(0.3, 1.2), mask_frac=0.1, seed=1005),
}

_ROWS_PER_CHUNK = 8


def f32_to_bf16_bits(x):
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(h):
    """bf16 bit patterns (uint16) -> float32 values (exact)."""
    return (np.ascontiguousarray(h).astype(np.uint32) << 16).view(np.float32)


def as_float32(logits):
    """Logits (float32 or bf16 bits) as float32 values."""
    return bf16_bits_to_f32(logits) if logits.dtype == np.uint16 else logits


def _pack(x, dtype):
    return f32_to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def _chunks(B):
    return [(s, min(B, s + _ROWS_PER_CHUNK)) for s in range(0, B, _ROWS_PER_CHUNK)]


def _parallel(fn, B, seed, tag):
    """Run fn(rng, lo, hi) over row chunks with one child generator per chunk."""
    chunks = _chunks(B)
    seqs = np.random.SeedSequence([seed, tag]).spawn(len(chunks))
    with ThreadPoolExecutor(max_workers=min(16, max(1, len(chunks)))) as ex:
        list(ex.map(lambda a: fn(np.random.Generator(np.random.PCG64(a[1])), *a[0]),
                    zip(chunks, seqs)))


def gumbel_max_tokens(draft_vals, temperature, rng):
    """One draw per row from softmax(draft_vals / T) via the Gumbel-max trick.

    draft_vals [..., V] float32 (may hold -inf); temperature broadcastable to
    draft_vals[..., :1].  Returns int32 [...].
    """
    u = rng.random(draft_vals.shape, dtype=np.float32)
    with np.errstate(divide="ignore"):
        g = -np.log(-np.log(u))  # u == 0 gives -inf: that entry is never drawn
    return np.argmax(draft_vals / temperature + g, axis=-1).astype(np.int32)


def chain_inputs(B, K, V, dtype="bf16", sigma=3.0, draft_scale=1.0, draft_noise=2.0,
                 temperature=1.0, peaks=0, peak_boost=0.0, mask_frac=0.0, greedy=False,
                 seed=0, **_):
    """Chain-verification inputs.

    Returns dict(target [B,K+1,V], draft [B,K,V], draft_tokens [B,K] int32,
    temperature [B] f32, u_accept [B,K] f32, u_sample [B,K+1] f32, dtype).
    greedy=True draws draft tokens as argmax of the draft logits instead.
    """
    tdt = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((B, K + 1, V), tdt)
    draft = np.empty((B, K, V), tdt)
    tokens = np.empty((B, K), np.int32)
    rng0 = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    if isinstance(temperature, tuple):
        temp = rng0.uniform(temperature[0], temperature[1], size=B).astype(np.float32)
    else:
        temp = np.full(B, temperature, np.float32)
    u_accept = rng0.random((B, K), dtype=np.float32)
    u_sample = rng0.random((B, K + 1), dtype=np.float32)

    def fill(rng, lo, hi):
        n = hi - lo
        t = rng.standard_normal((n, K + 1, V), dtype=np.float32) * np.float32(sigma)
        if peaks:
            for r in range(n):
                ids = rng.choice(V, size=peaks, replace=False)
                t[r][:, ids] += np.float32(peak_boost)
        d = t[:, :K] * np.float32(draft_scale) + \
            rng.standard_normal((n, K, V), dtype=np.float32) * np.float32(draft_noise)
        if mask_frac:
            d[rng.random((n, K, V), dtype=np.float32) < mask_frac] = -np.inf
        target[lo:hi] = _pack(t, dtype)
        draft[lo:hi] = _pack(d, dtype)
        dv = as_float32(draft[lo:hi])
        if greedy:
            tokens[lo:hi] = np.argmax(dv, axis=-1).astype(np.int32)
        else:
            tokens[lo:hi] = gumbel_max_tokens(dv, temp[lo:hi, None, None], rng)

    _parallel(fill, B, seed, 1)
    return dict(target=target, draft=draft, draft_tokens=tokens, temperature=temp,
                u_accept=u_accept, u_sample=u_sample, dtype=dtype)


def random_tree(N, max_depth, branch, rng):
    """Parent array of an N-node tree built breadth first.

    Node 0 is the root.  Each expanded node gets a branching factor drawn
    uniformly from branch=(lo, hi); nodes at max_depth are not expanded.
    Children are numbered in breadth-first order, so parent[i] < i.
    Returns (parent int32 [N], depth int32 [N]).
    """
    parent = [-1]
    depth = [0]
    frontier = [0]
    while len(parent) < N:
        if not frontier:  # every node so far is a leaf or at max depth: widen the shallowest
            frontier = [i for i in range(len(parent)) if depth[i] < max_depth]
        nxt = []
        for u in frontier:
            if len(parent) >= N:
                break
            if depth[u] >= max_depth:
                continue
            k = int(rng.integers(branch[0], branch[1] + 1))
            for _ in range(k):
                if len(parent) >= N:
                    break
                parent.append(u)
                depth.append(depth[u] + 1)
                nxt.append(len(parent) - 1)
        frontier = nxt
    return np.array(parent, np.int32), np.array(depth, np.int32)


def tree_inputs(B, N, V, dtype="bf16", sigma=3.0, draft_noise=2.0, max_depth=6,
                branch=(1, 4), kappa=0.3, seed=0, **_):
    """Tree-verification inputs.

    The children of node P carry the top-1, top-2, ... tokens of a draft row
    (target row P + N(0, draft_noise)), in child order.  Returns dict(target
    [B,N,V], parent [B,N], node_tokens [B,N], kappa, dtype).
    """
    tdt = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((B, N, V), tdt)
    parent = np.empty((B, N), np.int32)
    tokens = np.zeros((B, N), np.int32)

    def fill(rng, lo, hi):
        for b in range(lo, hi):
            par, _ = random_tree(N, max_depth, branch, rng)
            t = rng.standard_normal((N, V), dtype=np.float32) * np.float32(sigma)
            target[b] = _pack(t, dtype)
            d = as_float32(target[b]) + \
                rng.standard_normal((N, V), dtype=np.float32) * np.float32(draft_noise)
            parent[b] = par
            for p in range(N):
                kids = np.nonzero(par == p)[0]
                if len(kids):
                    cand = np.argpartition(-d[p], len(kids))[:len(kids) + 1]
                    top = cand[np.lexsort((cand, -d[p][cand]))][:len(kids)]
                    tokens[b, kids] = top.astype(np.int32)

    _parallel(fill, B, seed, 2)
    return dict(target=target, parent=parent, node_tokens=tokens, kappa=kappa, dtype=dtype)


def make(name, greedy=False, **overrides):
    """Inputs of a named workload (see CONFIGS), optionally with overrides."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    if cfg["kind"] == "tree":
        return tree_inputs(**cfg)
    return chain_inputs(greedy=greedy, **cfg)


def logits_bytes(name, greedy=False):
    """Bytes of logits one verification step must read (the algorithmic bytes)."""
    c = CONFIGS[name]
    esz = 2 if c["dtype"] == "bf16" else 4
    if c["kind"] == "tree":
        return c["B"] * c["N"] * c["V"] * esz
    rows = c["B"] * (c["K"] + 1) + (0 if greedy else c["B"] * c["K"])
    return rows * c["V"] * esz
