"""Planted mistakes in copies of the oracle must be caught by the pins.

Each case copies oracle/spec_oracle.c, applies one plausible slip (wrong
residual, missing clamp, swapped ratio, dropped temperature, wrong tie rule,
walk that does not stop), builds it into a temporary library and shows that
a page-fixed check fails on it while it passes on the real oracle.
"""
import os

import numpy as np
import pytest

from oracle import build as oracle_build
from oracle import oracle as O
from tests.util import grid_chain_inputs
from workloads import synthetic as S

SRC = oracle_build.SRC

DVC_P, DVC_Q = [0.6, 0.3, 0.1], [0.2, 0.5, 0.3]
CRS_P, CRS_Q = [0.5, 0.3, 0.2], [0.2, 0.5, 0.3]


def _mutant(tmp_path, name, old, new, count=1):
    src = open(SRC).read()
    assert src.count(old) == count, f"mutation anchor for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle_build.build(str(path), str(tmp_path / f"lib{name}.so"), force=True)
    return O.lib(lib)


# residual spread over two tokens, (0, 0.2, 0.1) / 0.3; breakpoints are
# multiples of 1/60
SPLIT_P, SPLIT_Q = [0.1, 0.5, 0.4], [0.4, 0.3, 0.3]


def _law(L, p_list, q_list, p_bonus, T=1.0, n=30):
    inp, w = grid_chain_inputs(p_list, q_list, p_bonus, n=n, temperature=T)
    out = O.verify_chain(**inp, L=L)
    return out, w


def _first_token_law_ok(L, p, q, T=1.0, n=30):
    out, w = _law(L, [p], [q], p, T, n)
    law = np.bincount(out["out_tokens"][:, 0], weights=w, minlength=3)
    return np.allclose(law, p, atol=1e-9), law


def test_real_oracle_passes_every_check():
    assert _first_token_law_ok(None, DVC_P, DVC_Q)[0]
    assert _first_token_law_ok(None, CRS_P, CRS_Q, T=0.7)[0]


def test_naive_restart_is_caught(tmp_path, golden):
    """Why correcting a rejection is not resampling -- section 3: restarting from p
    on rejection yields (0.35, 0.39, 0.26)."""
    L = _mutant(tmp_path, "naive", "token = Z > 0.0 ? inverse_cdf(r, V,",
                "token = Z > 0.0 ? inverse_cdf(p, V,")
    ok, law = _first_token_law_ok(L, CRS_P, CRS_Q)
    assert not ok
    g = golden("crs_abc_example.json")
    np.testing.assert_allclose(law, g["naive_restart_law"], atol=1e-9)
    assert abs(np.abs(law - np.array(CRS_P)).max() - g["naive_restart_tv"]) < 1e-9


def test_missing_positive_part_is_caught(tmp_path):
    L = _mutant(tmp_path, "noclamp", "r[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;",
                "r[v] = p[v] - q[v];")
    # with the whole residual on one token the slip is invisible; a residual
    # spread over two tokens exposes it
    assert not _first_token_law_ok(L, SPLIT_P, SPLIT_Q, n=60)[0]
    assert _first_token_law_ok(None, SPLIT_P, SPLIT_Q, n=60)[0]


def test_swapped_ratio_is_caught(tmp_path):
    L = _mutant(tmp_path, "swap", "double ratio = p[y] / q[y];", "double ratio = q[y] / p[y];")
    assert not _first_token_law_ok(L, DVC_P, DVC_Q)[0]


def test_dropped_temperature_is_caught(tmp_path):
    L = _mutant(tmp_path, "notemp", "double x = logit_at(base, dtype, off + (size_t)v) / T;",
                "double x = logit_at(base, dtype, off + (size_t)v) / 1.0;", count=2)
    assert _first_token_law_ok(L, DVC_P, DVC_Q, T=1.0)[0]  # invisible at T = 1
    assert not _first_token_law_ok(L, DVC_P, DVC_Q, T=0.7)[0]


def test_walk_that_does_not_stop_is_caught(tmp_path):
    """Verify several proposed tokens in one target pass: stop at the first rejection."""
    L = _mutant(tmp_path, "nostop", "if (stop >= 0) continue; /* walk already stopped: diagnostics only */",
                "")
    out, w = _law(L, [DVC_P, CRS_P], [DVC_Q, CRS_Q], CRS_P)
    law0 = np.bincount(out["out_tokens"][:, 0], weights=w, minlength=3)
    ok0 = np.allclose(law0, DVC_P, atol=1e-9)
    ok_len = np.all(out["accepted_len"] <= 2)
    assert not (ok0 and ok_len)


def test_argmax_tie_rule_is_caught(tmp_path):
    L = _mutant(tmp_path, "tie", "    if (x > best) {\n      best = x;\n      idx = v;",
                "    if (x >= best) {\n      best = x;\n      idx = v;")
    t = np.zeros((1, 2, 8), np.float32)
    t[0, :, 2] = t[0, :, 5] = 1.0
    toks = np.array([[2]], np.int32)
    good = O.verify_chain(t, None, toks, mode=O.GREEDY)
    bad = O.verify_chain(t, None, toks, mode=O.GREEDY, L=L)
    assert good["accepted_len"][0] == 1 and bad["accepted_len"][0] == 0


def test_tree_tie_rule_is_caught(tmp_path):
    L = _mutant(tmp_path, "treetie", "if (acc[i] && depth[i] > depth[best]) best = i;",
                "if (acc[i] && depth[i] >= depth[best]) best = i;")
    t = np.zeros((1, 3, 4), np.float32)
    t[0, 0, 1] = 1.0  # argmax after the root is token 1
    par = np.array([[-1, 0, 0]], np.int32)
    toks = np.array([[0, 1, 1]], np.int32)  # two siblings with the same accepted token
    assert O.verify_tree(t, par, toks)["path_nodes"][0, 0] == 1
    assert O.verify_tree(t, par, toks, L=L)["path_nodes"][0, 0] == 2


# ---------------------------------------------- band bookkeeping (row_margin)
# The parity tests forgive a disagreement only where row_margin < 1e-5, so a
# slip that inflates or shrinks these margins must fail a pin.

def _split_row_margin(L, u_smp):
    p, q = [0.1, 0.5, 0.4], [0.4, 0.3, 0.3]
    tgt = np.stack([np.log(np.array(p)), np.log(np.array(p))]).astype(np.float32)[None]
    drf = np.log(np.array(q)).astype(np.float32)[None, None]
    out = O.verify_chain(tgt, drf, np.array([[0]], np.int32),
                         u_accept=np.array([[0.5]], np.float32),
                         u_sample=np.full((1, 2), u_smp, np.float32), L=L)
    return out["row_margin"][0]


def test_gap_far_edge_is_caught(tmp_path):
    """The gap is the distance to the NEARER end of the chosen interval."""
    L = _mutant(tmp_path, "gapmax", "double g = fmin(t - prev, c - t);",
                "double g = fmax(t - prev, c - t);")
    assert abs(_split_row_margin(None, 0.5) - 0.05 / 0.3) < 1e-7
    assert abs(_split_row_margin(L, 0.5) - 0.05 / 0.3) > 1e-3


def test_gap_not_relative_is_caught(tmp_path):
    """The gap is measured relative to the total mass Z."""
    L = _mutant(tmp_path, "gapabs", "*gap = total > 0.0 ? g / total : 0.0;",
                "*gap = total > 0.0 ? g : 0.0;")
    assert abs(_split_row_margin(L, 0.5) - 0.05 / 0.3) > 1e-3


def test_accept_margin_against_raw_ratio_is_caught(tmp_path):
    """The accept margin is taken against min(1, ratio), not the ratio."""
    L = _mutant(tmp_path, "rawratio", "fabs((double)u - fmin(1.0, ratio))",
                "fabs((double)u - ratio)")
    p, q = [0.6, 0.3, 0.1], [0.2, 0.5, 0.3]
    tgt = np.log(np.array([p, p])).astype(np.float32)[None]
    drf = np.log(np.array(q)).astype(np.float32)[None, None]
    kw = dict(u_accept=np.array([[0.75]], np.float32), u_sample=np.full((1, 2), 0.5, np.float32))
    good = O.verify_chain(tgt, drf, np.array([[0]], np.int32), **kw)
    bad = O.verify_chain(tgt, drf, np.array([[0]], np.int32), L=L, **kw)
    assert abs(good["accept_margin"][0, 0] - 0.25) < 1e-7
    assert abs(bad["accept_margin"][0, 0] - 0.25) > 1e-3


def test_row_margin_without_the_draw_gap_is_caught(tmp_path):
    """row_margin includes the gap of the draw at a rejection."""
    L = _mutant(tmp_path, "nogap", "          if (gap < margin) margin = gap;\n", "")
    assert abs(_split_row_margin(L, 0.5) - 0.05 / 0.3) > 1e-3
