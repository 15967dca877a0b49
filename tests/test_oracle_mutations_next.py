"""Planted mistakes in the oracle's next-row functions must be caught.

Like the verifier's mutation tests: each case copies oracle/spec_oracle.c,
applies one plausible slip to the truncated verifier, the DRIFT residuals,
the KV path compaction, the tree-shape policy or the rollback lengths,
builds it into a temporary library, and runs one of the page-fixed pins
against it.  The pin must fail on the mutant (it passes on the real oracle
in its own file).
"""
import pytest

from oracle import build as oracle_build
from oracle import oracle as O
from tests import test_oracle_next as NEXT
from tests import test_oracle_pins as PINS
from tests import test_oracle_trunc as TRUNC

SRC = oracle_build.SRC


@pytest.fixture
def mutant(tmp_path, monkeypatch):
    """Build a mutant and make it the library every oracle call loads."""
    def make(name, old, new, count=1):
        src = open(SRC).read()
        assert src.count(old) == count, f"mutation anchor for {name} not found"
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(old, new))
        L = O.lib(oracle_build.build(str(path), str(tmp_path / f"lib{name}.so"), force=True))
        monkeypatch.setattr(O, "lib", lambda path=None: L)
    return make


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


# --------------------------------------------------- truncated verification
def test_strict_threshold_drops_boundary_ties(mutant):
    mutant("strict", "if (logit_at(base, dtype, off + (size_t)v) >= theta) S += p[v];",
           "if (logit_at(base, dtype, off + (size_t)v) > theta) S += p[v];")
    _fails(TRUNC.test_top_k_keeps_boundary_ties)


def test_missing_renormalisation_is_caught(mutant):
    mutant("norenorm", "    else p[v] = 0.0;\n  }\n  for (int v = 0; v < V; ++v) p[v] /= S;\n",
           "    else p[v] = 0.0;\n  }\n")
    _fails(TRUNC.test_truncated_worked_example, dict(top_k=[2] * 4))


def test_top_p_one_group_too_many_is_caught(mutant):
    mutant("pgroup", "if (cum >= top_p || e == n) {", "if (before >= top_p || e == n) {")
    _fails(TRUNC.test_truncated_worked_example, dict(top_p=[0.7] * 4))


def test_top_p_on_the_law_before_top_k_is_caught(mutant):
    mutant("pmass", "cum += g / mass;", "cum += g;")
    _fails(TRUNC.test_top_k_then_top_p_on_the_renormalised_law)


# ------------------------------------------------------- DRIFT residuals
def test_drift_residual_sign_is_caught(mutant):
    mutant("dsign", "res[i] = (float)(lp[best] - lq[best]);", "res[i] = (float)(lq[best] - lp[best]);")
    _fails(NEXT.test_drift_residual_closed_form, 1.0)


def test_drift_dropped_temperature_is_caught(mutant):
    mutant("dtemp", "const double xs = logit_at(base, dtype, off + (size_t)v) / T;",
           "const double xs = logit_at(base, dtype, off + (size_t)v);", count=3)
    _fails(NEXT.test_drift_residual_closed_form, 0.7)


def test_drift_ties_to_the_higher_index_are_caught(mutant):
    mutant("dties", "if (best < 0 || x > bv) {", "if (best < 0 || x >= bv) {")
    _fails(NEXT.test_drift_residual_closed_form, 1.0)


# ---------------------------------------------------------- KV compaction
def test_kv_destination_off_by_one_is_caught(mutant):
    mutant("kvslot", "memcpy(row + (size_t)(base + 1 + k) * tok_stride,",
           "memcpy(row + (size_t)(base + k) * tok_stride,")
    _fails(NEXT.test_kv_compaction_moves_each_path_entry_to_its_slot)


def test_kv_repeated_path_node_is_caught(mutant):
    mutant("kvrepeat", "if (n <= prev || n >= N) ok = 0;", "if (n < prev || n >= N) ok = 0;")
    _fails(NEXT.test_kv_compaction_rejects_bad_paths_and_skips_failed_rows)


# ----------------------------------------------------- tree-shape policy
def test_policy_swapped_ema_weights_are_caught(mutant):
    mutant("ema", "const double e = alpha * a + (1.0 - alpha) * ema[b];",
           "const double e = (1.0 - alpha) * a + alpha * ema[b];")
    _fails(NEXT.test_policy_ema_closed_form)


def test_policy_breaker_one_step_late_is_caught(mutant):
    mutant("breaker", "if (z >= breaker) {", "if (z > breaker) {")
    _fails(NEXT.test_policy_circuit_breaker_after_five_zero_accept_steps)


def test_policy_score_without_the_divisor_is_caught(mutant):
    mutant("divisor", "double dcs = p1 * e / divisor;", "double dcs = p1 * e;")
    _fails(NEXT.test_policy_divisor_saturates_the_score)


# ------------------------------------------------------- rollback lengths
def test_rollback_dropping_the_eos_token_is_caught(mutant):
    mutant("eos", "          n = e + 1;\n", "          n = e;\n")
    _fails(PINS.test_rollback_lengths_cases)


def test_rollback_room_without_the_root_is_caught(mutant):
    mutant("room", "long room = (long)max_len[b] - ((long)kv_len_in[b] + 1);",
           "long room = (long)max_len[b] - (long)kv_len_in[b];")
    _fails(PINS.test_rollback_lengths_cases)
