"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before touching CUDA (runs without a GPU)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verification_32_gb300 import build as lib_build
    from speculative_decoding_verification_32_gb300 import _binding

    lib_build.build()
    return _binding.lib()


def declared_functions(bounds=False):
    """Entry points the header declares; those under #ifdef SV_BOUNDS exist
    only in the bounds-check build (bounds=True: only those)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    guarded = "".join(re.findall(r"#ifdef SV_BOUNDS(.*?)#endif", text, flags=re.S))
    if bounds:
        text = guarded
    else:
        text = re.sub(r"#ifdef SV_BOUNDS.*?#endif", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "spec_verify_chain" in names and "spec_verify_tree" in names
    assert "spec_rollback_lengths" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in specverify.h but not exported"
    for n in declared_functions(bounds=True):  # bounds-check builds only
        assert not hasattr(L, n), f"{n} exported by the default build"


def test_bounds_build_exports_its_extra_entry_points():
    from speculative_decoding_verification_32_gb300 import build as lib_build
    B = ctypes.CDLL(lib_build.build(variant="bounds"))
    names = declared_functions(bounds=True)
    assert names == ["spec_debug_bounds", "spec_debug_bounds_selftest"]
    for n in names + declared_functions():
        assert hasattr(B, n), f"{n} not exported by the bounds-check build"


def test_status_strings(L):
    for code in range(8):
        s = L.spec_status_string(code).decode()
        assert s.startswith("SPEC_")


def test_workspace_sizes(L):
    assert L.spec_verify_chain_workspace_size(64, 5, 128256) > 64 * 6 * 16
    assert L.spec_verify_chain_workspace_size(0, 5, 100) >= 0
    assert L.spec_verify_chain_workspace_size(-1, 5, 100) == 0
    assert L.spec_verify_chain_workspace_size(4, -1, 100) == 0
    assert L.spec_verify_chain_workspace_size(4, 5, 0) == 0
    assert L.spec_verify_chain_workspace_size(4, 5, 262145) == 0
    assert L.spec_verify_tree_workspace_size(32, 60, 151936) > 32 * 60 * 16
    assert L.spec_verify_tree_workspace_size(32, 0, 100) == 0
    assert L.spec_verify_tree_workspace_size(32, 1025, 100) == 0


def test_truncated_workspace_holds_the_lists(L):
    """A truncated call lays out, each area 256-byte aligned: one record per
    (logit row, ring tile), the draft-token logits, the truncation records
    a 2-byte chunk maximum per (logit row, tile, consumer thread of 256) and
    a kept list of 64 8-byte entries per target row, with the 16-byte header
    in the last 256 bytes.  The size covers that for
    bf16 (8192-logit) and fp32 (4096-logit) tiles, and a truncated workspace
    also serves a plain call."""
    def al(x):
        return -(-x // 256) * 256
    for B, K, V in [(64, 5, 128256), (1, 0, 1), (3, 63, 4099), (256, 8, 262144), (5, 2, 8193)]:
        rows = B * (2 * K + 1)
        need = L.spec_verify_chain_truncated_workspace_size(B, K, V)
        assert need >= L.spec_verify_chain_workspace_size(B, K, V)
        for tile in (8192, 4096):
            nt = -(-V // tile)
            used = (al(rows * nt * 16) + al(rows * 8) + al(rows * 16) + al(rows * nt * 256 * 2) +
                    B * (K + 1) * 64 * 8 + 256)
            assert need >= used, (B, K, V, tile)
    assert L.spec_verify_chain_truncated_workspace_size(-1, 5, 100) == 0
    assert L.spec_verify_chain_truncated_workspace_size(4, -1, 100) == 0
    assert L.spec_verify_chain_truncated_workspace_size(4, 5, 262145) == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


def _chain_args(B=2, K=3, V=1000, dtype=1, mode=0, kappa=0.0, base=0x10000000):
    from speculative_decoding_verification_32_gb300._binding import SpecChainArgs, SpecChainOut
    a = SpecChainArgs(B, K, V, dtype, mode, kappa, _fake(base), _fake(base + 0x100000),
                      _fake(base + 0x200000), None, _fake(base + 0x300000), _fake(base + 0x400000))
    o = SpecChainOut(_fake(base + 0x500000), _fake(base + 0x600000), _fake(base + 0x700000),
                     _fake(base + 0x800000), None, None, None)
    return a, o


def test_chain_argument_errors_return_before_cuda(L):
    ws = _fake(0x20000000)
    big = 1 << 30
    a, o = _chain_args()
    assert L.spec_verify_chain(None, ctypes.byref(o), ws, big, None) == 1
    a, o = _chain_args(B=-1)
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 2
    a, o = _chain_args(K=2000)
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 2
    a, o = _chain_args(V=0)
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 2
    a, o = _chain_args(dtype=7)
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 3
    a, o = _chain_args(mode=3)
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 3
    a, o = _chain_args(kappa=float("nan"))
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 5
    a, o = _chain_args()
    a.u_sample = None
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 1
    a, o = _chain_args()
    o.row_status = None
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 1
    a, o = _chain_args()
    a.target_logits = _fake(0x10000001)  # bf16 needs 2-byte alignment
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 4
    a, o = _chain_args()
    a.draft_tokens = _fake(0x10000002)
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 4
    a, o = _chain_args()
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), None, big, None) == 7
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), _fake(0x20000010), big, None) == 7
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, 16, None) == 7
    # greedy mode does not need draft logits or uniforms, but needs tokens
    a, o = _chain_args(mode=1)
    a.draft_tokens = None
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 1
    # B == 0 is a valid no-op that never touches the device
    a, o = _chain_args(B=0)
    assert L.spec_verify_chain(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 0


def test_tree_and_rollback_argument_errors(L):
    from speculative_decoding_verification_32_gb300._binding import SpecTreeArgs, SpecTreeOut
    ws = _fake(0x20000000)
    big = 1 << 30
    b = 0x10000000

    def tree(N=8, V=100, dtype=1):
        a = SpecTreeArgs(2, N, V, dtype, 0.3, _fake(b), _fake(b + 0x1000), _fake(b + 0x2000), None)
        o = SpecTreeOut(_fake(b + 0x3000), _fake(b + 0x4000), _fake(b + 0x5000),
                        _fake(b + 0x6000), _fake(b + 0x7000))
        return a, o
    a, o = tree(N=0)
    assert L.spec_verify_tree(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 2
    a, o = tree(N=1025)
    assert L.spec_verify_tree(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 2
    a, o = tree(dtype=2)
    assert L.spec_verify_tree(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 3
    a, o = tree()
    a.parent = None
    assert L.spec_verify_tree(ctypes.byref(a), ctypes.byref(o), ws, big, None) == 1
    a, o = tree()
    assert L.spec_verify_tree(ctypes.byref(a), ctypes.byref(o), ws, 8, None) == 7
    p = _fake(b)
    assert L.spec_rollback_lengths(-1, 4, p, p, p, p, -1, None, p, p, None) == 2
    assert L.spec_rollback_lengths(2, 0, p, p, p, p, -1, None, p, p, None) == 2
    assert L.spec_rollback_lengths(2, 4, None, p, p, p, -1, None, p, p, None) == 1
    assert L.spec_rollback_lengths(2, 4, _fake(b + 2), p, p, p, -1, None, p, p, None) == 4
    assert L.spec_rollback_lengths(0, 4, p, p, p, p, -1, None, p, p, None) == 0


def test_wait_timeout_setting(L):
    old = L.spec_get_wait_timeout_ns()
    L.spec_set_wait_timeout_ns(12345)
    assert L.spec_get_wait_timeout_ns() == 12345
    L.spec_set_wait_timeout_ns(old)


def test_product_path_never_imports_the_oracle():
    """The package and its C sources name nothing under oracle/."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_32_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "spec_oracle" not in text and "so_verify" not in text, f


def test_kv_compact_and_policy_argument_errors(L):
    from speculative_decoding_verification_32_gb300._binding import (SpecAdaptiveParams,
                                                                      SpecKvCompactArgs)
    b = 0x10000000
    p = _fake(b)

    def kv(B=2, N=8, planes=2, E=256, kvp=b, ts=256):
        return SpecKvCompactArgs(B, N, planes, 0, 64, E, 2 * 64 * E, 64 * E, ts, _fake(kvp),
                                 p, p, p)
    assert L.spec_kv_compact_tree(None, None, None) == 1
    assert L.spec_kv_compact_tree(ctypes.byref(kv(N=0)), None, None) == 2
    assert L.spec_kv_compact_tree(ctypes.byref(kv(B=-1)), None, None) == 2
    assert L.spec_kv_compact_tree(ctypes.byref(kv(kvp=b + 8)), None, None) == 4
    assert L.spec_kv_compact_tree(ctypes.byref(kv(E=24)), None, None) == 4
    assert L.spec_kv_compact_tree(ctypes.byref(kv(ts=100)), None, None) == 4
    a = kv()
    a.path_nodes = None
    assert L.spec_kv_compact_tree(ctypes.byref(a), None, None) == 1
    assert L.spec_kv_compact_tree(ctypes.byref(kv(B=0)), None, None) == 0

    def par(alpha=0.3, d=1.0, e0=0.0, brk=5):
        t3 = ctypes.c_int32 * 3
        return SpecAdaptiveParams(alpha, d, e0, t3(3, 4, 4), t3(7, 1, 8), t3(3, 4, 4), brk)
    args = (p, p, p, p, p, p, None)
    assert L.spec_adaptive_tree_policy(None, 4, *args) == 1
    assert L.spec_adaptive_tree_policy(ctypes.byref(par()), -1, *args) == 2
    assert L.spec_adaptive_tree_policy(ctypes.byref(par(alpha=1.5)), 4, *args) == 5
    assert L.spec_adaptive_tree_policy(ctypes.byref(par(d=0.0)), 4, *args) == 5
    assert L.spec_adaptive_tree_policy(ctypes.byref(par(d=float("inf"))), 4, *args) == 5
    assert L.spec_adaptive_tree_policy(ctypes.byref(par(brk=0)), 4, *args) == 5
    assert L.spec_adaptive_tree_policy(ctypes.byref(par()), 4, None, p, p, p, p, p, None) == 1
    assert L.spec_adaptive_tree_policy(ctypes.byref(par()), 4, p, p, p, _fake(b + 4), p, p,
                                       None) == 4  # ema needs 8-byte alignment
    assert L.spec_adaptive_tree_policy(ctypes.byref(par()), 0, *args) == 0


def test_drift_argument_errors(L):
    from speculative_decoding_verification_32_gb300._binding import SpecChainArgs
    b = 0x10000000
    p = _fake(b)
    ws = _fake(0x20000000)
    big = 1 << 30

    def args(B=2, K=3, V=1000):
        return SpecChainArgs(B, K, V, 1, 0, 0.0, p, _fake(b + 0x100000), None, None, None, None)
    o = (p, p, p, ws, big, None)
    assert L.spec_drift_residuals(None, 8, *o) == 1
    assert L.spec_drift_residuals(ctypes.byref(args(K=65)), 8, *o) == 2
    assert L.spec_drift_residuals(ctypes.byref(args()), 0, *o) == 5
    assert L.spec_drift_residuals(ctypes.byref(args()), 65, *o) == 5
    assert L.spec_drift_residuals(ctypes.byref(args(V=20)), 32, *o) == 5
    assert L.spec_drift_residuals(ctypes.byref(args(B=0)), 8, *o) == 0
    assert L.spec_drift_residuals(ctypes.byref(args(K=0)), 8, *o) == 0
    assert L.spec_drift_residuals(ctypes.byref(args()), 8, None, p, p, ws, big, None) == 1
    assert L.spec_drift_residuals(ctypes.byref(args()), 8, p, p, p, ws, 16, None) == 7
