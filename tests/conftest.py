import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built library")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(GOLDEN, name)) as f:
            return json.load(f)
    return load


@pytest.fixture(autouse=True)
def _no_bad_index(request):
    """In a bounds-check build of the library (-DSV_BOUNDS), every GPU test
    must leave the kernels' record of bad indexes empty.  The default build
    has no such record and this check does nothing."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    mod = sys.modules.get("speculative_decoding_verification_32_gb300._binding")
    if mod is None or mod._lib is None or not hasattr(mod._lib, "spec_debug_bounds"):
        return
    import ctypes
    count, line = ctypes.c_uint(0), ctypes.c_uint(0)
    fn = mod._lib.spec_debug_bounds
    fn.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_uint)]
    fn.restype = ctypes.c_int
    assert fn(ctypes.byref(count), ctypes.byref(line)) == 0
    assert count.value == 0, f"{count.value} bad indexes, the first at source line {line.value}"
