"""The C-ABI library builds on a machine without a GPU, loads, and exports every function that
include/adp.h declares (no compute call is made)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "adp.h")).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    names = set(re.findall(r"\b(adp_[a-z0-9_]+)\s*\(", text))
    assert len(names) > 20
    return sorted(names)


def test_library_exports_every_declared_function():
    from autoregressive_decode_persistent_gb300 import build
    lib = ctypes.CDLL(build.build())
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_wraps_every_declared_function():
    from autoregressive_decode_persistent_gb300 import adp
    bound = {name for name, _, _ in adp._SIGS}
    assert set(_declared()) <= bound, sorted(set(_declared()) - bound)


def test_status_strings_without_a_gpu():
    from autoregressive_decode_persistent_gb300 import adp, build
    build.build()
    assert adp.status_string(adp.ADP_OK) == "ok"
    assert "max_ctx" in adp.status_string(adp.ADP_ERR_CONTEXT_OVERFLOW)
