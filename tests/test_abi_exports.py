"""The C-ABI library builds on a machine without a GPU, loads, and exports every function that
include/adp.h declares (no compute call is made)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _names(text):
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return set(re.findall(r"\b(adp_[a-z0-9_]+)\s*\(", text))


def _declared(test_only=None):
    """Functions adp.h declares: all (None), only those inside its #ifdef ADP_TEST_HOOKS blocks
    (True), or all others (False)."""
    text = open(os.path.join(ROOT, "include", "adp.h")).read()
    hooks = "".join(re.findall(r"#ifdef ADP_TEST_HOOKS(.*?)#endif", text, flags=re.S))
    names, hook_names = _names(text), _names(hooks)
    assert len(names) > 20 and len(hook_names) == 3
    if test_only is None:
        return sorted(names)
    return sorted(hook_names if test_only else names - hook_names)


def test_release_library_exports_every_declared_function_but_the_test_hooks():
    from autoregressive_decode_persistent_gb300 import build
    lib = ctypes.CDLL(build.build())
    missing = [n for n in _declared(test_only=False) if not hasattr(lib, n)]
    assert not missing, missing
    present = [n for n in _declared(test_only=True) if hasattr(lib, n)]
    assert not present, present


def test_test_library_exports_every_declared_function():
    from autoregressive_decode_persistent_gb300 import build
    build.build()
    lib = ctypes.CDLL(build.TEST_LIB)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_loads_the_test_build_in_the_test_suite():
    from autoregressive_decode_persistent_gb300 import adp
    assert adp.default_library_path() == adp.TEST_LIB_PATH
    assert set(adp.TEST_HOOKS) == set(_declared(test_only=True))


def test_binding_wraps_every_declared_function():
    from autoregressive_decode_persistent_gb300 import adp
    bound = {name for name, _, _ in adp._SIGS}
    assert set(_declared()) <= bound, sorted(set(_declared()) - bound)


def test_status_strings_without_a_gpu():
    from autoregressive_decode_persistent_gb300 import adp, build
    build.build()
    assert adp.status_string(adp.ADP_OK) == "ok"
    assert "max_ctx" in adp.status_string(adp.ADP_ERR_CONTEXT_OVERFLOW)
