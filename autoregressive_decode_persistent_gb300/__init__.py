"""Batch-1 persistent decode engine for one GB300 (sm_103a).

The C ABI lives in include/adp.h and libadp.so (built in-tree by `build.build()`);
`adp` is its ctypes binding with the same names, `model` a thin convenience layer that
uploads weights with PyTorch. `bound` is the pages' bandwidth bound and byte calculator.
"""
from . import bound  # noqa: F401

__all__ = ["adp", "bound", "build", "model"]
