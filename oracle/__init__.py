"""CPU oracle for the batch-1 decode step (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package. It shares no code with the CUDA engine.
"""
from .oracle import OracleModel, build_lib, lib, PLAIN, EXACT  # noqa: F401
