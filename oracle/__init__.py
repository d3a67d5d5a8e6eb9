"""CPU oracle for head-routed attention: TEST INFRASTRUCTURE ONLY.

Only the tests, the package entry point's smoke check and the benchmark's
CPU-baseline / reference arm may import anything here.  The CUDA library
never does, and the oracle never imports the library.

  headcast_ref  vectorised fp64 NumPy restatement of the method
  brute         pure-Python scalar twin for tiny inputs (key sets decided by
                a per-key predicate rather than by index lists)
"""
from . import headcast_ref, brute  # noqa: F401
