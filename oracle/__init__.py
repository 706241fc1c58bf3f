"""Oracle for the tensor-parallel layer forward -- TEST INFRASTRUCTURE ONLY.

Plain CPU numpy (float64) restatement of what the layer computes, used by the
tests, the smoke check and the CPU-baseline leg of the benchmark to judge the
CUDA library.  Nothing in the product imports it.
"""
from . import accounting, tp_layer  # noqa: F401
