"""Oracle for the tensor-parallel layer forward -- TEST INFRASTRUCTURE ONLY.

Plain CPU numpy (float64) restatement of what the layer computes, used by the
tests, the smoke check and the CPU-baseline leg of the benchmark to check the
CUDA library against.  Nothing in the product imports it.  Modules: tp_layer
(the layer and its sharded forms), accounting (byte and flop counts),
vocab_head (the vocabulary-parallel lm_head), weight_int8 (weight-only int8).
"""
from . import accounting, tp_layer, vocab_head, weight_int8  # noqa: F401
