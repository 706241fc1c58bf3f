"""Oracle for weight-only int8 decode -- TEST INFRASTRUCTURE ONLY.

Plain CPU restatement of the CUDA path's weight-only int8 MLP.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the product path never does, and it shares no code
with the CUDA library.

Source: [L4] "Lecture 4 - Distributed Serving" (CS349E notes), S5.5 "other
techniques and end-to-end results": int8 weights -- only the weights are
quantised, which saves the time spent reading them (PaLM 540B decode at B = 64:
28.5 ms per token with int8 weights against 36.9 ms in bf16); S6.2: the cheapest
configurations are the ones whose weights take half the bytes.

Readings where the section is silent:
  * Symmetric per-row quantisation: a row of W (one output feature) is split
    into `groups` contiguous column groups -- one per tensor-parallel shard for
    a row-parallel weight, so every device quantises only what it holds -- and
    each group gets the scale s = amax / 127 with q = round(w / s), ties to
    even, clamped to [-127, 127] (q = 0 where amax = 0).
  * These are decisions on floating-point values, so they are taken in the
    precision the kernel uses: amax, s and w / s in IEEE float32 (correctly
    rounded division), then rounding to the nearest integer.
  * Activations stay bf16 and the arithmetic is that of the bf16 path with the
    weights replaced by their dequantised values q * s: the layer computes
    exactly mlp_sharded(X, q_g * s_g, q_u * s_u, q_d * s_d) of the tp_layer
    oracle (the SwiGLU output rounded to bf16, partials fp32, shards summed in
    ascending order).
"""
from __future__ import annotations

import numpy as np

from oracle import tp_layer as O

QMAX = 127


def quantize_rows(W, groups: int = 1):
    """Per-(row, column group) symmetric int8 quantisation of W [rows, cols].

    Returns (q int8 [rows, cols], scale float32 [rows, groups])."""
    W32 = np.asarray(W, dtype=np.float32)
    rows, cols = W32.shape
    if groups < 1 or cols % groups:
        raise ValueError("cols must divide into groups")
    g = W32.reshape(rows, groups, cols // groups)
    amax = np.max(np.abs(g), axis=2)                                   # exact in float32
    scale = (amax / np.float32(QMAX)).astype(np.float32)              # one IEEE float32 division
    safe = np.where(scale > 0, scale, np.float32(1))
    ratio = (g / safe[:, :, None]).astype(np.float32)                 # IEEE float32 division
    q = np.clip(np.rint(ratio), -QMAX, QMAX)                          # rint: ties to even
    q = np.where(scale[:, :, None] > 0, q, 0)
    return q.reshape(rows, cols).astype(np.int8), scale


def dequantize_rows(q, scale):
    """q * s per (row, group), exactly (float64 holds every product)."""
    q = np.asarray(q, dtype=np.float64)
    rows, cols = q.shape
    groups = scale.shape[1]
    s = np.repeat(np.asarray(scale, dtype=np.float64), cols // groups, axis=1)
    return q * s


def mlp_sharded_w8(X, Qg, sg, Qu, su, Qd, sd, tp: int, bf16: bool = True):
    """The sharded SwiGLU MLP with int8 weights and bf16 activations: the
    tp_layer oracle's mlp_sharded on the dequantised weights.  Returns
    (Y, [P_0..P_{tp-1}], [H_0..H_{tp-1}])."""
    return O.mlp_sharded(X, dequantize_rows(Qg, sg), dequantize_rows(Qu, su), dequantize_rows(Qd, sd), tp,
                         bf16=bf16)


def weight_bytes_int8(D: int, F: int, tp: int) -> int:
    """Bytes one MLP forward reads with int8 weights: three D x F matrices of
    one byte per weight, plus the float32 scales (F + F per-row, D x tp)."""
    return 3 * D * F + 4 * (2 * F + D * tp)
