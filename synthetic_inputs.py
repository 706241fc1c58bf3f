"""Seeded synthetic inputs for the tensor-parallel layer workloads.

This module is the ONE piece shared by the oracle side (``oracle/``, tests) and
the CUDA side (tests, ``bench.py``).  It draws numbers and nothing else: it
holds none of the layer's arithmetic.

Generator
---------
Every element is a pure function of ``(seed, stream name, flat index)``, so any
subset of a tensor can be regenerated on the CPU without producing the rest,
and a tensor generated on the GPU is bit-identical to the same tensor
generated on the CPU:

* counter hash: Chris Wellons' ``lowbias32`` 32-bit integer mixer
  (xorshift-multiply-xorshift-multiply-xorshift, constants 0x7feb352d and
  0x846ca68b, "Prospecting for Hash Functions", 2018), applied to the element
  index and a per-tensor key.  Only integer operations, carried out in int64
  with every product kept below 2**48, so CPU and GPU agree exactly.
* approximately normal values: the Irwin-Hall construction -- the sum of four
  independent uniform 16-bit integers, centred and divided by its standard
  deviation sqrt((65536**2 - 1) / 3).  The integer sum is exact in fp32; one
  fp32 multiply by ``sigma / sd`` (IEEE round-to-nearest-even on both devices)
  and one cast to the target dtype (bf16 round-to-nearest-even) finish it.

The distribution has the mean and variance of N(0, sigma^2) and support
+-3.46 sigma; the workloads only fix the scale (N(0,1) activations, N(0,0.02)
or N(0,1)/sqrt(fan_in) weights), which this matches.
"""
from __future__ import annotations

import math
import zlib

import torch

_M32 = 0xFFFFFFFF
_SD4 = math.sqrt((65536.0 ** 2 - 1.0) / 3.0)   # std of a sum of four U{0..65535}
_MEAN4 = 2 * 65535                                # mean of that sum (exact integer)
_CHUNK = 1 << 25                                  # elements per generation chunk


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 0 <= x < 2**32; products stay below 2**48."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _mix32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    return x ^ (x >> 16)


def stream_key(seed: int, name: str) -> tuple[int, int]:
    """Two 32-bit keys for tensor ``name`` under ``seed``."""
    base = _mix32_int(_mix32_int(seed) ^ zlib.crc32(name.encode()))
    return _mix32_int(base ^ 0x632BE5AB), _mix32_int(base ^ 0x85157AF5)


def _normal_from_index(idx: torch.Tensor, keys: tuple[int, int], scale32: torch.Tensor) -> torch.Tensor:
    lo = idx & _M32
    hi = idx >> 32
    w0 = _mix32(_mix32(lo ^ keys[0]) ^ hi)
    w1 = _mix32(_mix32(lo ^ keys[1]) ^ hi)
    s = (w0 & 0xFFFF) + (w0 >> 16) + (w1 & 0xFFFF) + (w1 >> 16) - _MEAN4
    return s.to(torch.float32) * scale32


def normal(shape, sigma: float, seed: int, name: str, dtype=torch.bfloat16,
           device="cpu", index: torch.Tensor | None = None) -> torch.Tensor:
    """Tensor of ``shape`` with approximately N(0, sigma^2) entries.

    ``index`` (optional, int64) selects flat indices into the full tensor; the
    result then has ``index``'s shape and equals ``normal(shape, ...).flatten()[index]``
    bit for bit, without generating the rest.
    """
    keys = stream_key(seed, name)
    dev = torch.device(device)
    scale32 = torch.tensor(sigma / _SD4, dtype=torch.float32, device=dev)
    if index is not None:
        idx = index.to(device=dev, dtype=torch.int64)
        return _normal_from_index(idx, keys, scale32).to(dtype)
    n = math.prod(shape)
    out = torch.empty(n, dtype=dtype, device=dev)
    for start in range(0, n, _CHUNK):
        stop = min(n, start + _CHUNK)
        idx = torch.arange(start, stop, dtype=torch.int64, device=dev)
        out[start:stop] = _normal_from_index(idx, keys, scale32).to(dtype)
    return out.view(*shape)


def small_integers(shape, seed: int, name: str, lo: int = -2, hi: int = 2,
                   dtype=torch.bfloat16, device="cpu", zero_frac_num: int = 0) -> torch.Tensor:
    """Integer-valued tensor with entries uniform on {lo..hi} (exact in bf16/fp32).

    Used for bit-exact layout checks: sums of such products are exact in fp32.
    ``zero_frac_num``/16 of the entries (chosen by hash) are forced to zero.
    """
    keys = stream_key(seed, name)
    dev = torch.device(device)
    n = math.prod(shape)
    idx = torch.arange(n, dtype=torch.int64, device=dev)
    w = _mix32(_mix32((idx & _M32) ^ keys[0]) ^ (idx >> 32))
    v = (w % (hi - lo + 1)) + lo
    if zero_frac_num:
        z = _mix32(_mix32((idx & _M32) ^ keys[1]) ^ (idx >> 32)) & 15
        v = torch.where(z < zero_frac_num, torch.zeros_like(v), v)
    return v.to(dtype).view(*shape)


# --------------------------------------------------------------------------
# Workload recipes.  Draw order and names are fixed; every tensor has its own
# stream, so regenerating one never depends on the others.
# --------------------------------------------------------------------------

def tiny_mlp(seed: int = 0, device="cpu"):
    """Tiny Megatron MLP: X[8,256] fp32, Wg/Wu stored [1024,256], Wd stored [256,1024].

    X ~ N(0,1); weights ~ N(0,1)/sqrt(fan_in); fp32; tp = 2.
    """
    B, D, F = 8, 256, 1024
    f32 = torch.float32
    return dict(
        X=normal((B, D), 1.0, seed, "tiny.X", f32, device),
        Wg=normal((F, D), 1.0 / math.sqrt(D), seed, "tiny.Wg", f32, device),
        Wu=normal((F, D), 1.0 / math.sqrt(D), seed, "tiny.Wu", f32, device),
        Wd=normal((D, F), 1.0 / math.sqrt(F), seed, "tiny.Wd", f32, device),
        B=B, D=D, F=F, tp=2)


QWEN_DECODE = dict(D=1536, F=8960, n_q=12, n_kv=2, head_dim=128, tp=2, batches=(1, 8, 32, 64),
                   n_layers=28)
LLAMA_PREFILL = dict(B=4096, D=8192, F=28672, tp=8)
LLAMA_DECODE = dict(D=8192, F=28672, n_q=64, n_kv=8, head_dim=128, tp=8, batches=(1, 8, 32, 128),
                    n_layers=8)
SHARDED_CASES = dict(I=512, J=8192, K=28672, X=8)


def layer_weights(D, F, n_q, n_kv, head_dim, seed=0, layer=0, prefix="layer", sigma=0.02,
                  device="cpu", dtype=torch.bfloat16):
    """One transformer layer's projection weights, all stored [out, in] row-major.

    Wqkv [(n_q + 2 n_kv) head_dim, D] with rows [Q heads | K heads | V heads],
    Wo [D, n_q head_dim], Wg/Wu [F, D], Wd [D, F]; entries ~ N(0, sigma^2).
    """
    p = f"{prefix}{layer}"
    nqkv = (n_q + 2 * n_kv) * head_dim
    return dict(
        Wqkv=normal((nqkv, D), sigma, seed, p + ".Wqkv", dtype, device),
        Wo=normal((D, n_q * head_dim), sigma, seed, p + ".Wo", dtype, device),
        Wg=normal((F, D), sigma, seed, p + ".Wg", dtype, device),
        Wu=normal((F, D), sigma, seed, p + ".Wu", dtype, device),
        Wd=normal((D, F), sigma, seed, p + ".Wd", dtype, device))


def activations(B, D, seed=0, name="X", device="cpu", dtype=torch.bfloat16):
    """Token activations X[B, D] ~ N(0,1)."""
    return normal((B, D), 1.0, seed, name, dtype, device)


def lm_head(B, D, V, seed=0, device="cpu", dtype=torch.bfloat16, sigma=0.02):
    """Final hidden states x[B, D] ~ N(0,1) (unit rms, as after the final
    RMSNorm) and an lm_head weight W[V, D] ~ N(0, sigma^2)."""
    return (normal((B, D), 1.0, seed, "lm_head.x", dtype, device),
            normal((V, D), sigma, seed, "lm_head.W", dtype, device))


def sharded_case_operands(I, J, K, seed=0, device="cpu", dtype=torch.bfloat16):
    """A[I,J] ~ N(0,1) and B[J,K] ~ N(0,1)/sqrt(J), B stored transposed as Bt[K,J]."""
    return dict(A=normal((I, J), 1.0, seed, "cases.A", dtype, device),
                Bt=normal((K, J), 1.0 / math.sqrt(J), seed, "cases.Bt", dtype, device))


def prefill_mlp(B, D, F, seed=0, device="cpu", dtype=torch.bfloat16):
    """Prefill MLP operands: X[B,D] ~ N(0,1); Wg/Wu [F,D], Wd [D,F] ~ N(0,0.02)."""
    return dict(X=normal((B, D), 1.0, seed, "prefill.X", dtype, device),
                Wg=normal((F, D), 0.02, seed, "prefill.Wg", dtype, device),
                Wu=normal((F, D), 0.02, seed, "prefill.Wu", dtype, device),
                Wd=normal((D, F), 0.02, seed, "prefill.Wd", dtype, device))
