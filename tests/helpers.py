"""Shared test helpers: tolerance checks and device/host transfers.

Tolerances
----------
* bf16 inputs, fp32 accumulation (the stated bar): max |y - y_oracle| <=
  1e-2 * rms(y_oracle), checked on UNROUNDED fp32 results (out_dtype=float32,
  or fp32 partial sums).
* bf16 outputs add their own final rounding, at most half a bf16 ulp, i.e.
  2**-8 |y| (one ulp is at most 2**-7 |y|): bound 1e-2 rms + 2**-8 |y_oracle|.
* fp32 path (the tiny fp32 MLP): 1e-5 * rms, far above fp32 accumulation
  error for dot products of length <= 1024 (about sqrt(n) * 2**-24 relative).
* stacks of decoder layers (bf16 residual stream): the stated bar for the
  accumulated fp32 error, plus, for every bf16 rounding of the residual stream
  (h and y of each layer), the most two roundings of nearby values can differ
  by beyond their inputs' difference: 2**-8 (|a| + |b|) ~ 2**-7 |r|, with r
  the oracle's rounded residual value at that point.  A one-ulp flip of the
  residual stream passes unchanged through the identity path to the output,
  so these terms add up over the layers (see ``stack_allowance``).
"""
import numpy as np
import torch

BF16_REL = 1e-2
F32_REL = 1e-5


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rms(a) -> float:
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a)))


def stack_allowance(trace, y_ref, rel=BF16_REL):
    """Per-element bound for a decoder stack's bf16 output against the oracle's
    bf16 output: rel * rms(y) + 2**-7 * sum over the residual-stream roundings
    (``trace`` from the oracle's decoder_stack, ending with y itself) of |r|."""
    y_ref = np.asarray(y_ref, np.float64)
    mag = np.zeros_like(y_ref)
    for r in trace:
        mag += np.abs(np.asarray(r, np.float64))
    return rel * rms(y_ref) + 2.0 ** -7 * mag


def assert_within(got, ref, allow, what=""):
    g = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bad = err > allow
    r = rms(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} outside tolerance; "
                           f"max|err|/rms = {float(err.max() / max(r, 1e-300)):.3e}")
    return float(err.max() / max(r, 1e-300))


def assert_close(got, ref, rel=BF16_REL, bf16_out=False, what=""):
    g = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    r = rms(ref)
    allow = rel * r + (2.0 ** -8 * np.abs(ref) if bf16_out else 0.0)
    err = np.abs(g - ref)
    bad = err > allow
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} outside tolerance; "
                           f"max|err|/rms = {float(err.max() / max(r, 1e-300)):.3e}")
    return float(err.max() / max(r, 1e-300))


def assert_equal(got, ref, what=""):
    g = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    diff = g != ref
    assert not diff.any(), f"{what}: {int(diff.sum())} of {g.size} elements differ"
