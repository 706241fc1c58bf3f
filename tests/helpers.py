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
