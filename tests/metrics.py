"""Comparison metric used by every parity test.

max |GPU - oracle| over all compared elements, divided by the RMS of the
oracle's values over the same elements.  Bounds: 1e-4 for float32 inputs and
2e-2 for bfloat16 inputs with float32 accumulation; 1e-4 for the gradients,
which are computed in float32 for either input dtype.
"""
import numpy as np

TOL_F32 = 1e-4
TOL_BF16 = 2e-2
# Gradients of the causal form: fp32 arithmetic for both input dtypes (bf16
# inputs are exact in fp32), so the float32 bound applies to both.
TOL_BWD = 1e-4


def rel_max_err(got, ref) -> float:
    got = np.asarray(got.detach().cpu().double() if hasattr(got, "detach") else got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    assert np.isfinite(got).all(), "non-finite GPU output"
    rms = np.sqrt((ref ** 2).mean())
    return float(np.abs(got - ref).max() / max(rms, 1e-300))


def tol_for(dtype) -> float:
    import torch
    return TOL_F32 if dtype == torch.float32 else TOL_BF16
