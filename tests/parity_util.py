"""Helpers for GPU-vs-oracle parity: the error metric and its tolerances.

Metric (per output element): |gpu - oracle| / sum over the taps of |a|*|b|, i.e. the error
normalised by the sum of absolute products that formed that output (for the forward pass
sum |x||w|, for backward data sum |dy||w|, for the filter gradient sum |x||dy|).  The
denominator is the same convolution evaluated by the oracle on absolute values.  Elements
with no valid tap (denominator 0) must be exactly zero.

Tolerances: 1e-5 for fp32 inputs and 1e-2 for bf16/fp16 inputs, with fp32 accumulation in
both cases.  The bound is far above what fp32 accumulation of these sums produces (about
n * 2^-24 in the worst case for n terms, typically much less), so a wrong tap, index or
sign fails it while any correct summation order passes.
"""
import numpy as np

TOL = {"f32": 1e-5, "bf16": 1e-2, "f16": 1e-2}


def normalized_error(gpu, ref, denom):
    gpu = np.asarray(gpu, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    denom = np.asarray(denom, dtype=np.float64).ravel()
    assert gpu.shape == ref.shape == denom.shape
    assert np.all(np.isfinite(gpu)), "non-finite GPU output"
    zero = denom == 0
    if np.any(zero):
        assert np.all(gpu[zero] == 0.0), "output with no valid tap is not zero"
    if np.all(zero):
        return 0.0
    return float(np.max(np.abs(gpu[~zero] - ref[~zero]) / denom[~zero]))


def mare(gpu, ref):
    """Mean absolute relative error (the pages' accuracy metric, reported alongside)."""
    gpu = np.asarray(gpu, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    nz = ref != 0
    return float(np.mean(np.abs(gpu[nz] - ref[nz]) / np.abs(ref[nz]))) if np.any(nz) else 0.0
