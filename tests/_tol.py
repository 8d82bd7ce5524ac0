"""Parity tolerance for bf16-input / fp32-accumulate results against the float64 oracle.

max |gpu - ref| <= 2e-2 * max |ref|   and   sum |gpu - ref| / sum |ref| <= 5e-3
(the second is the "mean relative error", read as an L1 ratio because the
per-element relative error is unstable near zero).
"""
import numpy as np

MAX_REL = 2e-2
MEAN_REL = 5e-3


def parity(gpu, ref, name="", max_rel=MAX_REL, mean_rel=MEAN_REL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    fin = np.isfinite(ref)
    # infinities (empty rows: lse = -inf) must match exactly
    assert np.array_equal(np.isneginf(gpu), np.isneginf(ref)), f"{name}: -inf pattern differs"
    assert np.all(np.isfinite(gpu[fin])), f"{name}: non-finite values where the oracle is finite"
    if not fin.any():
        return 0.0, 0.0
    err = np.abs(gpu[fin] - ref[fin])
    denom_max = np.max(np.abs(ref[fin]))
    denom_sum = np.sum(np.abs(ref[fin]))
    e_max = float(np.max(err) / denom_max) if denom_max > 0 else float(np.max(err))
    e_mean = float(np.sum(err) / denom_sum) if denom_sum > 0 else float(np.sum(err))
    assert e_max <= max_rel, f"{name}: max rel err {e_max:.3e} > {max_rel}"
    assert e_mean <= mean_rel, f"{name}: mean rel err {e_mean:.3e} > {mean_rel}"
    return e_max, e_mean
