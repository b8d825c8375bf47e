"""Shared helpers for GPU-vs-oracle parity tests.

Tolerances are the ones the method's benchmark set states for bf16 outputs:
max |out - ref| <= 2e-2, mean |out - ref| <= 2e-3, and |lse - ref| <= 1e-3
(natural log).  An lse of -inf must match -inf exactly.
"""
import numpy as np

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_TOL = 1e-3


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    out = np.asarray(out, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64)
    assert out.shape == ref_out.shape, (what, out.shape, ref_out.shape)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    diff = np.abs(out - ref_out)
    assert diff.max() <= MAX_ABS, f"{what}: max abs error {diff.max():.3e}"
    assert diff.mean() <= MEAN_ABS, f"{what}: mean abs error {diff.mean():.3e}"
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        ref_lse = np.asarray(ref_lse, dtype=np.float64)
        assert lse.shape == ref_lse.shape
        inf_g, inf_r = np.isneginf(lse), np.isneginf(ref_lse)
        assert np.array_equal(inf_g, inf_r), f"{what}: -inf pattern of lse differs"
        assert not np.any(np.isnan(lse)), f"{what}: NaN lse"
        if (~inf_r).any():
            dl = np.abs(lse[~inf_r] - ref_lse[~inf_r]).max()
            assert dl <= LSE_TOL, f"{what}: lse error {dl:.3e}"
    return float(np.abs(out - ref_out).max())
