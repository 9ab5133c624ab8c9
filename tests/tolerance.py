"""Comparison rules for GPU results against the oracle.

Floating-point MoE outputs pass iff every element satisfies
    |gpu - ref| <= 1e-2 * RMS(ref) + 2e-2 * |ref|
(ref = the oracle's float64 result before any rounding; RMS over the compared
elements).  Integer and byte outputs (routing, requantised codes and scales)
must match exactly.
"""

import numpy as np

ATOL_RMS = 1e-2
RTOL = 2e-2


def moe_tolerance_report(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = ATOL_RMS * rms + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    return {
        "rms": rms,
        "max_err": float(err.max()) if err.size else 0.0,
        "max_err_over_rms": float(err.max() / rms) if err.size and rms > 0 else 0.0,
        "n_bad": int(bad.sum()),
        "first_bad": tuple(int(i) for i in np.argwhere(bad)[0]) if bad.any() else None,
    }


def assert_moe_close(got, ref):
    rep = moe_tolerance_report(got, ref)
    assert rep["n_bad"] == 0, f"MoE output outside tolerance: {rep}"
    return rep
