"""Tolerance checks between a GPU result and the float64 oracle.

fp16 NT:  |C_gpu - C_ref| <= 4e-3 * S + 1e-6 per element,
fp32 SGEMM: |C_gpu - C_ref| <= 1e-5 * S (+ 2^-22 |beta C0| for the rounding
of the beta term, which S does not cover),
where S = |alpha| * sum_k |A * B| comes from the oracle.  Every GPU output
must also be finite.
"""
import numpy as np

F16_REL = 4e-3
F16_ABS = 1e-6
SGEMM_REL = 1e-5


def check_f16(c_gpu, c_ref, s, what=""):
    c = np.asarray(c_gpu, dtype=np.float64)
    assert np.all(np.isfinite(c)), f"{what}: non-finite output"
    err = np.abs(c - c_ref)
    bound = F16_REL * s + F16_ABS
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first "
                             f"{idx.tolist()} err={err[bad][:5]} bound={bound[bad][:5]}")
    return float((err / bound).max()) if err.size else 0.0


def check_sgemm(c_gpu, c_ref, s, beta_c0=None, what=""):
    c = np.asarray(c_gpu, dtype=np.float64)
    assert np.all(np.isfinite(c)), f"{what}: non-finite output"
    err = np.abs(c - c_ref)
    bound = SGEMM_REL * s
    if beta_c0 is not None:
        bound = bound + 2.0 ** -22 * np.abs(beta_c0)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first "
                             f"{idx.tolist()} err={err[bad][:5]} bound={bound[bad][:5]}")
    return float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0
