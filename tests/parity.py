"""Tolerance checks between a GPU result and the float64 oracle.

fp16 NT:  |C_gpu - C_ref| <= 4e-3 * S + 1e-6 per element,
fp32 SGEMM: |C_gpu - C_ref| <= 1e-5 * S,
where S = |alpha| * sum_k |A * B| comes from the oracle.  (The SGEMM bound
has no term for beta * C0: its rounding, at most 2^-24 |result|, is far
below 1e-5 * S wherever the product is not empty, and the K = 0 case is
checked for exact equality with a beta whose product is exact.)  Every GPU output
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


def check_sgemm(c_gpu, c_ref, s, what=""):
    c = np.asarray(c_gpu, dtype=np.float64)
    assert np.all(np.isfinite(c)), f"{what}: non-finite output"
    err = np.abs(c - c_ref)
    bound = SGEMM_REL * s
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first "
                             f"{idx.tolist()} err={err[bad][:5]} bound={bound[bad][:5]}")
    return float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0


# The fused epilogue act(v) of the fp16 product: every activation it offers
# has |act'(v)| <= 1.13 (tanh-GELU; SiLU 1.10, ReLU 1) and |act(v)| <= |v|, so
# an error e in v becomes at most 1.13 e after the activation and the final
# rounding to half stays within 2^-11 |v|; 1.25 covers the first with room.
# The absolute 1e-5 covers the device's fp32 exp and tanh near v = 0, where
# S can be tiny.
EPI_LIPSCHITZ = 1.25
EPI_ABS = 1e-5


def check_f16_epilogue(c_gpu, y_ref, s, what=""):
    """|Y_gpu - Y_ref| <= 1.25 * 4e-3 * S + 1e-5 with S = |alpha| sum|AB| + |bias| + |beta R|."""
    c = np.asarray(c_gpu, dtype=np.float64)
    assert np.all(np.isfinite(c)), f"{what}: non-finite output"
    err = np.abs(c - y_ref)
    bound = EPI_LIPSCHITZ * F16_REL * s + EPI_ABS
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first "
                             f"{idx.tolist()} err={err[bad][:5]} bound={bound[bad][:5]}")
    return float((err / bound).max()) if err.size else 0.0
