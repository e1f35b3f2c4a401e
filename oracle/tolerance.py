"""The comparison bound for GPU results.

|y_gpu - y| <= 1e-4 * sum_j |w_hat_ij x_j| + 1/2 ulp_BF16(max(|y_gpu|, |y|)),
the ulp taken at the larger magnitude (at the smallest normal for 0).
"""
import numpy as np

from .formats import bf16_ulp

REL = 1e-4


def bound(y_ref, y_gpu, abs_sum, rel=REL):
    y_ref = np.asarray(y_ref, dtype=np.float64)
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    big = np.maximum(np.abs(y_ref), np.abs(y_gpu))
    return rel * np.asarray(abs_sum, dtype=np.float64) + 0.5 * bf16_ulp(big)


def check(y_ref, y_gpu, abs_sum, rel=REL, extra=0.0):
    """(ok, worst ratio |err|/bound, index of worst)."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    b = bound(y_ref, y_gpu, abs_sum, rel) + extra
    ratio = np.where(b > 0, err / np.where(b > 0, b, 1.0), np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isnan(y_gpu) | np.isnan(y_ref), np.inf, ratio)
    if ratio.size == 0:
        return True, 0.0, None
    i = int(np.argmax(ratio))
    return bool(ratio.reshape(-1)[i] <= 1.0), float(ratio.reshape(-1)[i]), np.unravel_index(i, ratio.shape)
