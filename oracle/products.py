"""Dequantization and exact matrix-vector products.

A matvec with d_out rows and d_in columns does one multiply and one add per
weight ([Spark27B] § "Decode speed is bytes divided by bandwidth"). The
oracle forms every dequantized weight exactly in FP64 (an E2M1 value times an
E4M3 or E8M0 scale times the FP32 tensor scale needs at most 24+4+2 bits) and
sums the products in FP64 with a library matmul.
"""
import numpy as np

from .formats import e2m1_decode, e4m3_decode, e8m0_decode
from .quant import unpack_nibbles, NVFP4_BLOCK, MXFP4_BLOCK, MXFP8_BLOCK


def nvfp4_dequantize(codes, scales, s_t):
    """w_hat = s_t * dec_E4M3(scale of its 16-block) * dec_E2M1(code), FP64."""
    q = e2m1_decode(unpack_nibbles(codes))
    d_out, d_in = q.shape
    sb = e4m3_decode(scales)
    w = q.reshape(d_out, d_in // NVFP4_BLOCK, NVFP4_BLOCK) * sb[..., None]
    return w.reshape(d_out, d_in) * np.float64(np.float32(s_t))


def mxfp4_dequantize(codes, scales):
    """w_hat = 2^(scale-127) * dec_E2M1(code), FP64."""
    q = e2m1_decode(unpack_nibbles(codes))
    rows, d_in = q.shape
    sb = e8m0_decode(scales)
    w = q.reshape(rows, d_in // MXFP4_BLOCK, MXFP4_BLOCK) * sb[..., None]
    return w.reshape(rows, d_in)


def mxfp8_dequantize(codes, scales):
    """x_hat = 2^(scale-127) * dec_E4M3(code), FP64 (MXFP8 activations)."""
    q = e4m3_decode(codes)
    n, d = q.shape
    sb = e8m0_decode(scales)
    x = q.reshape(n, d // MXFP8_BLOCK, MXFP8_BLOCK) * sb[..., None]
    return x.reshape(n, d)


def fp8_dequantize(codes, row_scale):
    """w_hat = s_r * dec_E4M3(code), FP64."""
    return e4m3_decode(codes) * np.asarray(row_scale, np.float32).astype(np.float64)[:, None]


def matvec(w_hat, X):
    """Y[n, i] = sum_j w_hat[i, j] * X[n, j] in FP64, with the absolute sum
    A[n, i] = sum_j |w_hat[i, j] * X[n, j]| that the tolerance uses.
    X is [N, d_in] (BF16 values held in FP64)."""
    X = np.atleast_2d(np.asarray(X, dtype=np.float64))
    w_hat = np.asarray(w_hat, dtype=np.float64)
    return X @ w_hat.T, np.abs(X) @ np.abs(w_hat).T


def nvfp4_gemv(codes, scales, s_t, X):
    """Y = X W_hat^T for NVFP4 W (one token row of X per output row of Y)."""
    return matvec(nvfp4_dequantize(codes, scales, s_t), X)


def mxfp4_gemv(codes, scales, X):
    return matvec(mxfp4_dequantize(codes, scales), X)


def w4a8_gemv(w_codes, w_scales, x_codes, x_scales):
    """W4A8: MXFP4 weights times MXFP8 activations, Y = X_hat W_hat^T with both
    operands dequantized exactly ([LingMoE] §三, the W4A8 baseline)."""
    return matvec(mxfp4_dequantize(w_codes, w_scales), mxfp8_dequantize(x_codes, x_scales))


def fp8_gemv(codes, row_scale, X):
    return matvec(fp8_dequantize(codes, row_scale), X)
