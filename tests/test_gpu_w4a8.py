"""W4A8 on the GPU against the oracle: the MXFP8 activation codes and scales
bit-exact (bws_mxfp8_quantize), and the tensor-core product
(bws_mxfp4_w4a8_gemv) within |y - y_ref| <= 1e-4 sum|w xq| + 1/2 ulp(y) of
the exact product of the dequantized MXFP4 weights and the oracle's MXFP8
activations; exact where every sum is representable (one-hot activations).
Against the BF16 activations themselves the W4A8 result differs by the
activation rounding, bounded by sum_j |w_ij| |x_j - xq_j| (checked too)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F, products as P, quant as Q, tolerance as T
from tests.gpu_util import device, bws
import synth

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_hand.json")


def _bf16_rows(X):
    return torch.tensor(np.asarray(X, dtype=np.float32)).to(torch.bfloat16).to(device())


def _mxfp4(d_out, d_in, seed):
    W = synth.weight_fp32((d_out, d_in), seed=seed, index=3).numpy()
    c, s = Q.mxfp4_quantize(W)
    return c, s, torch.from_numpy(c).to(device()), torch.from_numpy(s).to(device())


def test_quantizer_hand_rows():
    m = bws()
    g = json.load(open(GOLDEN))
    x = _bf16_rows(g["X"])
    codes, scales = m.mxfp8_quantize(x)
    torch.cuda.synchronize()
    assert scales.cpu().tolist() == g["scales"]
    assert codes.cpu().tolist() == g["codes"]


@pytest.mark.parametrize("N,d", [(1, 256), (3, 2560), (8, 5120), (13, 96)])
def test_quantizer_bit_exact(N, d):
    m = bws()
    x = synth.activation_bf16(N, d, seed=N + d, device=device())
    x[0, :32] = 0.0                      # a zero block
    x[-1, -32:] *= 2.0 ** -100           # a tiny block (the scale clamps)
    codes, scales = m.mxfp8_quantize(x)
    oc, os_ = Q.mxfp8_quantize(x.float().cpu().numpy())
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


def _check_product(c, s, cd, sd, x, y):
    X = x.float().cpu().numpy().astype(np.float64)
    xc, xs = Q.mxfp8_quantize(X.astype(np.float32))
    want, A = P.w4a8_gemv(c, s, xc, xs)
    ok, worst, at = T.check(want, y.float().cpu().numpy(), A)
    assert ok, (worst, at)
    # the activation rounding's effect, against the BF16 activations
    w_hat = P.mxfp4_dequantize(c, s)
    ref, A2 = P.matvec(w_hat, X)
    dx = np.abs(X - P.mxfp8_dequantize(xc, xs))
    q_bound = dx @ np.abs(w_hat).T
    err = np.abs(y.float().cpu().numpy() - ref)
    assert np.all(err <= q_bound + T.bound(want, y.float().cpu().numpy(), A))
    return worst


@pytest.mark.parametrize("d_out,d_in,N", [(128, 256, 1), (300, 512, 3), (2560, 768, 8), (1536, 2560, 4),
                                          (6912, 2560, 8), (1000, 5120, 2)])
def test_w4a8_product(d_out, d_in, N):
    # one unit, a ragged tile, the Ling expert down (2560 x 768) and gate/up
    # (1536 x 2560) shapes, the Ling dense MLP width, a stream-K split
    m = bws()
    c, s, cd, sd = _mxfp4(d_out, d_in, seed=d_out + N)
    x = synth.activation_bf16(N, d_in, seed=d_in + N, device=device())
    x[0, 32:64] = 0.0                     # a zero activation block (scale code 0)
    x[-1, 64:96] *= 2.0 ** -60            # a tiny block
    y = m.mxfp4_w4a8_gemv(cd, sd, x)
    torch.cuda.synchronize()
    _check_product(c, s, cd, sd, x, y)


def test_w4a8_one_hot_is_exact():
    # x = e_j: y is column j of w times the quantized 1.0 (scale 2^-8, code
    # 256 = 0x78), exactly representable, so the BF16 result is exact
    m = bws()
    c, s, cd, sd = _mxfp4(640, 512, seed=5)
    w_hat = P.mxfp4_dequantize(c, s)
    for j in (0, 33, 511):
        x = torch.zeros((1, 512), dtype=torch.bfloat16, device=device())
        x[0, j] = 1.0
        y = m.mxfp4_w4a8_gemv(cd, sd, x)
        torch.cuda.synchronize()
        want = F.round_bf16(w_hat[:, j])
        assert np.array_equal(y.float().cpu().numpy()[0], want)


def test_w4a8_tokens_are_independent():
    m = bws()
    c, s, cd, sd = _mxfp4(384, 1024, seed=8)
    x = synth.activation_bf16(8, 1024, seed=8, device=device())
    y8 = m.mxfp4_w4a8_gemv(cd, sd, x)
    for n in (0, 5, 7):
        y1 = m.mxfp4_w4a8_gemv(cd, sd, x[n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(y1[0], y8[n])


def test_w4a8_full_size_sampled_rows():
    # the 27B-shape MLP projection in MXFP4 at eight tokens, the configuration
    # the bench times; rows sampled (first and last two plus random ones)
    m = bws()
    d_out, d_in, N = 17408, 5120, 8
    W = synth.weight_fp32((d_out, d_in), seed=0, index=3, device=device())
    cd, sd = m.mxfp4_quantize(W)
    x = synth.activation_bf16(N, d_in, seed=1, device=device())
    y = m.mxfp4_w4a8_gemv(cd, sd, x)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = np.array(sorted(set([0, 1, d_out - 2, d_out - 1]) | set(rng.choice(d_out, 60, replace=False).tolist())))
    Wr = W[torch.from_numpy(rows).to(device())].cpu().numpy()
    c, s = Q.mxfp4_quantize(Wr)
    assert np.array_equal(cd[torch.from_numpy(rows).to(device())].cpu().numpy(), c)
    assert np.array_equal(sd[torch.from_numpy(rows).to(device())].cpu().numpy(), s)
    X = x.float().cpu().numpy()
    xc, xs = Q.mxfp8_quantize(X)
    want, A = P.w4a8_gemv(c, s, xc, xs)
    ok, worst, at = T.check(want, y.float().cpu().numpy()[:, rows], A)
    assert ok, (worst, at)
