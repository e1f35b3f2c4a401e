"""Pins for the oracle's products and layer recipe (CPU only)."""
from fractions import Fraction

import math

import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q
from oracle import products as P
from oracle import model as M
from oracle import tolerance as T
import synth


def _nvfp4(d_out, d_in, seed=0):
    W = synth.weight_fp32((d_out, d_in), seed=seed).numpy()
    return Q.nvfp4_quantize(W)


def test_brute_force_16x32_exact_rationals():
    codes, scales, s_t = _nvfp4(16, 32, seed=11)
    X = synth.activation_bf16(3, 32, seed=11).float().numpy().astype(np.float64)
    Y, A = P.nvfp4_gemv(codes, scales, s_t, X)
    q = Q.unpack_nibbles(codes)
    st = Fraction(float(np.float32(s_t)))
    for n in range(3):
        for i in range(16):
            acc = Fraction(0)
            acc_abs = Fraction(0)
            for j in range(32):
                w = st * Fraction(float(F.e4m3_decode(scales[i, j // 16]))) \
                    * Fraction(float(F.e2m1_decode(q[i, j])))
                t = w * Fraction(float(X[n, j]))
                acc += t
                acc_abs += abs(t)
            assert abs(Fraction(float(Y[n, i])) - acc) <= abs(acc) * Fraction(1, 2 ** 50)
            assert abs(Fraction(float(A[n, i])) - acc_abs) <= acc_abs * Fraction(1, 2 ** 50)


def test_one_hot_gives_a_column():
    codes, scales, s_t = _nvfp4(48, 64, seed=2)
    w_hat = P.nvfp4_dequantize(codes, scales, s_t)
    for j in (0, 17, 63):
        x = np.zeros((1, 64))
        x[0, j] = 1.0
        y, _ = P.nvfp4_gemv(codes, scales, s_t, x)
        assert np.array_equal(y[0], w_hat[:, j])


def test_rows_of_X_are_independent_tokens():
    codes, scales, s_t = _nvfp4(32, 64, seed=4)
    X = synth.activation_bf16(5, 64, seed=4).float().numpy()
    Y, _ = P.nvfp4_gemv(codes, scales, s_t, X)
    for n in range(5):
        y1, _ = P.nvfp4_gemv(codes, scales, s_t, X[n:n + 1])
        assert np.allclose(Y[n], y1[0], rtol=1e-15, atol=0)


def test_fp8_and_mxfp4_products_match_numpy_dot():
    W = synth.weight_fp32((40, 96), seed=9).numpy()
    X = synth.activation_bf16(2, 96, seed=9).float().numpy().astype(np.float64)
    c8, s8 = Q.fp8_rowwise_quantize(W)
    y8, _ = P.fp8_gemv(c8, s8, X)
    wd = np.array([[float(F.e4m3_decode(c)) * float(s8[i]) for c in row] for i, row in enumerate(c8)])
    assert np.allclose(y8, np.array([[np.dot(wd[i], X[n]) for i in range(40)] for n in range(2)]), rtol=1e-14)
    c4, e4 = Q.mxfp4_quantize(W)
    y4, _ = P.mxfp4_gemv(c4, e4, X)
    q = Q.unpack_nibbles(c4)
    wd4 = np.array([[float(F.e2m1_decode(q[i, j])) * 2.0 ** (int(e4[i, j // 32]) - 127)
                     for j in range(96)] for i in range(40)])
    assert np.allclose(y4, X @ wd4.T, rtol=1e-14)


def test_w4a8_brute_force_exact_rationals():
    # MXFP4 weights times MXFP8 activations, every product and sum in exact
    # rationals from the decoded codes and the power-of-two scales
    W = synth.weight_fp32((8, 64), seed=12).numpy()
    X = synth.activation_bf16(3, 64, seed=12).float().numpy()
    wc, ws = Q.mxfp4_quantize(W)
    xc, xs = Q.mxfp8_quantize(X)
    Y, A = P.w4a8_gemv(wc, ws, xc, xs)
    q = Q.unpack_nibbles(wc)
    for n in range(3):
        for i in range(8):
            acc = Fraction(0)
            acc_abs = Fraction(0)
            for j in range(64):
                w = Fraction(float(F.e2m1_decode(q[i, j]))) * Fraction(2) ** (int(ws[i, j // 32]) - 127)
                x = Fraction(float(F.e4m3_decode(xc[n, j]))) * Fraction(2) ** (int(xs[n, j // 32]) - 127)
                acc += w * x
                acc_abs += abs(w * x)
            assert abs(Fraction(float(Y[n, i])) - acc) <= abs(acc) * Fraction(1, 2 ** 50)
            assert abs(Fraction(float(A[n, i])) - acc_abs) <= acc_abs * Fraction(1, 2 ** 50)


def test_silu_identities():
    g = np.linspace(-30, 30, 1001)
    s = M.silu(g)
    assert np.allclose(s - M.silu(-g), g, rtol=0, atol=1e-12)   # x*sig(x) - (-x)*sig(-x) = x
    assert M.silu(0.0) == 0.0
    assert np.isclose(M.silu(1.0), 1.0 / (1.0 + np.exp(-1.0)))
    assert abs(M.silu(-40.0)) < 1e-15 and np.isclose(M.silu(40.0), 40.0)


def test_rmsnorm_properties():
    r = np.random.default_rng(0).standard_normal((3, 256)) * 7.0
    y = M.rmsnorm(r, eps=0.0)
    assert np.allclose(np.mean(y * y, axis=1), 1.0)
    assert np.allclose(M.rmsnorm(5.0 * r, eps=0.0), y)
    z = M.rmsnorm(np.zeros((1, 8)))
    assert np.all(z == 0)


def test_expected_distinct_experts_closed_form_and_sampling():
    assert M.expected_distinct(512, 8, 1) == 8.0
    e4 = M.expected_distinct(512, 8, 4)
    assert round(e4, 1) == 31.3
    counts = [len(M.distinct_experts(synth.expert_ids(4, 8, 512, seed=s, layer=0).numpy()))
              for s in range(600)]
    m, sd = np.mean(counts), np.std(counts) / np.sqrt(len(counts))
    assert abs(m - e4) < 4 * sd


def _expert_factory(E, d, inter, seed):
    cache = {}

    def expert(e):
        if e not in cache:
            Ws = [synth.weight_fp32(s, seed=seed, index=100 * e + k).numpy()
                  for k, s in enumerate([(inter, d), (inter, d), (d, inter)])]
            cache[e] = tuple(P.mxfp4_dequantize(*Q.mxfp4_quantize(w)) for w in Ws)
        return cache[e]
    return expert


def test_moe_reduces_to_one_expert():
    d, inter, E = 64, 32, 16
    expert = _expert_factory(E, d, inter, seed=1)
    X = F.round_bf16(synth.activation_bf16(3, d, seed=1).float().numpy())
    ids = np.array([[2, 5], [5, 9], [2, 9]])
    w = np.array([[1.0, 0.0], [1.0, 0.0], [0.0, 1.0]])
    Y = M.moe(X, ids, w, expert, shared=None)
    assert np.allclose(Y[0], M.mlp(*expert(2), X[0:1])[0], rtol=1e-15, atol=0)
    assert np.allclose(Y[1], M.mlp(*expert(5), X[1:2])[0], rtol=1e-15, atol=0)
    assert np.allclose(Y[2], M.mlp(*expert(9), X[2:3])[0], rtol=1e-15, atol=0)
    # shared expert only
    Y0 = M.moe(X, ids, np.zeros_like(w), expert, shared=expert(0))
    assert np.allclose(Y0, M.mlp(*expert(0), X), rtol=1e-15, atol=0)


def test_moe_linearity_in_route_weights():
    d, inter = 64, 32
    expert = _expert_factory(8, d, inter, seed=2)
    X = F.round_bf16(synth.activation_bf16(2, d, seed=2).float().numpy())
    ids = np.array([[1, 3, 4], [0, 3, 7]])
    w = synth.route_weights(2, 3, seed=2).numpy().astype(np.float64)
    Y = M.moe(X, ids, w, expert)
    Z = sum(w[:, k:k + 1] * np.stack([M.mlp(*expert(int(ids[t, k])), X[t:t + 1])[0]
                                      for t in range(2)]) for k in range(3))
    assert np.allclose(Y, Z, rtol=1e-14, atol=1e-18)


def test_dense_stack_zero_layers_is_the_head():
    d, V = 64, 40
    W = synth.weight_fp32((V, d), seed=3).numpy()
    head = P.fp8_dequantize(*Q.fp8_rowwise_quantize(W))
    x0 = F.round_bf16(synth.activation_bf16(2, d, seed=3).float().numpy())
    logits, A, r = M.decode_stack(x0, [], head)
    want, _ = P.matvec(head, F.round_bf16(M.rmsnorm(x0)))
    assert np.array_equal(logits, want) and np.array_equal(r, x0)


def test_rmsnorm_eps_inside_the_root_worked_by_hand():
    """r = [3, -4, 0, 12]: mean(r^2) = (9 + 16 + 0 + 144) / 4 = 42.25; with
    eps = 6.75, sqrt(42.25 + 6.75) = sqrt(49) = 7, so RMSNorm(r) =
    [3/7, -4/7, 0, 12/7]. (eps added after the root would divide by
    6.5 + 6.75 = 13.25 instead.)"""
    y = M.rmsnorm(np.array([[3.0, -4.0, 0.0, 12.0]]), eps=6.75)
    assert np.allclose(y, [[3 / 7, -4 / 7, 0.0, 12 / 7]], rtol=1e-15, atol=0)


def _silu_closed(g):
    return g / (1.0 + math.exp(-g))


def test_dense_layer_worked_by_hand():
    """One dense layer on hand-chosen matrices whose every intermediate value
    is known (hidden 4, N = 1, eps 1e-6):
      r0 = [2, 2, 2, 2]: mean square 4, a = BF16(r0 / sqrt(4 + 1e-6)) =
        [1, 1, 1, 1] (1 - 1.25e-7 rounds to 1 in BF16);
      u = W_in a = row sums of W_in = [1, 1, 2, 0.5, 3, 2] (exact in BF16);
      the mixer stand-in takes the first d_v = 2 entries: v = [1, 1];
      W_o v = [1, 3, -1, -1], so r_mid = [3, 5, 1, 1] (mean square 9);
      m = BF16(r_mid / 3) = [1, BF16(5/3), BF16(1/3), BF16(1/3)]
        = [1, 213/128, 171/512, 171/512] (5/3 = 1.1010101|01..b rounds
        down to 1.1010101b; 1/3 = 1.0101010|1010..b x 2^-2 rounds up);
      g = W_gate m = [3 m_2, -2 m_0, m_2 - m_3] = [513/512, -2, 0];
      up = W_up m = [3 m_1, m_0, 4 m_0] = [639/128, 1, 4];
      h = BF16(SiLU(g) * up) with SiLU(x) = x / (1 + e^-x);
      y = W_down h = [h0, h1, h0 + h1, h2] and r1 = r_mid + y.
    (Taking the last d_v entries of u instead gives W_o [3, 2] =
    [3, 7, -3, -2]; any slip in the order fails this.)"""
    W_in = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [1, 1, 0, 0], [0, 0, 0, 0.5], [3, 0, 0, 0], [0, 0, 1, 1]],
                    dtype=np.float64)
    W_o = np.array([[1, 0], [1, 2], [-1, 0], [0, -1]], dtype=np.float64)
    W_g = np.array([[0, 0, 3, 0], [-2, 0, 0, 0], [0, 0, 1, -1]], dtype=np.float64)
    W_u = np.array([[0, 3, 0, 0], [1, 0, 0, 0], [4, 0, 0, 0]], dtype=np.float64)
    W_d = np.array([[1, 0, 0], [0, 1, 0], [1, 1, 0], [0, 0, 1]], dtype=np.float64)
    layer = {"in": [W_in[:4], W_in[4:]], "out": W_o, "gate": W_g, "up": W_u, "down": W_d}
    r1 = M.dense_layer(np.array([[2.0, 2.0, 2.0, 2.0]]), layer)
    h = F.round_bf16(np.array([_silu_closed(513 / 512) * 639 / 128, _silu_closed(-2.0) * 1.0, 0.0]))
    want = np.array([[3 + h[0], 5 + h[1], 1 + h[0] + h[1], 1 + h[2]]])
    assert np.array_equal(r1, want), (r1, want)


def test_tolerance_bound():
    ok, worst, _ = T.check([1.0], [1.0 + 2 ** -8], [0.0])
    assert ok                      # half a BF16 ulp at 1.0 is 2^-8
    ok, worst, _ = T.check([1.0], [1.0 + 2 ** -7], [0.0])
    assert not ok
    ok, _, _ = T.check([0.0], [0.5e-4], [1.0])
    assert ok
    ok, _, _ = T.check([0.0], [1.5e-4], [1.0])
    assert not ok
