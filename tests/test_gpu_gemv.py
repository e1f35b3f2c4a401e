"""GPU weight-stream products against the oracle (tolerance
|err| <= 1e-4 * sum|w x| + 1/2 BF16 ulp)."""
import numpy as np
import pytest
import torch

from oracle import quant as Q, products as P, tolerance as T, model as M, formats as F
from tests.gpu_util import device, bws, np_, f64, rand_W, rand_x

pytestmark = pytest.mark.gpu


_QCACHE = {}


def _quant_nvfp4(W):
    """NVFP4 codes from the oracle's quantizer, uploaded: the product test
    then takes no input from the CUDA path."""
    key = (tuple(W.shape), float(W.float().abs().sum().item()))
    if key not in _QCACHE:
        c, s, t = Q.nvfp4_quantize(np_(W))
        dev = device()
        _QCACHE[key] = (torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev),
                        torch.tensor([float(t)], dtype=torch.float32, device=dev), (c, s, np.float32(t)))
    return _QCACHE[key]


SHAPES = [(16, 32), (32, 128), (48, 96), (100, 160), (333, 640), (1000, 2560), (4096, 4096)]


@pytest.mark.parametrize("N", [1, 2, 3, 8])
@pytest.mark.parametrize("shape", SHAPES)
def test_nvfp4_gemv_parity(shape, N):
    d_out, d_in = shape
    W = rand_W(shape, seed=d_out + d_in)
    x = rand_x(N, d_in, seed=N)
    c, s, t, host = _quant_nvfp4(W)
    y = bws().nvfp4_gemv(c, s, t, x)
    y_ref, A = P.nvfp4_gemv(*host, f64(x))
    ok, worst, at = T.check(y_ref, f64(y), A)
    assert ok, (worst, at)


def test_nvfp4_gemv_one_hot_is_exact():
    d_out, d_in = 200, 512
    W = rand_W((d_out, d_in), seed=5)
    c, s, t, host = _quant_nvfp4(W)
    w_hat = P.nvfp4_dequantize(*host)
    cols = [0, 1, 31, 32, 255, 511]
    x = torch.zeros((len(cols), d_in), dtype=torch.bfloat16, device=device())
    for n, j in enumerate(cols):
        x[n, j] = 1.0
    y = bws().nvfp4_gemv(c, s, t, x)
    want = F.round_bf16(w_hat[:, cols].T)
    assert np.array_equal(f64(y), want)


def test_nvfp4_gemv_exact_sums_are_bitexact():
    """Power-of-two activations and a unit tensor scale: every partial sum is
    exact in FP32, so the result must equal the oracle's rounded exactly."""
    d_out, d_in = 64, 1024
    rng = np.random.default_rng(3)
    W = rng.choice([-6, -4, -3, -2, -1, 0, 1, 2, 3, 4, 6], size=(d_out, d_in)).astype(np.float32)
    W[0, 0] = 2688.0
    x = np.ldexp(1.0, rng.integers(-3, 3, size=(4, d_in))) * rng.choice([-1, 1], size=(4, d_in))
    xt = torch.from_numpy(x.astype(np.float32)).to(device()).to(torch.bfloat16)
    c, s, t, host = _quant_nvfp4(torch.from_numpy(W).to(device()))
    y = bws().nvfp4_gemv(c, s, t, xt)
    y_ref, _ = P.nvfp4_gemv(*host, x)
    assert np.array_equal(f64(y), F.round_bf16(y_ref))


def test_nvfp4_gemv_rows_are_independent_tokens():
    W = rand_W((500, 1280), seed=9)
    c, s, t, _ = _quant_nvfp4(W)
    x = rand_x(8, 1280, seed=9)
    y8 = bws().nvfp4_gemv(c, s, t, x)
    for n in range(8):
        y1 = bws().nvfp4_gemv(c, s, t, x[n:n + 1].contiguous())
        assert torch.equal(y1[0], y8[n])


def test_nvfp4_gemv_deterministic():
    W = rand_W((3000, 5120), seed=11)
    c, s, t, _ = _quant_nvfp4(W)
    x = rand_x(3, 5120, seed=11)
    ys = [bws().nvfp4_gemv(c, s, t, x) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


def test_nvfp4_gemv_wide_dynamic_range_uses_second_band():
    d_out, d_in = 256, 1024
    W = rand_W((d_out, d_in), seed=13)
    c, s, t, host = _quant_nvfp4(W)
    rng = np.random.default_rng(13)
    x = rng.standard_normal((2, d_in)) * np.ldexp(1.0, rng.integers(-45, 8, size=(2, d_in)))
    xt = torch.from_numpy(x.astype(np.float32)).to(device()).to(torch.bfloat16)
    ws = bws().Workspace(device())
    y = bws().nvfp4_gemv(c, s, t, xt, ws=ws)
    assert bws().status_word(ws) & bws().BWS_STATUS_X_TWO_BANDS
    y_ref, A = P.nvfp4_gemv(*host, f64(xt))
    ok, worst, at = T.check(y_ref, f64(y), A)
    assert ok, (worst, at)


def test_nvfp4_gemv_zero_and_tiny_inputs():
    W = rand_W((64, 256), seed=2)
    c, s, t, host = _quant_nvfp4(W)
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device=device())
    x[1, 3] = 1e-30
    y = bws().nvfp4_gemv(c, s, t, x)
    y_ref, A = P.nvfp4_gemv(*host, f64(x))
    ok, worst, _ = T.check(y_ref, f64(y), A)
    assert ok and torch.all(y[0] == 0)


@pytest.mark.parametrize("N", [1, 8])
def test_gate_up_silu_parity(N):
    d_inter, d_in = 1100, 1024
    Wg = rand_W((d_inter, d_in), seed=21, index=0)
    Wu = rand_W((d_inter, d_in), seed=21, index=1)
    g_dev = _quant_nvfp4(Wg)
    u_dev = _quant_nvfp4(Wu)
    x = rand_x(N, d_in, seed=21)
    h = bws().nvfp4_gate_up_silu(g_dev[:3], u_dev[:3], x)
    g, Ag = P.nvfp4_gemv(*g_dev[3], f64(x))
    u, Au = P.nvfp4_gemv(*u_dev[3], f64(x))
    h_exact = M.silu(g) * u
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = np.abs(sig * (1.0 + g * (1.0 - sig))) + 0.0
    tg, tu = 1e-4 * Ag, 1e-4 * Au
    # first-order propagation of the g and u bounds, their product, and FP32
    # evaluation of SiLU(g) * u (a few ulp)
    extra = dsilu * np.abs(u) * tg + np.abs(M.silu(g)) * tu + 1.1 * tg * tu + 1e-6 * np.abs(h_exact)
    ok, worst, at = T.check(h_exact, f64(h), np.zeros_like(h_exact), extra=extra)
    assert ok, (worst, at)


@pytest.mark.parametrize("N", [1, 4])
@pytest.mark.parametrize("shape", [(40, 64), (1000, 2560), (7777, 5120)])
def test_fp8_head_parity(shape, N):
    V, d = shape
    W = rand_W(shape, seed=V)
    c, r = Q.fp8_rowwise_quantize(np_(W))
    codes, rs = torch.from_numpy(c).to(device()), torch.from_numpy(r).to(device())
    x = rand_x(N, d, seed=V)
    logits = bws().fp8_lmhead_gemv(codes, rs, x)
    y_ref, A = P.fp8_gemv(c, r, f64(x))
    ok, worst, at = T.check(y_ref, f64(logits), A)
    assert ok, (worst, at)


def test_empty_calls_are_noops():
    W = rand_W((64, 128), seed=1)
    c, s, t, _ = _quant_nvfp4(W)
    x = rand_x(1, 128, seed=1)
    y = torch.full((0, 64), 7.0, dtype=torch.bfloat16, device=device())
    bws().nvfp4_gemv(c, s, t, x[:0], y=y)


@pytest.mark.parametrize("N", [1, 3])
def test_prepared_products_match_one_call_products(N):
    """One prepare, several products of the same input (different d_out, up
    to d_out_max): bit-equal to bws_nvfp4_gemv of each matrix."""
    d_in = 1024
    x = rand_x(N, d_in, seed=31 + N)
    mats = [_quant_nvfp4(rand_W((d_out, d_in), seed=40 + d_out)) for d_out in (384, 100, 1000)]
    ws = bws().Workspace(device())
    bws().nvfp4_prepare(x, 1000, ws)
    ys = [bws().nvfp4_gemv_prepared(c, s, t, N, d_in, ws) for c, s, t, _ in mats]
    for (c, s, t, host), y in zip(mats, ys):
        assert torch.equal(y, bws().nvfp4_gemv(c, s, t, x))
        y_ref, A = P.nvfp4_gemv(*host, f64(x))
        ok, worst, at = T.check(y_ref, f64(y), A)
        assert ok, (worst, at)


def test_prepared_product_rejects_a_matrix_of_another_layout():
    """Activations prepared for 16-byte aligned matrices (d_in % 256 == 0);
    scales at an 8-byte offset need the other kernel's layout."""
    d_in = 512
    c, s, t, _ = _quant_nvfp4(rand_W((64, d_in), seed=50))
    s_off = torch.empty(s.numel() + 8, dtype=torch.uint8, device=device())[8:].view(s.shape)
    s_off.copy_(s)
    x = rand_x(1, d_in, seed=50)
    ws = bws().Workspace(device())
    bws().nvfp4_prepare(x, 64, ws)
    with pytest.raises(Exception, match="status 3"):
        bws().nvfp4_gemv_prepared(c, s_off, t, 1, d_in, ws)
