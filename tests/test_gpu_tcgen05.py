"""The opt-in one-token tensor-core product kernel (BWS_PRODUCT_KERNEL=tcgen05:
tcgen05.mma on TMA-unpacked E2M1 codes against E4M3 activation bands)
against the oracle, same tolerance as the other products."""
import numpy as np
import pytest
import torch

from oracle import products as P, tolerance as T, model as M, formats as F
from tests.gpu_util import device, bws, f64, rand_W, rand_x
from tests.test_gpu_gemv import _quant_nvfp4
from tests.stack_util import oracle_quantizers, oracle_logits, STACK_SLACK
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tcgen05(monkeypatch):
    monkeypatch.setenv("BWS_PRODUCT_KERNEL", "tcgen05")


def _gemv_checked(shape, seed_w, x):
    W = rand_W(shape, seed=seed_w)
    c, s, t, host = _quant_nvfp4(W)
    y = bws().nvfp4_gemv(c, s, t, x)
    y_ref, A = P.nvfp4_gemv(*host, f64(x))
    ok, worst, at = T.check(y_ref, f64(y), A)
    assert ok, (worst, at)
    return y


SHAPES = [(1, 256), (129, 512), (333, 1024), (640, 768), (1000, 2560), (2000, 5120), (5000, 256)]


@pytest.mark.parametrize("shape", SHAPES)
def test_one_token_parity(shape):
    """Ragged last tiles, one unit per tile, tiles cut between CTAs."""
    _gemv_checked(shape, shape[0] * 7 + shape[1], rand_x(1, shape[1], seed=shape[0]))


def _rounded_term(host, x):
    """sum over the activations below 2^-19 of the row's largest magnitude
    (which the E4M3 bands round, flagging status bit 8) of |w| |x|: the most
    their rounding can change a row."""
    xa = np.abs(x)
    E = np.floor(np.log2(xa.max(axis=1, keepdims=True)))
    small = (xa > 0) & (xa < np.ldexp(1.0, (E - 19).astype(int)))
    w_hat = P.nvfp4_dequantize(*host)
    return (xa * small) @ np.abs(w_hat).T


def test_the_tensor_core_path_runs():
    """Only the E4M3 band image flags activations below 2^-19 of the row's
    largest magnitude (status bit 8): the call went through that path. Row
    results stay within the tolerance plus the rounded activations' |w x| (a
    row whose only other weight is zero keeps just that term)."""
    x = torch.zeros((1, 512), dtype=torch.bfloat16, device=device())
    x[0, 0] = 1.0
    x[0, 7] = 2.0 ** -30
    ws = bws().Workspace(device())
    W = rand_W((64, 512), seed=1)
    c, s, t, host = _quant_nvfp4(W)
    y = bws().nvfp4_gemv(c, s, t, x, ws=ws)
    assert bws().status_word(ws) & bws().BWS_STATUS_X_ROUNDED
    y_ref, A = P.nvfp4_gemv(*host, f64(x))
    ok, worst, at = T.check(y_ref, f64(y), A, extra=_rounded_term(host, f64(x)))
    assert ok, (worst, at)


def test_one_hot_is_exact():
    d_out, d_in = 200, 512
    W = rand_W((d_out, d_in), seed=5)
    c, s, t, host = _quant_nvfp4(W)
    w_hat = P.nvfp4_dequantize(*host)
    for j in [0, 1, 15, 16, 31, 32, 255, 256, 511]:
        x = torch.zeros((1, d_in), dtype=torch.bfloat16, device=device())
        x[0, j] = -3.0
        y = bws().nvfp4_gemv(c, s, t, x)
        assert np.array_equal(f64(y), F.round_bf16(-3.0 * w_hat[:, [j]].T)), j


def test_exact_sums_are_bitexact():
    d_out, d_in = 64, 1024
    rng = np.random.default_rng(4)
    W = rng.choice([-6, -4, -3, -2, -1, 0, 1, 2, 3, 4, 6], size=(d_out, d_in)).astype(np.float32)
    W[0, 0] = 2688.0
    x = np.ldexp(1.0, rng.integers(-3, 3, size=(1, d_in))) * rng.choice([-1, 1], size=(1, d_in))
    xt = torch.from_numpy(x.astype(np.float32)).to(device()).to(torch.bfloat16)
    c, s, t, host = _quant_nvfp4(torch.from_numpy(W).to(device()))
    y = bws().nvfp4_gemv(c, s, t, xt)
    y_ref, _ = P.nvfp4_gemv(*host, x)
    assert np.array_equal(f64(y), F.round_bf16(y_ref))


def test_wide_dynamic_range():
    """Activations over 2^-45 .. 2^8: exact down to 2^-19 of the row's largest
    magnitude, rounded below."""
    rng = np.random.default_rng(14)
    x = rng.standard_normal((1, 1024)) * np.ldexp(1.0, rng.integers(-45, 8, size=(1, 1024)))
    xt = torch.from_numpy(x.astype(np.float32)).to(device()).to(torch.bfloat16)
    W = rand_W((256, 1024), seed=13)
    c, s, t, host = _quant_nvfp4(W)
    y = bws().nvfp4_gemv(c, s, t, xt)
    y_ref, A = P.nvfp4_gemv(*host, f64(xt))
    ok, worst, at = T.check(y_ref, f64(y), A, extra=_rounded_term(host, f64(xt)))
    assert ok, (worst, at)


def test_zero_and_tiny_inputs():
    W = rand_W((64, 256), seed=2)
    c, s, t, host = _quant_nvfp4(W)
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device=device())
    assert torch.all(bws().nvfp4_gemv(c, s, t, x) == 0)
    x[0, 3] = 1e-30
    y = bws().nvfp4_gemv(c, s, t, x)
    y_ref, A = P.nvfp4_gemv(*host, f64(x))
    ok, worst, _ = T.check(y_ref, f64(y), A)
    assert ok


def test_deterministic():
    W = rand_W((3000, 5120), seed=11)
    c, s, t, _ = _quant_nvfp4(W)
    x = rand_x(1, 5120, seed=12)
    ys = [bws().nvfp4_gemv(c, s, t, x) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


def test_gate_up_silu_parity():
    d_inter, d_in = 1100, 1024
    g_dev = _quant_nvfp4(rand_W((d_inter, d_in), seed=21, index=0))
    u_dev = _quant_nvfp4(rand_W((d_inter, d_in), seed=21, index=1))
    x = rand_x(1, d_in, seed=21)
    h = bws().nvfp4_gate_up_silu(g_dev[:3], u_dev[:3], x)
    g, Ag = P.nvfp4_gemv(*g_dev[3], f64(x))
    u, Au = P.nvfp4_gemv(*u_dev[3], f64(x))
    h_exact = M.silu(g) * u
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = np.abs(sig * (1.0 + g * (1.0 - sig)))
    tg, tu = 1e-4 * Ag, 1e-4 * Au
    extra = dsilu * np.abs(u) * tg + np.abs(M.silu(g)) * tu + 1.1 * tg * tu + 1e-6 * np.abs(h_exact)
    ok, worst, at = T.check(h_exact, f64(h), np.zeros_like(h_exact), extra=extra)
    assert ok, (worst, at)


def test_dense_stack_parity():
    """A one-token decode step whose NVFP4 products all take the tensor-core
    kernel (every d_in a multiple of 256), including the fused multi-matrix
    mixer input and the SwiGLU gate/up."""
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    stack = W.dense_27b(1, seed=8, n_layers=3, hidden=512, inter=1024, vocab=1000, attn=(768, 256, 256, 512),
                        gdn=(1280, 512), quant=oracle_quantizers(device()), device=device())
    x0 = synth.activation_bf16(1, stack.hidden, seed=8, device=device())
    logits = stack.step(x0)
    torch.cuda.synchronize()
    ref, A, _ = oracle_logits(stack, F.round_bf16(f64(x0)))
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    ok, worst, at = T.check(ref, f64(logits), A, extra=STACK_SLACK * rms)
    assert ok, (worst, at)
