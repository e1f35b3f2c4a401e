"""The single-matrix, MLP-layer and verify workloads at their full sizes,
through the C ABI, in the launch configuration the step uses (the TMA-fed
product kernel), against the oracle on every output row.

* 17408x5120 NVFP4 gate projection, one token;
* the layer MLP (gate and up 17408x5120, down 5120x17408) at N=1;
* the verify set at N=8: the same MLP plus Wq 12288x5120 and Wo 5120x6144,
  each applied to 8 token vectors of its input width.

W ~ N(0, 0.02) and x ~ N(0, 1) in BF16 from the seeded generators; codes
from the oracle's quantizer (run over row chunks in spawned processes) are
uploaded, so the device takes no input from the CUDA path. Bounds: products
|dy| <= 1e-4 sum|w x| + 1/2 ulp; h adds the propagated gate/up bounds; the
down projection adds sum_j |D_ij| dh_j for the largest legitimate difference
dh_j in its BF16 input h (derived from the h bound, not observed)."""
import numpy as np
import pytest
import torch

from oracle import products as P, model as M, formats as F, tolerance as T
from tests.gpu_util import device, bws, f64
from tests.oracle_pool import nvfp4_quantize_parallel
import synth

pytestmark = pytest.mark.gpu

HIDDEN, INTER, Q_ROWS, O_IN = 5120, 17408, 12288, 6144
SHAPES = {"gate": (INTER, HIDDEN), "up": (INTER, HIDDEN), "down": (HIDDEN, INTER),
          "wq": (Q_ROWS, HIDDEN), "wo": (HIDDEN, O_IN)}


@pytest.fixture(scope="module")
def mats():
    """name -> (device (codes, scales, s_t), host (codes, scales, s_t))."""
    out = {}
    for i, (name, shape) in enumerate(SHAPES.items()):
        W = synth.weight_fp32(shape, seed=0, index=i).numpy()
        c, s, t = nvfp4_quantize_parallel(W)
        del W
        dev = device()
        out[name] = ((torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev),
                      torch.tensor([float(t)], dtype=torch.float32, device=dev)), (c, s, np.float32(t)))
    return out


def _x(N, d, index):
    return synth.activation_bf16(N, d, seed=0, index=index, device=device())


def _product(mats, name, N, index):
    dev_m, host_m = mats[name]
    x = _x(N, SHAPES[name][1], index)
    y = bws().nvfp4_gemv(*dev_m, x)
    torch.cuda.synchronize()
    y_ref, A = P.nvfp4_gemv(*host_m, f64(x))
    ok, worst, at = T.check(y_ref, f64(y), A)
    assert ok, (name, N, worst, at)


def _mlp(mats, N):
    x = _x(N, HIDDEN, 100)
    h = bws().nvfp4_gate_up_silu(mats["gate"][0], mats["up"][0], x)
    y = bws().nvfp4_gemv(*mats["down"][0], h)
    torch.cuda.synchronize()
    X = f64(x)
    g, Ag = P.nvfp4_gemv(*mats["gate"][1], X)
    u, Au = P.nvfp4_gemv(*mats["up"][1], X)
    h_exact = M.silu(g) * u
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = np.abs(sig * (1.0 + g * (1.0 - sig)))
    tg, tu = 1e-4 * Ag, 1e-4 * Au
    extra = dsilu * np.abs(u) * tg + np.abs(M.silu(g)) * tu + 1.1 * tg * tu + 1e-6 * np.abs(h_exact)
    ok, worst, at = T.check(h_exact, f64(h), np.zeros_like(h_exact), extra=extra)
    assert ok, ("h", N, worst, at)
    h_ref = F.round_bf16(h_exact)
    e_h = extra + 0.5 * F.bf16_ulp(np.abs(h_exact) + extra)
    dh = e_h + F.bf16_ulp(np.abs(h_exact) + e_h)
    c, s, t = mats["down"][1]
    y_ref, A = P.nvfp4_gemv(c, s, t, h_ref)
    w_abs = np.abs(P.nvfp4_dequantize(c, s, t))
    ok, worst, at = T.check(y_ref, f64(y), A, extra=dh @ w_abs.T)
    assert ok, ("y", N, worst, at)


def test_gate_projection_17408x5120_one_token(mats):
    _product(mats, "gate", 1, 0)


def test_layer_mlp_one_token(mats):
    _mlp(mats, 1)


def test_verify_set_eight_tokens(mats):
    _mlp(mats, 8)
    _product(mats, "wq", 8, 1)
    _product(mats, "wo", 8, 2)
