"""GPU quantizers: codes and scales bit-identical to the oracle."""
import numpy as np
import pytest
import torch

from oracle import quant as Q
from tests.conftest import load_golden, golden_float
from tests.gpu_util import device, bws, np_, rand_W

pytestmark = pytest.mark.gpu


def _golden_W(name):
    g = load_golden(name)
    return g, np.array([[golden_float(v) for v in row] for row in g["W"]], dtype=np.float32)


def test_nvfp4_hand_example():
    g, W = _golden_W("nvfp4_hand.json")
    codes, scales, ts = bws().nvfp4_quantize(torch.from_numpy(W).to(device()))
    assert np_(codes).tolist() == g["codes"]
    assert np_(scales).tolist() == g["scales"]
    assert ts.item() == g["s_t"]


def test_mxfp4_hand_example():
    g, W = _golden_W("mxfp4_hand.json")
    codes, scales = bws().mxfp4_quantize(torch.from_numpy(W).to(device()))
    assert np_(codes).tolist() == g["codes"]
    assert np_(scales).tolist() == g["scales"]


def test_fp8_hand_example():
    g, W = _golden_W("fp8_hand.json")
    codes, rs = bws().fp8_rowwise_quantize(torch.from_numpy(W).to(device()))
    assert np_(codes).tolist() == g["codes"]
    assert np_(rs).tolist() == g["row_scale"]


def _edge_matrix(rows, cols, seed):
    W = np_(rand_W((rows, cols), seed))
    rng = np.random.default_rng(seed)
    W[0, :16] = 0.0                                   # zero block
    W[1, :16] = -0.0
    W[1, 16:32] = np.float32(1e-30)                   # block far below the tensor scale
    W[2, :16] = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25,
                            -0.75, -1.25, -2.5, -5.0, 6.0, 0.1, -0.1, 0.0]) * 0.01
    W[3, 5] = 0.9                                     # outlier
    W[4, :] = rng.standard_normal(cols).astype(np.float32) * np.float32(1e-20)
    W[5, 7] = -0.0
    return W


@pytest.mark.parametrize("shape", [(16, 32), (33, 64), (96, 512), (200, 2560)])
def test_nvfp4_quantize_bitexact(shape):
    W = _edge_matrix(*shape, seed=shape[0])
    codes, scales, ts = bws().nvfp4_quantize(torch.from_numpy(W).to(device()))
    c, s, t = Q.nvfp4_quantize(W)
    assert ts.item() == float(t)
    assert np.array_equal(np_(scales), s)
    assert np.array_equal(np_(codes), c)


@pytest.mark.parametrize("shape", [(8, 32), (40, 96), (300, 768)])
def test_mxfp4_quantize_bitexact(shape):
    W = _edge_matrix(*shape, seed=shape[0])
    W[6, :32] *= np.float32(1e25)
    codes, scales = bws().mxfp4_quantize(torch.from_numpy(W).to(device()))
    c, s = Q.mxfp4_quantize(W)
    assert np.array_equal(np_(scales), s)
    assert np.array_equal(np_(codes), c)


@pytest.mark.parametrize("shape", [(8, 32), (50, 200), (257, 2560)])
def test_fp8_rowwise_bitexact(shape):
    W = _edge_matrix(*shape, seed=shape[0])
    W[0, :] = 0.0
    codes, rs = bws().fp8_rowwise_quantize(torch.from_numpy(W).to(device()))
    c, r = Q.fp8_rowwise_quantize(W)
    assert np.array_equal(np_(rs), r)
    assert np.array_equal(np_(codes), c)


def test_e2m1_rounding_dense_sweep():
    """A dense sweep of FP32 values in [-6, 6] (plus every grid midpoint and
    its FP32 neighbours) through the quantizer with d_b = 1: each block holds
    a 6 so its scale is exactly 1, and the tensor amax 2688 makes s_t = 1."""
    vals = np.linspace(-6.0, 6.0, 1 << 22, dtype=np.float64).astype(np.float32)
    mids = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    near = np.concatenate([np.nextafter(mids, np.float32(0)), mids, np.nextafter(mids, np.float32(9))])
    vals = np.concatenate([vals, near, -near, np.float32([-0.0, 0.0])])
    vals = np.concatenate([vals, np.zeros((-len(vals)) % 15, np.float32)])
    blocks = vals.reshape(-1, 15)
    W = np.zeros((blocks.shape[0] + 1, 16), np.float32)
    W[:-1, 0] = 6.0
    W[:-1, 1:] = blocks
    W[-1, 0] = 2688.0
    codes, scales, ts = bws().nvfp4_quantize(torch.from_numpy(W).to(device()))
    c, s, t = Q.nvfp4_quantize(W)
    assert t == 1.0 and ts.item() == 1.0
    assert np.all(s[:-1] == 0x38)
    assert np.array_equal(np_(scales), s)
    assert np.array_equal(np_(codes), c)


def test_full_size_config0_sampled_rows():
    """17408 x 5120 (the MLP gate projection): codes of sampled rows."""
    dev = device()
    W = rand_W((17408, 5120), seed=0, index=0)
    codes, scales, ts = bws().nvfp4_quantize(W)
    torch.cuda.synchronize()
    amax = np.float32(W.abs().max().item())
    t = Q.nvfp4_tensor_scale(np.array([[amax]], np.float32))
    assert ts.item() == float(t)
    rows = np.random.default_rng(0).choice(17408, 64, replace=False)
    rows = np.concatenate([rows, [0, 17407]])
    Wr = np_(W[torch.from_numpy(rows).to(dev)])
    c, s, _ = Q.nvfp4_quantize(Wr, s_t=t)
    assert np.array_equal(np_(codes[torch.from_numpy(rows).to(dev)]), c)
    assert np.array_equal(np_(scales[torch.from_numpy(rows).to(dev)]), s)
