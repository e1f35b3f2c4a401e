"""Helpers shared by the GPU parity tests."""
import numpy as np
import pytest
import torch

import synth


def device():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    return torch.device("cuda:0")


def bws():
    import __graft_entry__ as g
    g.build()
    import bit_weight_streaming_gb300 as m
    return m


def np_(t):
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


def f64(t):
    return np_(t).astype(np.float64)


def rand_W(shape, seed, index=0, dev=None, std=0.02):
    return synth.weight_fp32(shape, seed=seed, index=index, std=std, device=dev or device())


def rand_x(n, d, seed, index=0, dev=None, std=1.0):
    return synth.activation_bf16(n, d, seed=seed, index=index, std=std, device=dev or device())
