"""Whole decode step on the GPU against the oracle's whole stack, end to end.

The parity gate of the step is stage by stage (test_gpu_stack_stages.py:
every stage from the GPU's own input at the product bound, no slack). A
chain of a few hundred products amplifies legitimate one-ulp BF16 flips, so
these end-to-end checks allow |dl| <= 1e-4 * sum|w x| + 1/2 ulp +
STACK_SLACK * rms(logits) (STACK_SLACK: see tests/stack_util.py and
test_oracle_stack_sensitivity). They are the only check of the opt-in
persistent step kernel, which has no verification tap; for the kernel chain
they are a second, whole-step view beside the staged gate."""
import numpy as np
import pytest
import torch

from oracle import tolerance as T, formats as F
from tests.gpu_util import device, bws, f64
from tests.stack_util import oracle_quantizers, oracle_logits, STACK_SLACK
import synth

pytestmark = pytest.mark.gpu


def _dense_small(N, n_layers=4):
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    return W.dense_27b(N, seed=3, n_layers=n_layers, hidden=256, inter=512, vocab=1000, attn=(384, 64, 64, 192),
                       gdn=(640, 192), quant=oracle_quantizers(device()), device=device())


def _dense_persistent(N, n_layers=4, inter=1024):
    """Shapes the persistent step kernel takes (every NVFP4 d_in % 256 == 0),
    with that kernel enabled: one launch runs the whole step after the init
    kernel."""
    import os
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    os.environ["BWS_STEP_KERNEL"] = "1"
    try:
        return _dense_persistent_build(N, n_layers, inter, W)
    finally:
        del os.environ["BWS_STEP_KERNEL"]


def _dense_persistent_build(N, n_layers, inter, W):
    return W.dense_27b(N, seed=6, n_layers=n_layers, hidden=512, inter=inter, vocab=1000,
                       attn=(768, 256, 256, 512), gdn=(1280, 512), quant=oracle_quantizers(device()),
                       device=device())


def _check(stack, N, seed):
    x0 = synth.activation_bf16(N, stack.hidden, seed=seed, device=device())
    logits = stack.step(x0)
    torch.cuda.synchronize()
    ref, A, _ = oracle_logits(stack, F.round_bf16(f64(x0)))
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    ok, worst, at = T.check(ref, f64(logits), A, extra=STACK_SLACK * rms)
    assert ok, (worst, at)
    return logits


@pytest.mark.parametrize("N", [1, 4, 8])
def test_dense_stack_parity(N):
    stack = _dense_small(N)
    _check(stack, N, seed=N)


def test_dense_stack_at_step_scale_one_token():
    """Shapes large enough (hundreds of units per product, the h row over 8192
    values) that at one token every path of the in-stack chain runs: products
    depositing raw tile sums and the preps that finish them (residual, BF16
    and SwiGLU stores, one- and long-row clusters), and the stream-K split
    that gives the CTAs starting behind the prep a lighter share."""
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    stack = W.dense_27b(1, seed=11, n_layers=2, hidden=2048, inter=9216, vocab=1000, attn=(2048, 256, 256, 1536),
                        gdn=(6144, 1536), quant=oracle_quantizers(device()), device=device())
    _check(stack, 1, seed=12)


def test_dense_stack_graph_replay_is_deterministic():
    stack = _dense_small(2)
    x0 = synth.activation_bf16(2, 256, seed=1, device=device())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = stack.step(x0).clone()     # records the graph
        b = stack.step(x0).clone()     # replays it
        c = stack.step(x0).clone()
    s.synchronize()
    assert torch.equal(a, b) and torch.equal(b, c)
    d = stack.step(x0)                 # default stream: direct launches
    torch.cuda.synchronize()
    assert torch.equal(a, d)


def test_zero_layer_stack_is_the_head():
    stack = _dense_small(3, n_layers=0)
    _check(stack, 3, seed=5)
    assert stack.kernel_count == 2


def test_moe_stack_parity():
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    for N in (1, 4):
        layers = W.moe_stack_layers(N, seed=4, n_dense=1, n_moe=2, hidden=256, inter=64, n_experts=32, topk=4,
                                    dense_inter=384, quant=oracle_quantizers(device()), device=device())
        head = W.make_matrix(3, (900, 256), 4, 7, oracle_quantizers(device()), device())
        stack = bws().stack.DecodeStack(256, layers, head, N, device=device())
        assert stack.kernel_count == 4 + 2 * 4 + 2
        _check(stack, N, seed=10 + N)


@pytest.mark.parametrize("N", [1, 3, 8])
def test_dense_stack_persistent_kernel(N):
    stack = _dense_persistent(N)
    assert stack.kernel_count == 2
    _check(stack, N, seed=20 + N)


def test_dense_stack_persistent_kernel_many_slabs():
    """N = 8 with a 3072-wide MLP: the down projection's activations do not
    fit one shared-memory slab, so its k range is cut into three slabs whose
    partial sums meet in the tile fix-up."""
    stack = _dense_persistent(8, n_layers=2, inter=3072)
    assert stack.kernel_count == 2
    _check(stack, 8, seed=31)


def test_dense_stack_persistent_kernel_replay_is_deterministic():
    stack = _dense_persistent(2, n_layers=2)
    x0 = synth.activation_bf16(2, 512, seed=4, device=device())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = stack.step(x0).clone()
        b = stack.step(x0).clone()
    s.synchronize()
    d = stack.step(x0)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, d)
